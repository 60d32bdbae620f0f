"""Tensor-core operand layouts (K-major / MN-major row panels, fp16 / bf16)
checked against a float64 product of the same rounded operands."""

import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k", [(32, 32), (64, 64), (64, 128), (128, 64), (128, 128), (32, 128)])
@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("bf16", [False, True])
def test_tcgen05_layouts(n, k, a_mn, b_mn, bf16):
    A = W.randn((128, k), 1, f"umma.A{n}{k}")
    B = W.randn((n, k), 1, f"umma.B{n}{k}")
    dt = torch.bfloat16 if bf16 else torch.float16
    Ar, Br = A.to(dt).double(), B.to(dt).double()
    expect = Ar @ Br.T
    D = torch.full((128, n), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lin_state_selftest_mma(A.cuda(), B.cuda(), D, a_mn, b_mn, bf16, status=st)
    assert L.lin_state_read_status(st) == 0
    err = (D.double().cpu() - expect).abs().max().item()
    assert err < 1e-3 * expect.abs().max().item(), err
