"""The outputs-only verify (lin_state_decode with n_draft > 1 and no spec
buffer: the replay form of speculative decoding, Kimi-K3 notes "ReplaySSM",
MambaRadixCache page 9.2 - 9.10), which runs the drafts as one chunk from the
slot state, against the oracle's outputs-only verify (the state carried
unrounded across the drafts): head shapes, draft counts up to the limit,
state and input dtypes, both gate modes, the additive form, padding and bad
slots. The pool is never written."""

import numpy as np
import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import TOL_F32, fill_pool, max_rel_per_head, np64, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("K,V,sdt,io,gate,ND,flags", [
    (128, 128, torch.bfloat16, torch.bfloat16, L.LIN_GATE_PER_KEY, 4, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
    (128, 128, torch.float32, torch.bfloat16, L.LIN_GATE_PER_HEAD, 7, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
    (128, 128, torch.float32, torch.float32, L.LIN_GATE_PER_KEY, 16, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
    (128, 128, torch.bfloat16, torch.bfloat16, L.LIN_GATE_PER_HEAD, 2, L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE),
    (128, 64, torch.bfloat16, torch.bfloat16, L.LIN_GATE_PER_KEY, 5, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
    (128, 64, torch.float32, torch.bfloat16, L.LIN_GATE_PER_HEAD, 3, L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE),
    (64, 64, torch.bfloat16, torch.float32, L.LIN_GATE_PER_KEY, 9, L.LIN_QK_L2NORM),
    (32, 32, torch.float32, torch.float32, L.LIN_GATE_PER_KEY, 32, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
    (16, 16, torch.float32, torch.float32, L.LIN_GATE_PER_HEAD, 6, L.LIN_QK_L2NORM | L.LIN_CONV_SILU),
])
def test_outputs_only_verify_matches_oracle(K, V, sdt, io, gate, ND, flags):
    H, B, S = 3, 6, 12
    dims = W.LayerDims(num_heads=H, head_k=K, head_v=V)
    cdt = torch.float32 if io == torch.float32 else torch.bfloat16
    pool = L.StatePool(1, S, H, K, state_dtype=sdt, conv_dtype=cdt, device=DEV, head_v=V)
    fill_pool(pool, 81, std=0.1)
    before_t, before_c = pool.temporal.clone(), pool.conv.clone()
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 81, "vc.w", std=0.5).to(io).to(DEV)
    kind = "ssd" if flags & L.LIN_UPDATE_ADDITIVE else "softplus"
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, gate, io, 81, tag="vc",
                                                           gate=kind))
    slots = [3, -1, 7, 1, 11, 5]
    out = torch.full((B, ND, H, V), -5.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, out=out, slot=_i32(slots),
                       pos=_i32([100] * B), gate_mode=gate, flags=flags, status=st)
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pool.temporal, before_t) and torch.equal(pool.conv, before_c)
    ov, ost = O.verify_outputs(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, gate, flags)
    assert ost == 0
    live = [r for r in range(B) if slots[r] >= 0]
    assert max_rel_per_head(np64(out)[live], ov[live], 2) < TOL_F32
    assert torch.all(out[1] == -5.0)  # padding: nothing written


def test_outputs_only_verify_bad_slot_and_limits():
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    pool = L.StatePool(1, 4, 2, 128, device=DEV)
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, 2, 4, L.LIN_GATE_PER_KEY,
                                                           torch.bfloat16, 5, tag="vcb"))
    conv_w = W.randn((dims.conv_channels, 4), 5, "vcb.w").to(torch.bfloat16).to(DEV)
    out = torch.full((2, 4, 2, 128), -5.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, out=out, slot=_i32([4, 2]),
                       pos=_i32([0, 0]), gate_mode=L.LIN_GATE_PER_KEY, status=st)
    assert L.lin_state_read_status(st) == L.LIN_ST_BAD_SLOT
    assert torch.all(out[0] == -5.0) and not torch.all(out[1] == -5.0)
    # more drafts than one chunk takes (a bf16 pool: within the staging limit)
    pool = L.StatePool(1, 4, 2, 128, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16, device=DEV)
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, 1, 33, L.LIN_GATE_PER_KEY,
                                                           torch.bfloat16, 5, tag="vcl"))
    with pytest.raises(L.LinStateError, match="at most 32 drafts"):
        L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta,
                           out=torch.zeros((1, 33, 2, 128), device=DEV), slot=_i32([1]),
                           pos=_i32([0]), gate_mode=L.LIN_GATE_PER_KEY)
