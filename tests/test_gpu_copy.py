"""Slot copies and restore on the GPU against the oracle (bit-exact)."""

import numpy as np
import pytest
import torch

import bench
import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import fill_pool, np64, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("sdt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [16, 128])
def test_copy_slots_matches_oracle(sdt, D):
    pool = L.StatePool(3, 12, 2, D, state_dtype=sdt, conv_dtype=sdt, device=DEV)
    fill_pool(pool, 1)
    op = oracle_pool(pool)
    src, dst = [2, 2, 7, -1, 5, 9], [3, 4, 1, 6, 5, 0]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_copy_slots(pool, _i32(src), _i32(dst), 1, 3, status=st)
    assert O.copy_slots(op, src, dst, 1, 3) == 0
    assert L.lin_state_read_status(st) == 0
    assert np.array_equal(np64(pool.temporal), op["temporal"])
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_copy_slots_validate_and_bad_ids():
    pool = L.StatePool(2, 10, 2, 16, device=DEV)
    fill_pool(pool, 2)
    op = oracle_pool(pool)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    src, dst = [3, 8, 1], [9, 3, 2]  # pair 1 writes slot 3, which pair 0 reads
    L.lin_state_copy_slots(pool, _i32(src), _i32(dst), flags=L.LIN_VALIDATE, status=st)
    ost = O.copy_slots(op, src, dst, 0, 2, O.FLAG_VALIDATE)
    assert L.lin_state_read_status(st) == ost == L.LIN_ST_COPY_ALIAS
    assert np.array_equal(np64(pool.temporal), op["temporal"])
    L.lin_state_copy_slots(pool, _i32([0, 1]), _i32([10, 4]), status=st)
    ost = O.copy_slots(op, [0, 1], [10, 4], 0, 2)
    assert L.lin_state_read_status(st) == ost == L.LIN_ST_BAD_SLOT
    assert np.array_equal(np64(pool.temporal), op["temporal"])


def test_restore_matches_oracle():
    pool = L.StatePool(4, 10, 2, 64, state_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 3)
    op = oracle_pool(pool)
    ops = [(1, 1, 5), (2, 1, -1), (3, 0, 6), (-1, 1, 5), (4, 1, 99), (6, 1, 6)]
    his = torch.full((len(ops),), 7, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_restore(pool, _i32(ops), his, status=st)
    ohis = np.full(len(ops), 7, np.int64)
    ost = O.restore(op, ops, ohis)
    assert L.lin_state_read_status(st) == ost
    assert his.cpu().tolist() == ohis.tolist() == [1, 0, 7, 7, 0, 1]
    assert np.array_equal(np64(pool.temporal), op["temporal"])
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_copy_bench_workload_full_size():
    """The benchmark's copy workload as it is timed: 64 pairs of 69-layer
    Kimi-K3 slots over a 128-slot pool, each slot used once. Every destination
    holds its source's bytes from before the call; nothing else changes."""
    wl = bench.make_workload("slot_copy_kimi_k3_69l", L, DEV)
    before_t = wl.pool.temporal.clone()
    before_c = wl.pool.conv.clone()
    src, dst = wl.pairs[0]
    assert len(set(src.tolist()) | set(dst.tolist())) == 128
    wl.step(0)
    torch.cuda.synchronize()
    assert L.lin_state_read_status(wl.status) == 0
    exp_t, exp_c = before_t.clone(), before_c.clone()
    exp_t[:, dst.long()] = before_t[:, src.long()]
    exp_c[:, dst.long()] = before_c[:, src.long()]
    assert torch.equal(wl.pool.temporal.view(torch.int16), exp_t.view(torch.int16))
    assert torch.equal(wl.pool.conv.view(torch.int16), exp_c.view(torch.int16))


def test_copy_engine_kimi_k3_full_size():
    """Copy-engine workload at full size: 69-layer Kimi-K3 TP8 slots (12 x 128 x 128
    bf16 + [4608][3] bf16 per layer) in a 256-slot pool, 64 pairs with distinct
    destinations and sources drawn from the other slots. Every destination must hold
    its source's bytes from before the call; every other slot is untouched."""
    pool = L.StatePool(69, 256, 12, 128, state_dtype=torch.bfloat16,
                       conv_dtype=torch.bfloat16, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    pool.temporal.view(torch.int16).random_(generator=g)
    pool.conv.view(torch.int16).random_(generator=g)
    perm = W.randperm(256, 0, "cp.batch0")
    dst = perm[:64]
    src = perm[64:][W.randint(0, 191, (64,), 0, "cp.src0")]
    before_t = pool.temporal.clone()
    before_c = pool.conv.clone()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert L.lin_state_slot_bytes(pool) == 29039616
    L.lin_state_copy_slots(pool, src.to(torch.int32).to(DEV), dst.to(torch.int32).to(DEV), status=st)
    assert L.lin_state_read_status(st) == 0
    exp_t, exp_c = before_t, before_c
    exp_t[:, dst.to(DEV)] = before_t[:, src.to(DEV)].clone()
    exp_c[:, dst.to(DEV)] = before_c[:, src.to(DEV)].clone()
    # compare bit patterns: the random fill holds NaN encodings
    assert torch.equal(pool.temporal.view(torch.int16), exp_t.view(torch.int16))
    assert torch.equal(pool.conv.view(torch.int16), exp_c.view(torch.int16))
