"""Prefill on the GPU (both the chunked tensor-core path and the recurrent
path) against the oracle: tiny workload, reduced Qwen3.5-style GDN and Kimi-K3
KDA workloads, placement examples, warm == cold, edge cases."""

import json
import os

import numpy as np
import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import (TOL_BF16, TOL_F32, compare_outputs, compare_slots, fill_pool,
                           np64, oracle_pool)

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAGS = L.LIN_QK_L2NORM | L.LIN_CONV_SILU
PATHS = {"chunked": 0, "recurrent": L.LIN_PREFILL_RECURRENT}


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def run_both(pool, op, b, slots, tracks, cu_track, stride, path, out_dtype=torch.float32,
             flags=FLAGS, q_scale=1.0, expect_status=0):
    T = b.total_tokens
    H, V = b.dims.num_heads, b.dims.head_v
    out = torch.full((T, H, V), -9.0, dtype=out_dtype, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
              beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
              prefix_len=b.prefix_len.to(DEV), slot=_i32(slots),
              has_initial_state=b.has_initial_state.to(DEV),
              track_slots=_i32(tracks) if stride else None,
              cu_track=_i32(cu_track) if stride else None, track_stride=stride,
              gate_mode=b.gate_mode, flags=flags | PATHS[path], q_scale=q_scale, status=st)
    want = L.LIN_KERNEL_CHUNKED if path == "chunked" else L.LIN_KERNEL_RECURRENT
    if L.lin_state_prefill_kernel(pool, **kw) != want:
        pytest.skip(f"the {path} kernel does not cover these shapes")
    L.lin_state_prefill(pool, **kw)
    oo = np.full((T, H, V), -9.0)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                        b.cu_seqlens.tolist(), b.prefix_len.tolist(), slots,
                        b.has_initial_state.tolist(), tracks, cu_track, stride, b.gate_mode,
                        flags, q_scale, "bf16" if out_dtype == torch.bfloat16 else "f32", out=oo)
    got = L.lin_state_read_status(st)
    assert got == ost == expect_status, (got, ost)
    return out, oo


@pytest.mark.parametrize("path", list(PATHS))
def test_tiny_gdn_workload(path):
    """Tiny GDN: 2 heads, K=V=16, 96 conv channels, requests of 128 and 200 tokens,
    fp32; request 2's first 64 tokens equal request 1's. Run 1: both cold with
    per-boundary track lists. Run 2: request 2 warm from request 1's checkpoint
    at 64 (P = 64, L = 136) reproduces run 1's outputs and final state."""
    dims = W.TINY_GDN
    b = W.make_prefill_batch(dims, [128, 200], W.GATE_PER_HEAD, dtype=torch.float32, seed=0,
                             tag="t1", qk_prenorm=True)
    b.x[128:192] = b.x[0:64]
    b.g[128:192] = b.g[0:64]
    b.beta[128:192] = b.beta[0:64]
    pool = L.StatePool(1, 16, 2, 16, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    op = oracle_pool(pool)
    tracks, cu_track = [2, 3, 4, 5, 6], [0, 2, 5]  # req1: 64,128; req2: 64,128,192
    out1, oo1 = run_both(pool, op, b, [0, 1], tracks, cu_track, 64, path)
    compare_outputs(out1, oo1, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [0, 1, 2, 3, 4, 5, 6], TOL_F32)
    assert torch.equal(pool.temporal[0, 2], pool.temporal[0, 4])  # same first 64 tokens
    # run 2: request 2 warm from request 1's checkpoint (slot 2)
    L.lin_state_copy_slots(pool, _i32([2]), _i32([9]))
    O.copy_slots(op, [2], [9], 0, 1)
    b2 = W.PrefillBatch(dims, W.GATE_PER_HEAD, b.x[192:], b.conv_w, b.g[192:], b.beta[192:],
                        torch.tensor([0, 136], dtype=torch.int32), torch.tensor([64], dtype=torch.int32),
                        torch.tensor([1], dtype=torch.int64))
    out2, oo2 = run_both(pool, op, b2, [9], [], [0, 0], 0, path)
    compare_outputs(out2, oo2, [0, 136], TOL_F32)
    compare_slots(pool, op, [9], TOL_F32)
    # warm == cold: against run 1's request 2
    tol = 0.0 if path == "chunked" else 1e-5
    diff = (out2 - out1[192:]).abs().max().item()
    assert diff <= tol * out1[192:].abs().max().item(), diff
    sd = (pool.temporal[0, 9] - pool.temporal[0, 1]).abs().max().item()
    assert sd <= tol * pool.temporal[0, 1].abs().max().item() + (0 if path == "chunked" else 1e-6)


@pytest.mark.parametrize("path", list(PATHS))
def test_qwen35_gdn_reduced(path):
    """Qwen3.5-style GDN at reduced size: 32 heads, K=V=128, bf16 inputs, fp32
    state and outputs, scalar log-decay in [-0.1, 0], two requests of 1024 and
    700 tokens (ragged tail), track stride 64 into ping-pong pairs."""
    dims = W.QWEN35_GDN
    b = W.make_prefill_batch(dims, [1024, 700], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=0,
                             gate="uniform", tag="q")
    pool = L.StatePool(1, 8, 32, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    op = oracle_pool(pool)
    out, oo = run_both(pool, op, b, [1, 2], [3, 4, 5, 6], [0, 2, 4], 64, path)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [1, 2, 3, 4, 5, 6], TOL_F32)


@pytest.mark.parametrize("pingpong", [False, True])
@pytest.mark.parametrize("gate", [W.GATE_PER_KEY, W.GATE_PER_HEAD])
def test_single_request_in_segments(gate, pingpong):
    """A batch of one long request run as parallel segments (offset and
    transition runs, the fp32 scan, final runs) equals the oracle: a warm
    start at a 64-multiple prefix, a ragged last segment, snapshots every 64
    into distinct slots that cross segment boundaries (or into a ping-pong
    pair, where segments share track slots and only the last two snapshots
    may remain), outputs, the final state and conv window; and it equals the
    same call run in one piece."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    L_, P_ = 1500, 128
    b = W.make_prefill_batch(dims, [L_], gate, dtype=torch.bfloat16, seed=4,
                             gate="softplus" if gate == W.GATE_PER_KEY else "uniform", tag="seg",
                             prefixes=[P_], warm=[1])
    sdt = torch.bfloat16 if gate == W.GATE_PER_KEY else torch.float32
    n_tr = (P_ + L_) // 64 - P_ // 64
    pool = L.StatePool(1, 2 + n_tr, 2, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 4, std=0.1)
    ref = L.StatePool(1, 2 + n_tr, 2, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV,
                      temporal=pool.temporal.clone(), conv=pool.conv.clone())
    op = oracle_pool(pool)
    tracks = [2, 3] if pingpong else list(range(2, 2 + n_tr))
    n_tr = len(tracks)
    tol = TOL_BF16 if gate == W.GATE_PER_KEY else TOL_F32
    out, oo = run_both(pool, op, b, [1], tracks, [0, n_tr], 64, "chunked",
                       out_dtype=torch.float32, flags=FLAGS | L.LIN_PREFILL_SEGMENTED)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), tol)
    compare_slots(pool, op, [1] + tracks, tol)
    # one piece (no segments) on a copy: the same placement, values within rounding
    out1 = torch.zeros_like(out)
    kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV), beta=b.beta.to(DEV),
              out=out1, cu_seqlens=b.cu_seqlens.to(DEV), prefix_len=b.prefix_len.to(DEV),
              slot=_i32([1]), has_initial_state=b.has_initial_state.to(DEV), track_slots=_i32(tracks),
              cu_track=_i32([0, n_tr]), track_stride=64, gate_mode=gate, flags=FLAGS)
    L.lin_state_prefill(ref, **kw)
    assert torch.equal(pool.conv, ref.conv)  # windows are copies of inputs: bit-exact
    assert (out - out1).norm() <= tol * out1.norm()


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float32])
def test_kda_decay_beyond_chunk_range_is_rerun(sdt):
    """KDA where some (request, head) pairs decay far faster than the chunked
    kernel's factored range allows (log-decay -30 * softplus(N(0,1)) per key
    channel: across half a chunk a channel decays by far more than e^80). The
    chunked call itself must return the right outputs, states and snapshots for
    every pair: the out-of-range pairs through the token-by-token rerun the call
    queues, the others through the chunked kernel; no status bit is set."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    lengths, prefixes, warm = [200, 333, 130], [0, 64, 128], [0, 1, 1]
    b = W.make_prefill_batch(dims, lengths, W.GATE_PER_KEY, dtype=torch.bfloat16, seed=5,
                             gate="softplus", tag="dr", prefixes=prefixes, warm=warm)
    cu = b.cu_seqlens.tolist()
    b.g[cu[0]:cu[1]] *= 30.0              # request 0: both heads out of range
    b.g[cu[1] + 150:cu[1] + 260, 1] *= 30.0  # request 1: head 1 from its third chunk on
    pool = L.StatePool(1, 12, 2, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 6)
    op = oracle_pool(pool)
    out, oo = run_both(pool, op, b, [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 64, "chunked")
    tol = TOL_BF16 if sdt == torch.bfloat16 else TOL_F32
    compare_outputs(out, oo, cu, tol)
    compare_slots(pool, op, list(range(1, 10)), tol)


@pytest.mark.parametrize("where", ["middle", "last"])
def test_kda_decay_beyond_range_in_segments(where):
    """The same in the segmented mode of a long single request: an out-of-range
    stretch inside a middle segment (caught by the offset and transition runs,
    so the final runs skip the head) or inside the last segment (caught by its
    final run, which stops before the write-back); the rerun redoes that head."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    L_ = 1500
    b = W.make_prefill_batch(dims, [L_], W.GATE_PER_KEY, dtype=torch.bfloat16, seed=7,
                             gate="softplus", tag="drs")
    lo = 600 if where == "middle" else 1400
    b.g[lo:lo + 60, 0] *= 30.0
    n_tr = L_ // 64
    pool = L.StatePool(1, 2 + n_tr, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    op = oracle_pool(pool)
    tracks = list(range(2, 2 + n_tr))
    out, oo = run_both(pool, op, b, [1], tracks, [0, n_tr], 64, "chunked",
                       flags=FLAGS | L.LIN_PREFILL_SEGMENTED)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [1] + tracks, TOL_F32)


@pytest.mark.parametrize("path", list(PATHS))
def test_gdn_strong_decay(path):
    """GDN with log-decay U[-12, 0] per (token, head): 16 consecutive tokens can
    decay by far more than e^80, so the chunked kernel's separable decay factors
    must fall back to the direct exponential on those columns; ragged requests."""
    dims = W.LayerDims(num_heads=4, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [300, 130], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=3,
                             gate="uniform", tag="sd")
    b.g = b.g * 120.0
    b.g[5:9] = 0.0  # a few tokens with no decay
    pool = L.StatePool(1, 8, 4, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    op = oracle_pool(pool)
    out, oo = run_both(pool, op, b, [1, 2], [3, 4, 5, 6], [0, 2, 4], 64, path)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [1, 2, 3, 4, 5, 6], TOL_F32)


@pytest.mark.parametrize("path", list(PATHS))
def test_kimi_k3_kda_varlen_reduced(path):
    """Kimi-K3 TP8 KDA varlen prefill at reduced size: 12 heads, bf16 inputs and
    state, per-key decay exp(-softplus(N(0,1))), three requests (two warm from a
    restored checkpoint at a 64-multiple prefix), track stride 256, ping-pong."""
    dims = W.KIMI_K3_TP8
    lengths, prefixes, warm = [700, 333, 1030], [128, 0, 768], [1, 0, 1]
    b = W.make_prefill_batch(dims, lengths, W.GATE_PER_KEY, dtype=torch.bfloat16, seed=0,
                             prefixes=prefixes, warm=warm, tag="kp")
    pool = L.StatePool(1, 12, 12, 128, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 20)
    op = oracle_pool(pool)
    out, oo = run_both(pool, op, b, [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 256, path,
                       out_dtype=torch.bfloat16)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_BF16)
    compare_slots(pool, op, list(range(1, 10)), TOL_BF16)


@pytest.mark.parametrize("path", list(PATHS))
def test_long_request_placement_page_example(path):
    """Ping-Pong page long-request flow: 1200 tokens, chunk 512, three calls;
    B <- S_512, C <- S_1024, A holds S_1200, fork A -> D is bit-identical."""
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "placement_examples.json")))["long_request"]
    A, B_, C, D = (gold["slots"][k] for k in "ABCD")
    dims = W.LayerDims(num_heads=2, head_k=64, head_v=64)
    full = W.make_prefill_batch(dims, [1200], W.GATE_PER_KEY, dtype=torch.float32, seed=0,
                                tag="pp")
    pool = L.StatePool(1, 8, 2, 64, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    pool.temporal.fill_(-7.0)
    op = oracle_pool(pool)
    lst, nxt, pos = [B_, C], 0, 0
    for n in gold["calls"]:
        part = W.PrefillBatch(dims, W.GATE_PER_KEY, full.x[pos:pos + n], full.conv_w,
                              full.g[pos:pos + n], full.beta[pos:pos + n],
                              torch.tensor([0, n], dtype=torch.int32),
                              torch.tensor([pos], dtype=torch.int32),
                              torch.tensor([1 if pos else 0], dtype=torch.int64))
        rot = lst[nxt:] + lst[:nxt]
        out, oo = run_both(pool, op, part, [A], rot, [0, 2], gold["chunk"], path)
        compare_outputs(out, oo, [0, n], TOL_F32)
        if (pos + n) // gold["chunk"] > pos // gold["chunk"]:
            nxt ^= 1
        pos += n
    L.lin_state_copy_slots(pool, _i32([A]), _i32([D]))
    O.copy_slots(op, [A], [D], 0, 1)
    compare_slots(pool, op, [A, B_, C, D], TOL_F32)
    assert torch.equal(pool.temporal[0, D], pool.temporal[0, A])
    # the whole request in one call places the same snapshots
    pool2 = L.StatePool(1, 8, 2, 64, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    op2 = oracle_pool(pool2)
    run_both(pool2, op2, full, [A], [B_, C], [0, 2], gold["chunk"], path)
    tol = 0.0 if path == "chunked" else 1e-5
    for s in (A, B_, C):
        d = (pool2.temporal[0, s] - pool.temporal[0, s]).abs().max().item()
        assert d <= tol * pool.temporal[0, s].abs().max().item() + (0 if path == "chunked" else 1e-6)


@pytest.mark.parametrize("gate", [W.GATE_PER_HEAD, W.GATE_PER_KEY])
@pytest.mark.parametrize("path", list(PATHS))
def test_edge_cases(path, gate):
    """Empty and very short requests, a padding slot, a misaligned prefix, a
    track slot equal to the live slot, a bad slot id: the bad ones are
    reported and skipped, the rest complete."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    lengths = [0, 1, 2, 65, 64, 5, 9, 70]
    prefixes = [0, 64, 0, 0, 32, 0, 0, 128]
    warm = [1, 1, 0, 1, 1, 0, 0, 1]
    b = W.make_prefill_batch(dims, lengths, gate, dtype=torch.bfloat16, seed=0,
                             prefixes=prefixes, warm=warm, tag="edge")
    pool = L.StatePool(1, 16, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 30)
    op = oracle_pool(pool)
    slots = [1, 2, 3, 4, 5, -1, 16, 7]
    tracks = [8, 9, 10, 4, 11, 12, 13, 14]  # request 3's list holds its own slot (4)
    cu_track = [0, 1, 2, 3, 4, 5, 6, 7, 8]
    expect = O.ST_BAD_PREFIX | O.ST_TRACK_ALIAS | O.ST_BAD_SLOT
    out, oo = run_both(pool, op, b, slots, tracks, cu_track, 64, path, expect_status=expect)
    ok_reqs = [0, 1, 2, 7]
    skip = [r for r in range(len(lengths)) if r not in ok_reqs]
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32, skip=skip)
    compare_slots(pool, op, list(range(16)), TOL_F32)
    o = np64(out)
    for r in skip:
        a, e = int(b.cu_seqlens[r]), int(b.cu_seqlens[r + 1])
        assert np.all(o[a:e] == -9.0)


@pytest.mark.parametrize("path", list(PATHS))
def test_multi_layer_pool_and_q_scale(path):
    dims = W.LayerDims(num_heads=2, head_k=64, head_v=64)
    b = W.make_prefill_batch(dims, [100, 64], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=0,
                             tag="ml", warm=[1, 0])
    pool = L.StatePool(3, 6, 2, 64, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 31)
    before = pool.temporal.clone()
    op = oracle_pool(pool)
    T, H, V = b.total_tokens, 2, 64
    out = torch.zeros((T, H, V), device=DEV)
    kw = dict(layer=2, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
              beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
              prefix_len=b.prefix_len.to(DEV), slot=_i32([0, 5]),
              has_initial_state=b.has_initial_state.to(DEV), gate_mode=b.gate_mode,
              flags=FLAGS | PATHS[path], q_scale=0.125)
    want = L.LIN_KERNEL_CHUNKED if path == "chunked" else L.LIN_KERNEL_RECURRENT
    if L.lin_state_prefill_kernel(pool, **kw) != want:
        pytest.skip(f"the {path} kernel does not cover these shapes")
    L.lin_state_prefill(pool, **kw)
    oo, _ = O.prefill(op, 2, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                      b.cu_seqlens.tolist(), [0, 0], [0, 5], [1, 0], [], [0, 0, 0], 0,
                      b.gate_mode, FLAGS, 0.125, "f32")
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_BF16)
    compare_slots(pool, op, [0, 5], TOL_BF16, layer=2)
    assert torch.equal(pool.temporal[:2], before[:2])
