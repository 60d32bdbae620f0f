"""The additive (Mamba2 SSD) form, LIN_UPDATE_ADDITIVE: S' = S Diag(alpha) +
beta v k^T (MambaRadixCache page, section 9.3: S_new = A S_old + B x), on the
same pool, tracking, verify and commit machinery, against the oracle. Inputs
follow the SSD recipe: dt = softplus(N(0,1) - 3), A = -U[1, 16] per head,
g = dt A, beta = dt; SiLU after the conv, no q/k normalisation."""

import numpy as np
import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import (TOL_BF16, TOL_F32, compare_outputs, compare_slots, fill_pool,
                           max_rel_per_head, np64, oracle_pool)

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAGS = L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE
PATHS = {"chunked": 0, "recurrent": L.LIN_PREFILL_RECURRENT}


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def _prefill_both(pool, op, b, slots, tracks, cu_track, stride, path, out_dtype, extra=0):
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
              gate_mode=b.gate_mode, flags=FLAGS | PATHS[path] | extra, status=st)
    want = L.LIN_KERNEL_CHUNKED if path == "chunked" else L.LIN_KERNEL_RECURRENT
    if L.lin_state_prefill_kernel(pool, **kw) != want:
        pytest.skip(f"the {path} kernel does not cover these shapes")
    L.lin_state_prefill(pool, **kw)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                        b.cu_seqlens.tolist(), b.prefix_len.tolist(), slots,
                        b.has_initial_state.tolist(), tracks, cu_track, stride, b.gate_mode,
                        FLAGS, 1.0, "bf16" if out_dtype == torch.bfloat16 else "f32")
    assert L.lin_state_read_status(st) == ost == 0
    return out, oo


@pytest.mark.parametrize("path", list(PATHS))
def test_ssd_prefill_fp32_state(path):
    """8 heads, K = V = 128, bf16 inputs, fp32 state and outputs, three ragged
    requests (two warm from a 64-multiple prefix), snapshots every 64 into
    ping-pong pairs."""
    dims = W.LayerDims(num_heads=8, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [700, 333, 1030], W.GATE_PER_HEAD, dtype=torch.bfloat16,
                             seed=5, gate="ssd", prefixes=[128, 0, 768], warm=[1, 0, 1],
                             tag="ssd")
    pool = L.StatePool(1, 12, 8, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 50, std=0.2)
    op = oracle_pool(pool)
    out, oo = _prefill_both(pool, op, b, [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 64,
                            path, torch.float32)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, list(range(1, 10)), TOL_F32)


@pytest.mark.parametrize("path", list(PATHS))
def test_ssd_prefill_bf16_per_key_gates(path):
    """The additive form with per-key gates (alpha a vector, as in GLA-style
    layers): 4 heads, bf16 state and outputs, track stride 256."""
    dims = W.LayerDims(num_heads=4, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [520, 77], W.GATE_PER_KEY, dtype=torch.bfloat16, seed=6,
                             prefixes=[256, 0], warm=[1, 0], tag="ssdk")
    b.beta = b.beta * 0.1
    pool = L.StatePool(1, 8, 4, 128, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 51, std=0.2)
    op = oracle_pool(pool)
    out, oo = _prefill_both(pool, op, b, [1, 2], [3, 4, 5, 6], [0, 2, 4], 256, path,
                            torch.bfloat16)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_BF16)
    compare_slots(pool, op, list(range(1, 7)), TOL_BF16)


def test_ssd_prefill_in_segments():
    """One 1,500-token request in segments (the affine-map scan) from a warm
    slot, snapshots every 64 into 4 distinct slots cycled."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [1500], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=7,
                             gate="ssd", prefixes=[64], warm=[1], tag="ssds")
    pool = L.StatePool(1, 8, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 52, std=0.2)
    op = oracle_pool(pool)
    out, oo = _prefill_both(pool, op, b, [1], [2, 3, 4, 5], [0, 4], 64, "chunked",
                            torch.float32, extra=L.LIN_PREFILL_SEGMENTED)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [1, 2, 3, 4, 5], TOL_F32)


@pytest.mark.parametrize("D", [64, 128])
def test_ssd_decode_vs_oracle(D):
    """Eight decode steps of 5 requests, fp32 state, interval 256 crossed."""
    H = 3
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pool = L.StatePool(1, 16, H, D, state_dtype=torch.float32, conv_dtype=torch.float32,
                       device=DEV)
    fill_pool(pool, 53, std=0.2)
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 53, "ssd.w", std=0.5)
    slots, track, pos = [4, 9, 1, 13, 7], [5, -1, 2, 3, 8], [250, 10, 255, 511, 3]
    worst = 0.0
    for step in range(8):
        x, g, beta = W.make_decode_inputs(dims, 5, 1, L.LIN_GATE_PER_HEAD, torch.float32, 53,
                                          tag="ssdd", step=step, gate="ssd")
        out = torch.zeros((5, 1, H, D), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.lin_state_decode(pool, layer=0, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                           beta=beta.to(DEV), out=out, slot=_i32(slots), pos=_i32(pos),
                           track_slot=_i32(track), track_interval=256,
                           gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS, status=st)
        oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, track,
                           256, O.GATE_PER_HEAD, FLAGS, 1.0, "f32")
        assert L.lin_state_read_status(st) == ost == 0
        worst = max(worst, max_rel_per_head(np64(out), oo, 2))
        pos = [p + 1 for p in pos]
    assert worst < TOL_F32
    t = np64(pool.temporal[0])
    for s in range(16):
        assert max_rel_per_head(t[s], op["temporal"][0, s], 0) < TOL_F32
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_ssd_verify_replay_and_spec_commit():
    """Verify 4 drafts with a per-step buffer and without one (against the
    oracle's outputs-only verify), then commit from the buffer on one pool and replay the accepted
    prefix on the other: identical slots and track slots, equal to the
    oracle's verify + commit."""
    H, D, ND, B, S = 2, 128, 4, 5, 16
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pa = L.StatePool(1, S, H, D, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                     device=DEV)
    fill_pool(pa, 54, std=0.1)
    pb = L.StatePool(1, S, H, D, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                     device=DEV, temporal=pa.temporal.clone(), conv=pa.conv.clone())
    op = oracle_pool(pa)
    conv_w = W.randn((dims.conv_channels, 4), 54, "ssdv.w", std=0.5).to(torch.bfloat16).to(DEV)
    slots, track = [3, 7, 11, 12, 1], [4, 8, -1, 13, 2]
    pos, acc = [254, 100, 253, 255, 0], [3, 4, 0, 1, 2]
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, L.LIN_GATE_PER_HEAD,
                                                           torch.bfloat16, 54, tag="ssdv",
                                                           gate="ssd"))
    spec = L.SpecBuffer(pa, B, ND)
    oa = torch.zeros((B, ND, H, D), device=DEV)
    ob = torch.zeros((B, ND, H, D), device=DEV)
    common = dict(layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots), pos=_i32(pos),
                  gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS)
    L.lin_state_decode(pa, out=oa, spec=spec, **common)
    L.lin_state_decode(pb, out=ob, **common)
    ov, _ = O.verify_outputs(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots,
                             O.GATE_PER_HEAD, FLAGS)
    assert max_rel_per_head(np64(ob), ov, 2) < TOL_F32
    assert max_rel_per_head(np64(ob), np64(oa), 2) < TOL_BF16
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_spec_commit(pa, spec=spec, slot=_i32(slots), pos=_i32(pos), accept_len=_i32(acc),
                            n_draft=ND, track_slot=_i32(track), track_interval=256, status=st)
    L.lin_state_replay_commit(pb, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots),
                              pos=_i32(pos), accept_len=_i32(acc), track_slot=_i32(track),
                              track_interval=256, gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS,
                              status=st)
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pa.temporal, pb.temporal)
    assert torch.equal(pa.conv, pb.conv)
    ospec = O.make_spec_buffer(1, B, ND, H, D, D, dims.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       O.GATE_PER_HEAD, FLAGS, 1.0, "f32", spec=ospec)
    assert ost == 0
    assert max_rel_per_head(np64(ob), oo, 2) < TOL_BF16
    O.spec_commit(op, ospec, 0, 1, slots, pos, acc, track, 256, ND)
    t = np64(pb.temporal[0])
    for s_ in range(S):
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < TOL_BF16
    assert np.array_equal(np64(pb.conv), op["conv"])


def test_ssd_recurrent_small_head_and_noalloc():
    """The additive form on the token-by-token prefill at head dim 32 (fp32
    pool, two ragged requests, one warm), and through lin_state_prefill_noalloc
    on the chunked kernel (head dim 128, a batch of two)."""
    dims = W.LayerDims(num_heads=3, head_k=32, head_v=32)
    b = W.make_prefill_batch(dims, [150, 77], W.GATE_PER_HEAD, dtype=torch.float32, seed=8,
                             gate="ssd", prefixes=[64, 0], warm=[1, 0], tag="ssdr")
    pool = L.StatePool(1, 8, 3, 32, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    fill_pool(pool, 55, std=0.2)
    op = oracle_pool(pool)
    out, oo = _prefill_both(pool, op, b, [1, 2], [3, 4, 5, 6], [0, 2, 4], 64, "recurrent",
                            torch.float32)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, list(range(1, 7)), TOL_F32)

    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [333, 200], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=9,
                             gate="ssd", tag="ssdn")
    pool = L.StatePool(1, 8, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                       device=DEV)
    op = oracle_pool(pool)
    T = b.total_tokens
    out = torch.zeros((T, 2, 128), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_prefill_noalloc(pool, layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
                                beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
                                prefix_len=b.prefix_len.to(DEV), slot=_i32([1, 2]),
                                has_initial_state=b.has_initial_state.to(DEV),
                                track_slots=_i32([3, 4, 5, 6]), cu_track=_i32([0, 2, 4]),
                                track_stride=64, gate_mode=W.GATE_PER_HEAD, flags=FLAGS, status=st)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                        b.cu_seqlens.tolist(), b.prefix_len.tolist(), [1, 2],
                        b.has_initial_state.tolist(), [3, 4, 5, 6], [0, 2, 4], 64,
                        W.GATE_PER_HEAD, FLAGS, 1.0, "f32")
    assert L.lin_state_read_status(st) == ost == 0
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, [1, 2, 3, 4, 5, 6], TOL_F32)


def test_ssd_tree_verify_and_commit():
    """Draft-tree verify and commit in the additive form: outputs, per-step
    states and the committed node against the oracle (head dim 64, fp32)."""
    H, D, ND = 2, 64, 8
    trees = [[-1, -1, 0, 0, 1, 2, 2, 5], [-1, 0, 0, 2, 2, 2, 5, 1]]
    B = len(trees)
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pool = L.StatePool(1, 12, H, D, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    fill_pool(pool, 56, std=0.1)
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 56, "ssdt.w", std=0.5).to(DEV)
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, L.LIN_GATE_PER_HEAD,
                                                           torch.float32, 56, tag="ssdt",
                                                           gate="ssd"))
    slots, pos, track = [1, 2], [254, 100], [3, 4]
    spec = L.SpecBuffer(pool, B, ND)
    out = torch.zeros((B, ND, H, D), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    par = _i32(trees).view(B, ND)
    L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, out=out, slot=_i32(slots),
                       pos=_i32(pos), spec=spec, gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS,
                       status=st, parent=par)
    assert L.lin_state_read_status(st) == 0
    ospec = O.make_spec_buffer(1, B, ND, H, D, D, dims.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       O.GATE_PER_HEAD, FLAGS, 1.0, "f32", spec=ospec, parent=trees)
    assert ost == 0
    assert max_rel_per_head(np64(out), oo, 3) < TOL_F32
    sp = np64(spec.temporal)
    for r in range(B):
        for j in range(ND):
            assert max_rel_per_head(sp[0, r, j], ospec["temporal"][0, r, j], 0) < TOL_F32
    acc_node = [7, 6]
    L.lin_state_spec_commit(pool, spec=spec, slot=_i32(slots), pos=_i32(pos), n_draft=ND,
                            track_slot=_i32(track), track_interval=256, status=st, parent=par,
                            accept_node=_i32(acc_node))
    assert L.lin_state_read_status(st) == 0
    O.spec_commit(op, ospec, 0, 1, slots, pos, None, track, 256, ND, parent=trees,
                  accept_node=acc_node)
    t = np64(pool.temporal[0])
    for s_ in slots + track:
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < TOL_F32
    assert np.array_equal(np64(pool.conv)[0, slots + track], op["conv"][0, slots + track])
