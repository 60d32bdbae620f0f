"""Heads with 128 key channels and 64 value channels (state [64][128]: the SSD
head of the Mamba2 layer, state size 128 and head dim 64; the pool layout of
the MambaRadixCache page, 1.3, with V != K), against the oracle. Prefill of
this shape runs on the chunked tensor-core kernel (its value side padded to
128 rows) and on the token-by-token kernel; decode, verify, replay, tree
verify, commit and slot copies run on the same kernels as the square heads."""

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
H, K, V = 3, 128, 64
DIMS = W.LayerDims(num_heads=H, head_k=K, head_v=V)
GDN = L.LIN_CONV_SILU | L.LIN_QK_L2NORM
SSD = L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE
SDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def _pool(sdt, slots, seed, cdt=torch.bfloat16, layers=1):
    pool = L.StatePool(layers, slots, H, K, state_dtype=SDT[sdt], conv_dtype=cdt, device=DEV,
                       head_v=V)
    assert tuple(pool.temporal.shape[2:]) == (H, V, K)
    assert pool.conv_channels == 2 * H * K + H * V
    fill_pool(pool, seed, std=0.2)
    return pool


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
@pytest.mark.parametrize("sdt,gate,flags", [("f32", "gdn", GDN), ("bf16", "kda", GDN),
                                            ("f32", "kda", GDN), ("f32", "ssd", SSD)])
def test_prefill_head_v64(sdt, gate, flags, path):
    """Three ragged requests (two warm from a 64-multiple prefix), snapshots
    every 64 into ping-pong pairs; the delta rule with per-head and per-key
    gates, and the additive form; both prefill kernels."""
    if path == "recurrent":
        flags = flags | L.LIN_PREFILL_RECURRENT
    gm = W.GATE_PER_KEY if gate == "kda" else W.GATE_PER_HEAD
    b = W.make_prefill_batch(DIMS, [300, 97, 415], gm, dtype=torch.bfloat16, seed=60,
                             gate="ssd" if gate == "ssd" else "softplus", prefixes=[128, 0, 64],
                             warm=[1, 0, 1], tag=f"hv64.{gate}")
    pool = _pool(sdt, 12, 61)
    op = oracle_pool(pool)
    T = b.total_tokens
    odt = torch.bfloat16 if sdt == "bf16" else torch.float32
    out = torch.full((T, H, V), -9.0, dtype=odt, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, tracks, cu_track = [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6]
    kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
              beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
              prefix_len=b.prefix_len.to(DEV), slot=_i32(slots),
              has_initial_state=b.has_initial_state.to(DEV), track_slots=_i32(tracks),
              cu_track=_i32(cu_track), track_stride=64, gate_mode=gm, flags=flags, status=st)
    want = L.LIN_KERNEL_CHUNKED if path == "chunked" else L.LIN_KERNEL_RECURRENT
    assert L.lin_state_prefill_kernel(pool, **kw) == want
    L.lin_state_prefill(pool, **kw)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                        b.cu_seqlens.tolist(), b.prefix_len.tolist(), slots,
                        b.has_initial_state.tolist(), tracks, cu_track, 64, gm, flags, 1.0,
                        "bf16" if odt == torch.bfloat16 else "f32")
    assert L.lin_state_read_status(st) == ost == 0
    tol = TOL_BF16 if sdt == "bf16" else TOL_F32
    compare_outputs(out, oo, b.cu_seqlens.tolist(), tol)
    compare_slots(pool, op, list(range(1, 10)), tol)
    # slots the call does not name are untouched
    assert np.array_equal(np64(pool.temporal[0, 10:]), op["temporal"][0, 10:])


@pytest.mark.parametrize("gate", ["kda", "ssd"])
def test_prefill_head_v64_in_segments(gate):
    """One long request in segments on the chunked kernel (offset and
    transition runs, the fp32 scan, final runs) with a 64-channel value side:
    the transition runs carry all 128 key rows of the affine map while the
    value rows beyond 64 stay zero."""
    gm = W.GATE_PER_KEY if gate == "kda" else W.GATE_PER_HEAD
    flags = (GDN if gate == "kda" else SSD) | L.LIN_PREFILL_SEGMENTED
    n = 1200
    b = W.make_prefill_batch(DIMS, [n], gm, dtype=torch.bfloat16, seed=64,
                             gate="ssd" if gate == "ssd" else "softplus", prefixes=[64], warm=[1],
                             tag=f"hv64s.{gate}")
    n_tr = (64 + n) // 64 - 1
    pool = _pool("f32", 2 + n_tr, 65)
    op = oracle_pool(pool)
    out = torch.zeros((n, H, V), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tracks = list(range(2, 2 + n_tr))
    kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
              beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
              prefix_len=b.prefix_len.to(DEV), slot=_i32([1]),
              has_initial_state=b.has_initial_state.to(DEV), track_slots=_i32(tracks),
              cu_track=_i32([0, n_tr]), track_stride=64, gate_mode=gm, flags=flags, status=st)
    assert L.lin_state_prefill_kernel(pool, **kw) == L.LIN_KERNEL_CHUNKED
    assert L.lin_state_prefill_workspace(pool, **kw) > 16 * 1024  # per-segment states
    L.lin_state_prefill(pool, **kw)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta), [0, n], [64],
                        [1], [1], tracks, [0, n_tr], 64, gm, flags, 1.0, "f32")
    assert L.lin_state_read_status(st) == ost == 0
    compare_outputs(out, oo, [0, n], TOL_F32)
    compare_slots(pool, op, [1] + tracks, TOL_F32)


@pytest.mark.parametrize("sdt,gate,flags", [("f32", "gdn", GDN), ("bf16", "kda", GDN),
                                            ("bf16", "ssd", SSD)])
def test_decode_head_v64(sdt, gate, flags):
    """Six decode steps of 5 requests on distinct slots, track interval 256
    crossed by two of them; one request with no slot (-1) is skipped."""
    gm = W.GATE_PER_KEY if gate == "kda" else W.GATE_PER_HEAD
    pool = _pool(sdt, 16, 62)
    op = oracle_pool(pool)
    conv_w = W.randn((DIMS.conv_channels, 4), 62, "hv64d.w", std=0.5).to(torch.bfloat16)
    slots, track, pos = [4, 9, -1, 13, 7], [5, -1, 2, 3, 8], [250, 10, 255, 253, 3]
    worst = 0.0
    for step in range(6):
        x, g, beta = W.make_decode_inputs(DIMS, 5, 1, gm, torch.bfloat16, 62, tag=f"hv64d.{gate}",
                                          step=step, gate="ssd" if gate == "ssd" else "softplus")
        out = torch.zeros((5, 1, H, V), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.lin_state_decode(pool, layer=0, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                           beta=beta.to(DEV), out=out, slot=_i32(slots), pos=_i32(pos),
                           track_slot=_i32(track), track_interval=256, gate_mode=gm, flags=flags,
                           status=st)
        oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, track,
                           256, gm, flags, 1.0, "f32")
        assert L.lin_state_read_status(st) == ost == 0
        live = [r for r, s in enumerate(slots) if s >= 0]
        worst = max(worst, max_rel_per_head(np64(out)[live], oo[live], 2))
        pos = [p + 1 for p in pos]
    tol = TOL_BF16 if sdt == "bf16" else TOL_F32
    assert worst < tol, worst
    t = np64(pool.temporal[0])
    for s in range(16):
        assert max_rel_per_head(t[s], op["temporal"][0, s], 0) < tol
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_verify_replay_and_spec_commit_head_v64():
    """Verify 4 drafts into a per-step buffer and without one (against the
    oracle's outputs-only verify, the state unrounded across the drafts), commit from the buffer on one pool and replay the accepted
    prefix on the other: identical pools, equal to the oracle's verify and
    commit (bf16 state, per-key gates)."""
    ND, B, S = 4, 5, 16
    pa = _pool("bf16", S, 63)
    pb = L.StatePool(1, S, H, K, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                     device=DEV, head_v=V, temporal=pa.temporal.clone(), conv=pa.conv.clone())
    op = oracle_pool(pa)
    conv_w = W.randn((DIMS.conv_channels, 4), 63, "hv64v.w", std=0.5).to(torch.bfloat16).to(DEV)
    slots, track = [3, 7, 11, 12, 1], [4, 8, -1, 13, 2]
    pos, acc = [254, 100, 253, 255, 0], [3, 4, 0, 1, 2]
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(DIMS, B, ND, L.LIN_GATE_PER_KEY,
                                                           torch.bfloat16, 63, tag="hv64v"))
    spec = L.SpecBuffer(pa, B, ND)
    assert tuple(spec.temporal.shape[3:]) == (H, V, K)
    oa = torch.zeros((B, ND, H, V), device=DEV)
    ob = torch.zeros((B, ND, H, V), device=DEV)
    common = dict(layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots), pos=_i32(pos),
                  gate_mode=L.LIN_GATE_PER_KEY, flags=GDN)
    L.lin_state_decode(pa, out=oa, spec=spec, **common)
    L.lin_state_decode(pb, out=ob, **common)
    ov, _ = O.verify_outputs(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots,
                             O.GATE_PER_KEY, GDN)
    assert max_rel_per_head(np64(ob), ov, 2) < TOL_F32
    assert max_rel_per_head(np64(ob), np64(oa), 2) < TOL_BF16
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_spec_commit(pa, spec=spec, slot=_i32(slots), pos=_i32(pos), accept_len=_i32(acc),
                            n_draft=ND, track_slot=_i32(track), track_interval=256, status=st)
    L.lin_state_replay_commit(pb, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots),
                              pos=_i32(pos), accept_len=_i32(acc), track_slot=_i32(track),
                              track_interval=256, gate_mode=L.LIN_GATE_PER_KEY, flags=GDN,
                              status=st)
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pa.temporal, pb.temporal)
    assert torch.equal(pa.conv, pb.conv)
    ospec = O.make_spec_buffer(1, B, ND, H, K, V, DIMS.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       O.GATE_PER_KEY, GDN, 1.0, "f32", spec=ospec)
    assert ost == 0
    assert max_rel_per_head(np64(ob), oo, 2) < TOL_BF16
    sp = np64(spec.temporal)
    for r in range(B):
        for j in range(ND):
            assert max_rel_per_head(sp[0, r, j], ospec["temporal"][0, r, j], 0) < TOL_BF16
    O.spec_commit(op, ospec, 0, 1, slots, pos, acc, track, 256, ND)
    t = np64(pb.temporal[0])
    for s_ in range(S):
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < TOL_BF16
    assert np.array_equal(np64(pb.conv), op["conv"])


def test_tree_verify_and_commit_head_v64():
    """Draft-tree verify (8 drafts per request, branching) and commit of an
    accepted node, fp32 state, against the oracle."""
    ND = 8
    trees = [[-1, -1, 0, 0, 1, 2, 2, 5], [-1, 0, 0, 2, 2, 2, 5, 1]]
    B = len(trees)
    pool = _pool("f32", 12, 64, cdt=torch.float32)
    op = oracle_pool(pool)
    conv_w = W.randn((DIMS.conv_channels, 4), 64, "hv64t.w", std=0.5).to(DEV)
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(DIMS, B, ND, L.LIN_GATE_PER_HEAD,
                                                           torch.float32, 64, tag="hv64t"))
    slots, pos, track = [1, 2], [254, 100], [3, 4]
    spec = L.SpecBuffer(pool, B, ND)
    out = torch.zeros((B, ND, H, V), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    par = _i32(trees).view(B, ND)
    L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, out=out, slot=_i32(slots),
                       pos=_i32(pos), spec=spec, gate_mode=L.LIN_GATE_PER_HEAD, flags=GDN,
                       status=st, parent=par)
    assert L.lin_state_read_status(st) == 0
    ospec = O.make_spec_buffer(1, B, ND, H, K, V, DIMS.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       O.GATE_PER_HEAD, GDN, 1.0, "f32", spec=ospec, parent=trees)
    assert ost == 0
    assert max_rel_per_head(np64(out), oo, 3) < TOL_F32
    sp = np64(spec.temporal)
    for r in range(B):
        for j in range(ND):
            assert max_rel_per_head(sp[0, r, j], ospec["temporal"][0, r, j], 0) < TOL_F32
    assert np.array_equal(np64(spec.conv), ospec["conv"])
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


def test_copy_slots_head_v64():
    """Fork copies on a 3-layer pool of these heads: bit-exact, layers 1..2."""
    pool = _pool("bf16", 10, 65, layers=3)
    op = oracle_pool(pool)
    src, dst = [1, 4, 7], [2, 9, 0]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_copy_slots(pool, _i32(src), _i32(dst), 1, 3, status=st)
    assert O.copy_slots(op, src, dst, 1, 3) == 0
    assert L.lin_state_read_status(st) == 0
    assert np.array_equal(np64(pool.temporal), op["temporal"])
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_unsupported_head_shapes_rejected():
    """(128, 32) and (64, 32) heads are refused with LIN_EUNSUPPORTED before
    any launch."""
    for k, v in [(128, 32), (64, 32)]:
        pool = L.StatePool(1, 4, 2, k, state_dtype=torch.float32, device=DEV, head_v=v)
        dims = W.LayerDims(num_heads=2, head_k=k, head_v=v)
        x, g, beta = W.make_decode_inputs(dims, 1, 1, L.LIN_GATE_PER_HEAD, torch.float32, 1)
        out = torch.zeros((1, 1, 2, v), device=DEV)
        with pytest.raises(L.LinStateError) as e:
            L.lin_state_decode(pool, layer=0, x=x.to(DEV),
                               conv_w=torch.zeros((dims.conv_channels, 4), device=DEV),
                               g=g.to(DEV), beta=beta.to(DEV), out=out, slot=_i32([0]),
                               pos=_i32([0]), gate_mode=L.LIN_GATE_PER_HEAD, flags=GDN)
        assert e.value.code == L.LIN_EUNSUPPORTED
