"""Decode, speculative verify and commit on the GPU against the oracle."""

import json
import os

import numpy as np
import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import TOL_BF16, TOL_F32, fill_pool, max_rel_per_head, np64, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAGS = L.LIN_QK_L2NORM | L.LIN_CONV_SILU


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def _decode_both(pool, op, dims, conv_w, slots, pos, track, interval, gate, seed, step,
                 out_dtype, n_draft=1, spec=None, ospec=None):
    B = len(slots)
    x, g, beta = W.make_decode_inputs(dims, B, n_draft, gate, dtype=conv_w.dtype, seed=seed,
                                      step=step)
    out = torch.zeros((B, n_draft, dims.num_heads, dims.head_v), dtype=out_dtype, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_decode(pool, layer=0, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                       beta=beta.to(DEV), out=out, slot=_i32(slots), pos=_i32(pos),
                       track_slot=_i32(track) if track is not None else None,
                       track_interval=interval, spec=spec, gate_mode=gate, flags=FLAGS,
                       status=st)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, track,
                       interval, gate, FLAGS, 1.0, "bf16" if out_dtype == torch.bfloat16 else "f32",
                       spec=ospec)
    assert L.lin_state_read_status(st) == ost
    return np64(out), oo


@pytest.mark.parametrize("gate", [L.LIN_GATE_PER_HEAD, L.LIN_GATE_PER_KEY])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_decode_fp32_state_vs_oracle(gate, D):
    dims = W.LayerDims(num_heads=3, head_k=D, head_v=D)
    pool = L.StatePool(1, 20, 3, D, state_dtype=torch.float32, conv_dtype=torch.float32, device=DEV)
    fill_pool(pool, 10, std=0.2)
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 0, "dec.w", std=0.5)
    slots, track = [4, 9, 1, 17], [5, -1, 2, 3]
    pos = [250, 10, 255, 511]
    worst = 0.0
    for step in range(8):
        o, oo = _decode_both(pool, op, dims, conv_w, slots, pos, track, 256, gate, 10, step,
                             torch.float32)
        worst = max(worst, max_rel_per_head(o, oo, 2))
        pos = [p + 1 for p in pos]
    assert worst < TOL_F32
    t = np64(pool.temporal[0])
    for s in range(20):
        assert max_rel_per_head(t[s], op["temporal"][0, s], 0) < TOL_F32
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_decode_kda_bf16_crossing_track_boundary():
    """KDA decode workload at reduced size: 16 requests x 300 steps, 12 heads,
    bf16 state, interval 256 crossed by every request."""
    dims = W.KIMI_K3_TP8
    pool = L.StatePool(1, 64, 12, 128, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                       device=DEV)
    fill_pool(pool, 11)
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 0, "kd.w", std=0.5).to(torch.bfloat16)
    perm = W.randperm(64, 0, "kd.slots").tolist()
    slots, track = perm[:16], perm[16:32]
    pos = [1024 + 16 * i + (i % 5) for i in range(16)]  # all cross 1280 within 300 steps
    worst = 0.0
    for step in range(300):
        o, oo = _decode_both(pool, op, dims, conv_w, slots, pos, track, 256, L.LIN_GATE_PER_KEY,
                             11, step, torch.bfloat16)
        worst = max(worst, max_rel_per_head(o, oo, 2))
        pos = [p + 1 for p in pos]
    assert worst < TOL_BF16, worst
    t = np64(pool.temporal[0])
    for s in slots + track:
        assert max_rel_per_head(t[s], op["temporal"][0, s], 0) < TOL_BF16
    assert np.array_equal(np64(pool.conv), op["conv"])


def test_decode_track_positions_page_example():
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "decode_track_interval.json")))
    dims = W.LayerDims(num_heads=1, head_k=16, head_v=16)
    pool = L.StatePool(1, 4, 1, 16, device=DEV)
    conv_w = W.randn((dims.conv_channels, 4), 0, "trk.w", std=0.5)
    hits = []
    pos = gold["prompt_len"]
    for step in range(1, gold["decode_tokens_processed"][-1] + 5):
        pool.temporal[0, 2].fill_(float("nan"))
        x, g, b = W.make_decode_inputs(dims, 1, 1, L.LIN_GATE_PER_HEAD, torch.float32, 0,
                                       tag="trk", step=step)
        out = torch.zeros((1, 1, 1, 16), device=DEV)
        L.lin_state_decode(pool, layer=0, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                           beta=b.to(DEV), out=out, slot=_i32([1]), pos=_i32([pos]),
                           track_slot=_i32([2]), track_interval=gold["interval"],
                           gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS)
        if not torch.isnan(pool.temporal[0, 2]).any():
            hits.append(step)
            assert torch.equal(pool.temporal[0, 2], pool.temporal[0, 1])
        pos += 1
    assert hits == gold["decode_tokens_processed"]


@pytest.mark.parametrize("sdt", [torch.float32, torch.bfloat16])
def test_verify_commit_vs_oracle_and_linear_chain(sdt):
    """MambaRadixCache page 8.4 / 9.4: after verify + commit(a) the slot equals a
    single-token decodes, bit for bit on the GPU, and matches the oracle."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    D = 4
    B = 6
    pool = L.StatePool(2, 24, 2, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 12)
    ref_pool = L.StatePool(2, 24, 2, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV,
                           temporal=pool.temporal.clone(), conv=pool.conv.clone())
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 0, "v.w", std=0.5).to(torch.bfloat16)
    slots, track = [3, 7, 11, 15, 19, 21], [4, 8, 12, 16, -1, 22]
    pos = [254, 100, 253, 255, 1, 600]
    acc = [3, 4, 0, 1, 2, 4]
    spec = L.SpecBuffer(pool, B, D)
    ospec = O.make_spec_buffer(2, B, D, 2, 128, 128, dims.conv_channels)
    for layer in range(2):
        x, g, beta = W.make_decode_inputs(dims, B, D, L.LIN_GATE_PER_KEY, torch.bfloat16, 12,
                                          tag=f"v{layer}")
        out = torch.zeros((B, D, 2, 128), device=DEV)
        L.lin_state_decode(pool, layer=layer, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                           beta=beta.to(DEV), out=out, slot=_i32(slots), pos=_i32(pos), spec=spec,
                           gate_mode=L.LIN_GATE_PER_KEY, flags=FLAGS)
        oo, _ = O.decode(op, layer, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None,
                         0, O.GATE_PER_KEY, O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU, spec=ospec)
        assert max_rel_per_head(np64(out), oo, 2) < (TOL_F32 if sdt == torch.float32 else TOL_BF16)
        # the same tokens, one decode at a time, on a copy of the pool
        for r in range(B):
            for j in range(acc[r]):
                o1 = torch.zeros((1, 1, 2, 128), device=DEV)
                L.lin_state_decode(ref_pool, layer=layer, x=x[r:r + 1, j:j + 1].contiguous().to(DEV),
                                   conv_w=conv_w.to(DEV), g=g[r:r + 1, j:j + 1].contiguous().to(DEV),
                                   beta=beta[r:r + 1, j:j + 1].contiguous().to(DEV), out=o1,
                                   slot=_i32([slots[r]]), pos=_i32([pos[r] + j]),
                                   track_slot=_i32([track[r]]), track_interval=256,
                                   gate_mode=L.LIN_GATE_PER_KEY, flags=FLAGS)
                assert torch.equal(o1[0, 0], out[r, j])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_spec_commit(pool, spec=spec, slot=_i32(slots), pos=_i32(pos), accept_len=_i32(acc),
                            n_draft=D, track_slot=_i32(track), track_interval=256, status=st)
    assert L.lin_state_read_status(st) == 0
    O.spec_commit(op, ospec, 0, 2, slots, pos, acc, track, 256, D)
    assert torch.equal(pool.temporal, ref_pool.temporal)
    assert torch.equal(pool.conv, ref_pool.conv)
    tol = TOL_F32 if sdt == torch.float32 else TOL_BF16
    t = np64(pool.temporal)
    for layer in range(2):
        for s in slots + [t_ for t_ in track if t_ >= 0]:
            assert max_rel_per_head(t[layer, s], op["temporal"][layer, s], 0) < tol
    assert np.array_equal(np64(pool.conv), op["conv"])
    # accept_len out of range is reported and skipped
    L.lin_state_spec_commit(pool, spec=spec, slot=_i32([3]), pos=_i32([0]), accept_len=_i32([5]),
                            n_draft=D, status=st)
    assert L.lin_state_read_status(st) == L.LIN_ST_BAD_ACCEPT


def test_decode_and_verify_many_items_per_cta():
    """Enough (request, head) items that every CTA of the persistent decode runs
    several of them and wraps its ring of stages; empty slots (-1) sit between
    live ones. One tracked decode step, then a 3-draft verify, against the oracle."""
    H, D, B, S = 4, 64, 300, 400
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pool = L.StatePool(1, S, H, D, state_dtype=torch.float32, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 21, std=0.1)
    op = oracle_pool(pool)
    perm = W.randperm(S, 21, "many.perm").tolist()
    slots = [(-1 if r % 7 == 3 else perm[r]) for r in range(B)]
    track = [(perm[B + r // 3] if r % 3 == 0 else -1) for r in range(B)]
    pos = [255 if r % 5 == 0 else 17 + r for r in range(B)]
    conv_w = W.randn((dims.conv_channels, 4), 21, "many.w", std=0.5).to(torch.bfloat16)
    o, oo = _decode_both(pool, op, dims, conv_w, slots, pos, track, 256, L.LIN_GATE_PER_KEY, 21, 0,
                         torch.float32)
    live = [r for r in range(B) if slots[r] >= 0]
    assert max_rel_per_head(o[live], oo[live], 2) < TOL_F32
    pos = [p + 1 for p in pos]
    spec = L.SpecBuffer(pool, B, 3)
    ospec = O.make_spec_buffer(1, B, 3, H, D, D, dims.conv_channels)
    o, oo = _decode_both(pool, op, dims, conv_w, slots, pos, None, 0, L.LIN_GATE_PER_KEY, 21, 1,
                         torch.float32, n_draft=3, spec=spec, ospec=ospec)
    assert max_rel_per_head(o[live], oo[live], 2) < TOL_F32
    t = np64(pool.temporal[0])
    for s_ in range(S):
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < TOL_F32
    assert np.array_equal(np64(pool.conv), op["conv"])
    st = np64(spec.temporal)
    for r in live[::10]:
        for j in range(3):
            assert max_rel_per_head(st[0, r, j], ospec["temporal"][0, r, j], 0) < TOL_F32


@pytest.mark.parametrize("sdt,gate", [(torch.bfloat16, L.LIN_GATE_PER_KEY),
                                      (torch.float32, L.LIN_GATE_PER_HEAD)])
def test_replay_commit_equals_spec_commit(sdt, gate):
    """The replay form of speculative decoding ([K3] ReplaySSM, [MRC] 9): a
    verify that keeps no per-step states writes the drafts' outputs with the
    state carried unrounded across them (the oracle's outputs-only verify; the
    per-step verify's outputs within the pool dtype's rounding), and
    re-running the accepted prefix into the slot leaves
    every slot and track slot bit-identical to committing from the per-step
    buffer; both match the oracle. Accept lengths 0 .. D, boundary crossings
    at 256, a padding request, layer 1 of a 2-layer pool."""
    H, D, ND, B, S = 2, 128, 4, 7, 24
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pa = L.StatePool(2, S, H, D, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pa, 31, std=0.1)
    pb = L.StatePool(2, S, H, D, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV,
                     temporal=pa.temporal.clone(), conv=pa.conv.clone())
    op = oracle_pool(pa)
    conv_w = W.randn((dims.conv_channels, 4), 31, "rp.w", std=0.5).to(torch.bfloat16).to(DEV)
    slots = [3, 7, -1, 11, 15, 19, 21]
    track = [4, 8, 9, 12, 16, -1, 22]
    pos = [254, 100, 0, 253, 255, 1, 510]
    acc = [3, 4, 2, 0, 1, 2, 4]
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, gate, torch.bfloat16, 31, tag="rp"))
    spec = L.SpecBuffer(pa, B, ND)
    oa = torch.zeros((B, ND, H, D), device=DEV)
    ob = torch.zeros((B, ND, H, D), device=DEV)
    common = dict(layer=1, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots), pos=_i32(pos),
                  gate_mode=gate, flags=FLAGS)
    L.lin_state_decode(pa, out=oa, spec=spec, **common)
    L.lin_state_decode(pb, out=ob, **common)  # no spec buffer: outputs only
    # the outputs-only verify carries the state unrounded across its drafts
    ov, ost = O.verify_outputs(op, 1, np64(x), np64(conv_w), np64(g), np64(beta), slots, gate, FLAGS)
    assert ost == 0
    assert max_rel_per_head(np64(ob), ov, 2) < TOL_F32
    assert max_rel_per_head(np64(ob), np64(oa), 2) < (TOL_F32 if sdt == torch.float32 else TOL_BF16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_spec_commit(pa, spec=spec, slot=_i32(slots), pos=_i32(pos), accept_len=_i32(acc),
                            n_draft=ND, track_slot=_i32(track), track_interval=256, layer_begin=1,
                            layer_end=2, status=st)
    assert L.lin_state_read_status(st) == 0
    L.lin_state_replay_commit(pb, layer=1, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots),
                              pos=_i32(pos), accept_len=_i32(acc), track_slot=_i32(track),
                              track_interval=256, gate_mode=gate, flags=FLAGS, status=st)
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pa.temporal, pb.temporal)
    assert torch.equal(pa.conv, pb.conv)
    # the oracle: verify into its own per-step buffer, then commit
    ospec = O.make_spec_buffer(2, B, ND, H, D, D, dims.conv_channels)
    oo, ost = O.decode(op, 1, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       gate, FLAGS, 1.0, "f32", spec=ospec)
    assert ost == 0
    live = [r for r in range(B) if slots[r] >= 0]
    tol = TOL_F32 if sdt == torch.float32 else TOL_BF16
    assert max_rel_per_head(np64(ob)[live], oo[live], 2) < tol
    O.spec_commit(op, ospec, 1, 2, slots, pos, acc, track, 256, ND)
    t = np64(pb.temporal[1])
    for s_ in range(S):
        assert max_rel_per_head(t[s_], op["temporal"][1, s_], 0) < tol
    assert np.array_equal(np64(pb.conv), op["conv"])


TREES = [[-1, -1, 0, 0, 1, 2, 2, 5],   # the MambaRadixCache page's shape (9.6): two roots, depth 4
         [-1, 0, 1, 2, 3, 4, 5, 6],     # a chain written as parents
         [-1, -1, -1, 0, 1, 2, 3, 3],   # three roots
         [-1, 0, 0, 2, 2, 2, 5, 1]]


def _path(par, node):
    p = []
    while node >= 0:
        p.insert(0, node)
        node = par[node]
    return p


@pytest.mark.parametrize("sdt,gate", [(torch.bfloat16, L.LIN_GATE_PER_KEY),
                                      (torch.float32, L.LIN_GATE_PER_HEAD)])
def test_tree_verify_and_commit(sdt, gate):
    """Draft-tree verify (MambaRadixCache page 8.3, 9.6: retrieve_parent_token):
    every node's output and per-step state equal, bit for bit, the linear
    verify of its root-to-node path, and match the oracle; committing an
    accepted node equals the oracle's commit (boundaries at 256 included); a
    request whose tree has a parent outside [-1, j) is skipped with
    LIN_ST_BAD_TREE."""
    H, D, ND = 2, 128, 8
    B = len(TREES) + 1
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    pool = L.StatePool(1, 16, H, D, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 41, std=0.1)
    op = oracle_pool(pool)
    conv_w = W.randn((dims.conv_channels, 4), 41, "tr.w", std=0.5).to(torch.bfloat16).to(DEV)
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, gate, torch.bfloat16, 41, tag="tr"))
    parents = TREES + [[-1, 0, 2, 0, 1, 2, 2, 5]]  # the last tree is malformed (draft 2 is its own parent)
    slots, pos = [1, 2, 3, 4, 5], [253, 100, 254, 7, 0]  # trees 0 and 2 cross 256 (ancestor, node)
    spec = L.SpecBuffer(pool, B, ND)
    out = torch.zeros((B, ND, H, D), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    par = _i32(parents).view(B, ND)
    L.lin_state_decode(pool, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, out=out, slot=_i32(slots),
                       pos=_i32(pos), spec=spec, gate_mode=gate, flags=FLAGS, status=st, parent=par)
    assert L.lin_state_read_status(st) == L.LIN_ST_BAD_TREE
    ospec = O.make_spec_buffer(1, B, ND, H, D, D, dims.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0, gate,
                       FLAGS, 1.0, "f32", spec=ospec, parent=parents)
    assert ost == O.ST_BAD_TREE
    tol = TOL_F32 if sdt == torch.float32 else TOL_BF16
    good = list(range(len(TREES)))
    assert max_rel_per_head(np64(out)[good], oo[good], 3) < tol
    # every node equals the linear verify of its path, bit for bit
    for r in good:
        for node in range(ND):
            path = _path(parents[r], node)
            if len(path) < 2:
                continue
            n = len(path)
            sp = L.SpecBuffer(pool, 1, n)
            o1 = torch.zeros((1, n, H, D), device=DEV)
            L.lin_state_decode(pool, layer=0, x=x[r:r + 1, path].contiguous(), conv_w=conv_w,
                               g=g[r:r + 1, path].contiguous(), beta=beta[r:r + 1, path].contiguous(),
                               out=o1, slot=_i32([slots[r]]), pos=_i32([pos[r]]), spec=sp,
                               gate_mode=gate, flags=FLAGS)
            assert torch.equal(o1[0, -1], out[r, node]), (r, node)
            assert torch.equal(sp.temporal[0, 0, -1], spec.temporal[0, r, node]), (r, node)
            assert torch.equal(sp.conv[0, 0, -1], spec.conv[0, r, node]), (r, node)
    # commit an accepted node of each tree
    track = [9, 10, 11, 12, 13]
    acc_node = [7, 5, 4, -1, 3]
    L.lin_state_spec_commit(pool, spec=spec, slot=_i32(slots), pos=_i32(pos), n_draft=ND,
                            track_slot=_i32(track), track_interval=256, status=st, parent=par,
                            accept_node=_i32(acc_node))
    assert L.lin_state_read_status(st) == 0
    O.spec_commit(op, ospec, 0, 1, slots[:4], pos[:4], None, track[:4], 256, ND,
                  parent=parents[:4], accept_node=acc_node[:4])
    t = np64(pool.temporal[0])
    for s_ in slots[:4] + track[:4]:
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < tol
    assert np.array_equal(np64(pool.conv)[0, slots[:4] + track[:4]],
                          op["conv"][0, slots[:4] + track[:4]])


def test_decode_status_bits():
    dims = W.LayerDims(num_heads=1, head_k=32, head_v=32)
    pool = L.StatePool(1, 8, 1, 32, device=DEV)
    fill_pool(pool, 13)
    before = pool.temporal.clone()
    conv_w = W.randn((dims.conv_channels, 4), 0, "s.w")
    x, g, b = W.make_decode_inputs(dims, 3, 1, L.LIN_GATE_PER_HEAD, torch.float32, 0, tag="s")
    out = torch.zeros((3, 1, 1, 32), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_decode(pool, layer=0, x=x.to(DEV), conv_w=conv_w.to(DEV), g=g.to(DEV),
                       beta=b.to(DEV), out=out, slot=_i32([8, 2, -1]), pos=_i32([0, 0, 0]),
                       track_slot=_i32([1, 2, 3]), track_interval=256,
                       gate_mode=L.LIN_GATE_PER_HEAD, flags=FLAGS, status=st)
    assert L.lin_state_read_status(st) == L.LIN_ST_BAD_SLOT | L.LIN_ST_TRACK_ALIAS
    assert torch.equal(pool.temporal, before)


@pytest.mark.parametrize("D,sdt,io,ND,gate", [
    (128, torch.float32, torch.bfloat16, 7, L.LIN_GATE_PER_HEAD),   # groups of 4 + 3
    (64, torch.bfloat16, torch.bfloat16, 9, L.LIN_GATE_PER_KEY),    # 4 + 4 + 1
    (128, torch.float32, torch.float32, 17, L.LIN_GATE_PER_KEY),    # the staging limit: smaller groups
])
def test_long_chains_in_groups(D, sdt, io, ND, gate):
    """Chains longer than one group of drafts: verify with a per-step buffer
    and without one (the latter against the oracle's outputs-only verify),
    buffer commit and replay commit
    (same pools bit for bit), both equal to running the accepted tokens as
    single-token decodes, bit for bit, and to the oracle. Accept lengths span
    the groups; positions cross the 256 boundary inside later groups."""
    H, B, S = 2, 5, 20
    dims = W.LayerDims(num_heads=H, head_k=D, head_v=D)
    cdt = torch.float32 if io == torch.float32 else torch.bfloat16
    pa = L.StatePool(1, S, H, D, state_dtype=sdt, conv_dtype=cdt, device=DEV)
    fill_pool(pa, 71, std=0.1)
    pb = L.StatePool(1, S, H, D, state_dtype=sdt, conv_dtype=cdt, device=DEV,
                     temporal=pa.temporal.clone(), conv=pa.conv.clone())
    pc = L.StatePool(1, S, H, D, state_dtype=sdt, conv_dtype=cdt, device=DEV,
                     temporal=pa.temporal.clone(), conv=pa.conv.clone())
    op = oracle_pool(pa)
    conv_w = W.randn((dims.conv_channels, 4), 71, "lc.w", std=0.5).to(io).to(DEV)
    slots, track = [2, 5, 9, 13, 17], [3, 6, -1, 14, 18]
    pos = [250, 256 - ND + 2, 100, 511 - ND // 2, 7]
    acc = [ND, ND - 2, 5, 1, 0]
    x, g, beta = (t.to(DEV) for t in W.make_decode_inputs(dims, B, ND, gate, io, 71, tag="lc"))
    spec = L.SpecBuffer(pa, B, ND)
    oa = torch.zeros((B, ND, H, D), device=DEV)
    ob = torch.zeros((B, ND, H, D), device=DEV)
    common = dict(layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots), pos=_i32(pos),
                  gate_mode=gate, flags=FLAGS)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lin_state_decode(pa, out=oa, spec=spec, status=st, **common)
    L.lin_state_decode(pb, out=ob, status=st, **common)
    assert L.lin_state_read_status(st) == 0
    # without a spec buffer: the drafts as one chunk, the state unrounded across them
    ov, _ = O.verify_outputs(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, gate, FLAGS)
    assert max_rel_per_head(np64(ob), ov, 2) < TOL_F32
    assert max_rel_per_head(np64(ob), np64(oa), 2) < (TOL_F32 if sdt == torch.float32 else TOL_BF16)
    L.lin_state_spec_commit(pa, spec=spec, slot=_i32(slots), pos=_i32(pos), accept_len=_i32(acc),
                            n_draft=ND, track_slot=_i32(track), track_interval=256, status=st)
    L.lin_state_replay_commit(pb, layer=0, x=x, conv_w=conv_w, g=g, beta=beta, slot=_i32(slots),
                              pos=_i32(pos), accept_len=_i32(acc), track_slot=_i32(track),
                              track_interval=256, gate_mode=gate, flags=FLAGS, status=st)
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pa.temporal, pb.temporal)
    assert torch.equal(pa.conv, pb.conv)
    # the linear chain: the accepted tokens as single-token decodes
    for j in range(ND):
        sl = [s if acc[r] > j else -1 for r, s in enumerate(slots)]
        oc = torch.zeros((B, 1, H, D), device=DEV)
        L.lin_state_decode(pc, layer=0, x=x[:, j:j + 1].contiguous(), conv_w=conv_w,
                           g=g[:, j:j + 1].contiguous(), beta=beta[:, j:j + 1].contiguous(),
                           out=oc, slot=_i32(sl), pos=_i32([p + j for p in pos]),
                           track_slot=_i32(track), track_interval=256, gate_mode=gate,
                           flags=FLAGS, status=st)
        live = [r for r in range(B) if acc[r] > j]
        assert torch.equal(oc[live, 0], oa[live, j])
    assert L.lin_state_read_status(st) == 0
    assert torch.equal(pa.temporal, pc.temporal)
    assert torch.equal(pa.conv, pc.conv)
    # the oracle's verify and commit
    ospec = O.make_spec_buffer(1, B, ND, H, D, D, dims.conv_channels)
    oo, ost = O.decode(op, 0, np64(x), np64(conv_w), np64(g), np64(beta), slots, pos, None, 0,
                       gate, FLAGS, 1.0, "f32", spec=ospec)
    assert ost == 0
    tol = TOL_F32 if sdt == torch.float32 else TOL_BF16
    assert max_rel_per_head(np64(oa), oo, 2) < tol
    sp = np64(spec.temporal)
    for r in range(B):
        for j in range(ND):
            assert max_rel_per_head(sp[0, r, j], ospec["temporal"][0, r, j], 0) < tol
    assert np.array_equal(np64(spec.conv), ospec["conv"])
    O.spec_commit(op, ospec, 0, 1, slots, pos, acc, track, 256, ND)
    t = np64(pa.temporal[0])
    for s_ in range(S):
        assert max_rel_per_head(t[s_], op["temporal"][0, s_], 0) < tol
    assert np.array_equal(np64(pa.conv), op["conv"])
