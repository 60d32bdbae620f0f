"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the whole workload runs on the GPU, and sampled (request, head) slices
are recomputed by the oracle. Heads are independent, so the oracle runs on the
slice's own channels, gates and state rows."""

import numpy as np
import pytest
import torch

import bench
import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import TOL_BF16, TOL_F32, np64, rel_l2

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
FLAGS = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU


def head_channels(H, D, heads, V=None):
    """Conv channels of the given heads, q | k | v parts (D key channels per
    head in q and k, V value channels, V = D unless given)."""
    V = D if V is None else V
    idx = []
    for part in range(3):
        n = D if part < 2 else V
        for h in heads:
            idx.extend(range(part * H * D + h * n, part * H * D + (h + 1) * n))
    return np.array(idx)


def oracle_slice_prefill(wl, req, heads, pool_before_t, pool_before_c):
    """Run the oracle for one request on the given heads of a PrefillWorkload."""
    b = wl.b
    H, D, Vd = b.dims.num_heads, b.dims.head_k, b.dims.head_v
    ch = head_channels(H, D, heads, Vd)
    a, e = int(b.cu_seqlens[req]), int(b.cu_seqlens[req + 1])
    x = np64(b.x[a:e])[:, ch]
    w = np64(b.conv_w)[ch]
    g = np64(b.g[a:e])[:, heads]
    beta = np64(b.beta[a:e])[:, heads]
    slot = int(wl.slot[req])
    cu_tr = wl.cu_track.cpu().tolist()
    tracks = wl.track.cpu().tolist()[cu_tr[req]:cu_tr[req + 1]]
    S = pool_before_t.shape[1]
    sd = "bf16" if wl.pool.temporal.dtype == torch.bfloat16 else "f32"
    pool = {"temporal": np.zeros((1, S, len(heads), Vd, D)), "conv": np.zeros((1, S, len(ch), 3)),
            "state_dtype": sd, "conv_dtype": "bf16"}
    pool["temporal"][0, slot] = np64(pool_before_t[0, slot][heads])
    pool["conv"][0, slot] = np64(pool_before_c[0, slot][ch])
    od = "bf16" if wl.out.dtype == torch.bfloat16 else "f32"
    out, st = O.prefill(pool, 0, x, w, g, beta, [0, e - a], [int(b.prefix_len[req])], [slot],
                        [int(b.has_initial_state[req])], tracks, [0, len(tracks)],
                        wl.track_stride, b.gate_mode, wl.kw["flags"], 1.0, od)
    assert st == 0
    return out, pool, slot, tracks, (a, e), ch


def check_prefill_slice(wl, req, heads, tol):
    before_t = wl.pool.temporal.clone().cpu()
    before_c = wl.pool.conv.clone().cpu()
    wl.step(0)
    torch.cuda.synchronize()
    out, op, slot, tracks, (a, e), ch = oracle_slice_prefill(wl, req, heads, before_t, before_c)
    got = np64(wl.out[a:e][:, heads])
    for k in range(len(heads)):
        assert rel_l2(got[:, k], out[:, k]) <= tol, (req, heads[k], rel_l2(got[:, k], out[:, k]))
    for s in [slot] + [t for t in tracks if t >= 0]:
        gt = np64(wl.pool.temporal[0, s][heads])
        for k in range(len(heads)):
            assert rel_l2(gt[k], op["temporal"][0, s, k]) <= tol, (s, heads[k])
        assert np.array_equal(np64(wl.pool.conv[0, s])[ch], op["conv"][0, s])


def test_qwen35_gdn_prefill_full_size_sampled():
    wl = bench.make_workload("qwen35_gdn_prefill", L, DEV)
    check_prefill_slice(wl, 5, [0, 31], TOL_F32)


def test_mamba2_ssd_prefill_full_size_sampled():
    wl = bench.make_workload("mamba2_ssd_prefill", L, DEV)
    assert wl.kw["flags"] & L.LIN_UPDATE_ADDITIVE
    check_prefill_slice(wl, 3, [7, 30], TOL_F32)


def test_mamba2_ssd_prefill_hd64_full_size_sampled():
    """Head dim 64, state size 128 (64 heads), on the chunked kernel with its
    value side padded: sampled requests and heads against the oracle."""
    wl = bench.make_workload("mamba2_ssd_prefill_hd64", L, DEV)
    assert wl.kernel_kind == L.LIN_KERNEL_CHUNKED
    check_prefill_slice(wl, 6, [0, 63], TOL_F32)


def test_kimi_k3_kda_varlen_full_size_sampled():
    wl = bench.make_workload("kimi_k3_kda_varlen_prefill", L, DEV)
    lens = (wl.b.cu_seqlens[1:] - wl.b.cu_seqlens[:-1]).cpu()
    longest = int(torch.argmax(lens))
    warm = [r for r in range(wl.B) if int(wl.b.has_initial_state[r])]
    check_prefill_slice(wl, longest, [3, 11], TOL_BF16)
    # a warm request on a fresh copy of the workload (the step above moved the pool on)
    wl2 = bench.make_workload("kimi_k3_kda_varlen_prefill", L, DEV)
    check_prefill_slice(wl2, warm[0], [0], TOL_BF16)


def test_kda_recurrent_prefill_full_size_sampled():
    """The token-by-token kernel at the benchmark's size: a sampled request
    and heads against the oracle."""
    wl = bench.make_workload("kda_recurrent_prefill", L, DEV)
    assert wl.kernel_kind == L.LIN_KERNEL_RECURRENT
    check_prefill_slice(wl, 17, [2, 9], TOL_BF16)


def test_kimi_k3_kda_varlen_fp32_state_full_size_sampled():
    """The Kimi-K3 varlen workload (32 requests of U{1k..16k} tokens, half warm
    at a 64-multiple prefix, per-key decay, snapshots every 256) with an fp32
    pool and fp32 outputs: the chunked kernel's fp32-state path holds the fp32
    bar at full size, on the longest request and on a warm one."""
    Ls, Ps = W.kp_lengths(0)
    ext = [l - p for l, p in zip(Ls, Ps)]
    warm = [1 if p else 0 for p in Ps]

    def make():
        return bench.PrefillWorkload(L, DEV, "kimi_k3_kda_varlen_prefill", W.KIMI_K3_TP8, ext, Ps,
                                     warm, W.GATE_PER_KEY, torch.bfloat16, torch.float32,
                                     torch.float32, 256, 2, "softplus")

    wl = make()
    assert wl.kernel_kind == L.LIN_KERNEL_CHUNKED
    longest = int(torch.argmax(torch.tensor(ext)))
    check_prefill_slice(wl, longest, [3, 11], TOL_F32)
    wl2 = make()
    check_prefill_slice(wl2, warm.index(1), [5], TOL_F32)


def test_long_single_request_full_size_snapshots():
    """131,072 tokens, 12 heads, snapshots every 64 into 2,048 distinct slots:
    every snapshot's conv window equals the 3 inputs before its boundary (bit for
    bit, so every snapshot sits in the right slot), and one head's outputs and
    states at sampled boundaries match the oracle."""
    wl = bench.make_workload("kda_long_prefill_131k", L, DEV)
    before_t = wl.pool.temporal.clone().cpu()
    before_c = wl.pool.conv.clone().cpu()
    wl.step(0)
    torch.cuda.synchronize()
    b = wl.b
    H, D = 12, 128
    tracks = wl.track.cpu().tolist()
    assert len(tracks) == 2048
    conv = wl.pool.conv[0].cpu()
    xs = b.x.cpu()
    for i, s in enumerate(tracks):
        bnd = 64 * (i + 1)
        assert torch.equal(conv[s].view(torch.int16), xs[bnd - 3:bnd].T.contiguous().view(torch.int16))
    out, op, slot, _, (a, e), ch = oracle_slice_prefill(wl, 0, [7], before_t, before_c)
    got = np64(wl.out[:, 7])
    assert rel_l2(got, out[:, 0]) <= TOL_BF16
    for i in [0, 1, 1023, 2047]:
        s = tracks[i]
        assert rel_l2(np64(wl.pool.temporal[0, s, 7]), op["temporal"][0, s, 0]) <= TOL_BF16


def test_kda_decode_full_size_sampled():
    """The decode workload (2000-slot pools, 256 requests, track interval 256):
    eight steps as bench.py runs them (rotating 4 pool replicas), then two
    requests x two heads of replica 0 against the oracle."""
    wl = bench.make_workload("kda_decode", L, DEV)
    rep0_t = wl.pools[0].temporal.clone().cpu()
    rep0_c = wl.pools[0].conv.clone().cpu()
    outs = []
    for i in range(8):
        wl.step(i)
        if i % 4 == 0:
            outs.append(wl.out.clone())
        torch.cuda.synchronize()
    dims = W.KIMI_K3_TP8
    heads = [2, 9]
    ch = head_channels(12, 128, heads)
    for req in [0, 200]:
        slot = int(wl.slot[req])
        ts = int(wl.track[req])
        pool = {"temporal": np.zeros((1, 2000, 2, 128, 128)), "conv": np.zeros((1, 2000, len(ch), 3)),
                "state_dtype": "bf16", "conv_dtype": "bf16"}
        pool["temporal"][0, slot] = np64(rep0_t[0, slot][heads])
        pool["conv"][0, slot] = np64(rep0_c[0, slot][ch])
        for n, i in enumerate([0, 4]):
            x, g, beta = wl.inputs[i % len(wl.inputs)]
            pos = int(wl.pos0[req]) + i // 4
            o, st = O.decode(pool, 0, np64(x[req:req + 1])[:, :, ch], np64(wl.conv_w)[ch],
                             np64(g[req:req + 1])[:, :, heads], np64(beta[req:req + 1])[:, :, heads],
                             [slot], [pos], [ts], 256, O.GATE_PER_KEY, FLAGS, 1.0, "bf16")
            assert st == 0
            got = np64(outs[n][req][:, heads])
            for k in range(2):
                assert rel_l2(got[0, k], o[0, 0, k]) <= TOL_BF16
        gt = np64(wl.pools[0].temporal[0, slot][heads])
        for k in range(2):
            assert rel_l2(gt[k], pool["temporal"][0, slot, k]) <= TOL_BF16
        assert np.array_equal(np64(wl.pools[0].conv[0, slot])[ch], pool["conv"][0, slot])


def test_kda_verify4_replay_full_size_sampled():
    """The verify-4 + replay-commit workload (2000-slot pools, 256 requests):
    one step as bench.py runs it, then two requests x two heads of replica 0
    against the oracle's verify and commit."""
    wl = bench.make_workload("kda_spec_verify4_replay", L, DEV)
    rep0_t = wl.pools[0].temporal.clone().cpu()
    rep0_c = wl.pools[0].conv.clone().cpu()
    wl.step(0)
    torch.cuda.synchronize()
    heads = [1, 10]
    ch = head_channels(12, 128, heads)
    x, g, beta = wl.inputs[0]
    acc = wl.acc.cpu().tolist()
    for req in [3, 250]:
        slot = int(wl.slot[req])
        ts = int(wl.track[req])
        pos = int(wl.pos0[req])
        pool = {"temporal": np.zeros((1, 2000, 2, 128, 128)), "conv": np.zeros((1, 2000, len(ch), 3)),
                "state_dtype": "bf16", "conv_dtype": "bf16"}
        pool["temporal"][0, slot] = np64(rep0_t[0, slot][heads])
        pool["conv"][0, slot] = np64(rep0_c[0, slot][ch])
        ospec = O.make_spec_buffer(1, 1, 4, 2, 128, 128, len(ch))
        o, st = O.decode(pool, 0, np64(x[req:req + 1])[:, :, ch], np64(wl.conv_w)[ch],
                         np64(g[req:req + 1])[:, :, heads], np64(beta[req:req + 1])[:, :, heads],
                         [slot], [pos], None, 0, O.GATE_PER_KEY, FLAGS, 1.0, "bf16", spec=ospec)
        assert st == 0
        got = np64(wl.out[req][:, heads])
        # the outputs-only verify: the state unrounded across the drafts
        ov, _ = O.verify_outputs(pool, 0, np64(x[req:req + 1])[:, :, ch], np64(wl.conv_w)[ch],
                                 np64(g[req:req + 1])[:, :, heads],
                                 np64(beta[req:req + 1])[:, :, heads], [slot], O.GATE_PER_KEY,
                                 FLAGS, 1.0, "bf16")
        for k in range(2):
            assert rel_l2(got[:, k], o[0, :, k]) <= TOL_BF16
            assert rel_l2(got[:, k], ov[0, :, k]) <= TOL_BF16
        O.spec_commit(pool, ospec, 0, 1, [slot], [pos], [acc[req]], [ts], 256, 4)
        gt = np64(wl.pools[0].temporal[0, slot][heads])
        for k in range(2):
            assert rel_l2(gt[k], pool["temporal"][0, slot, k]) <= TOL_BF16
        assert np.array_equal(np64(wl.pools[0].conv[0, slot])[ch], pool["conv"][0, slot])


def test_kda_verify4_commit_full_size_sampled():
    """The verify-4 + commit workload (2000-slot pools, 256 requests, per-step
    states in a spec buffer): one step as bench.py runs it, then two requests x
    two heads of replica 0 against the oracle: outputs, every per-step state
    and window in the spec buffer, and the committed slot and track slot."""
    wl = bench.make_workload("kda_spec_verify4_commit", L, DEV)
    rep0_t = wl.pools[0].temporal.clone().cpu()
    rep0_c = wl.pools[0].conv.clone().cpu()
    wl.step(0)
    torch.cuda.synchronize()
    heads = [4, 11]
    ch = head_channels(12, 128, heads)
    x, g, beta = wl.inputs[0]
    acc = wl.acc.cpu().tolist()
    spec = wl.specs[0]
    for req in [7, 131]:
        slot = int(wl.slot[req])
        ts = int(wl.track[req])
        pos = int(wl.pos0[req])
        pool = {"temporal": np.zeros((1, 2000, 2, 128, 128)), "conv": np.zeros((1, 2000, len(ch), 3)),
                "state_dtype": "bf16", "conv_dtype": "bf16"}
        pool["temporal"][0, slot] = np64(rep0_t[0, slot][heads])
        pool["conv"][0, slot] = np64(rep0_c[0, slot][ch])
        pool["temporal"][0, ts] = np64(rep0_t[0, ts][heads])
        pool["conv"][0, ts] = np64(rep0_c[0, ts][ch])
        ospec = O.make_spec_buffer(1, 1, 4, 2, 128, 128, len(ch))
        o, st = O.decode(pool, 0, np64(x[req:req + 1])[:, :, ch], np64(wl.conv_w)[ch],
                         np64(g[req:req + 1])[:, :, heads], np64(beta[req:req + 1])[:, :, heads],
                         [slot], [pos], None, 0, O.GATE_PER_KEY, FLAGS, 1.0, "bf16", spec=ospec)
        assert st == 0
        got = np64(wl.out[req][:, heads])
        for k in range(2):
            assert rel_l2(got[:, k], o[0, :, k]) <= TOL_BF16
        for j in range(4):
            gs = np64(spec.temporal[0, req, j][heads])
            for k in range(2):
                assert rel_l2(gs[k], ospec["temporal"][0, 0, j, k]) <= TOL_BF16
            assert np.array_equal(np64(spec.conv[0, req, j])[ch], ospec["conv"][0, 0, j])
        O.spec_commit(pool, ospec, 0, 1, [slot], [pos], [acc[req]], [ts], 256, 4)
        for s_ in (slot, ts):
            gt = np64(wl.pools[0].temporal[0, s_][heads])
            for k in range(2):
                assert rel_l2(gt[k], pool["temporal"][0, s_, k]) <= TOL_BF16
            assert np.array_equal(np64(wl.pools[0].conv[0, s_])[ch], pool["conv"][0, s_])


def test_kda_tree_verify8_commit_full_size_sampled():
    """The draft-tree verify + commit workload (2000-slot pools, 256 requests,
    8 drafts in the MambaRadixCache page's tree shape, a random accepted node
    per request): one step as bench.py runs it, then two requests x two heads
    of replica 0 against the oracle: outputs, every node's state and window in
    the spec buffer, and the committed slot and track slot."""
    wl = bench.make_workload("kda_tree_verify8_commit", L, DEV)
    rep0_t = wl.pools[0].temporal.clone().cpu()
    rep0_c = wl.pools[0].conv.clone().cpu()
    wl.step(0)
    torch.cuda.synchronize()
    assert L.lin_state_read_status(wl.status) == 0
    heads = [4, 11]
    ch = head_channels(12, 128, heads)
    x, g, beta = wl.inputs[0]
    node = wl.accept_node.cpu().tolist()
    spec = wl.specs[0]
    ND = len(wl.TREE)
    for req in [7, 131]:
        slot = int(wl.slot[req])
        ts = int(wl.track[req])
        pos = int(wl.pos0[req])
        pool = {"temporal": np.zeros((1, 2000, 2, 128, 128)), "conv": np.zeros((1, 2000, len(ch), 3)),
                "state_dtype": "bf16", "conv_dtype": "bf16"}
        pool["temporal"][0, slot] = np64(rep0_t[0, slot][heads])
        pool["conv"][0, slot] = np64(rep0_c[0, slot][ch])
        pool["temporal"][0, ts] = np64(rep0_t[0, ts][heads])
        pool["conv"][0, ts] = np64(rep0_c[0, ts][ch])
        ospec = O.make_spec_buffer(1, 1, ND, 2, 128, 128, len(ch))
        o, st = O.decode(pool, 0, np64(x[req:req + 1])[:, :, ch], np64(wl.conv_w)[ch],
                         np64(g[req:req + 1])[:, :, heads], np64(beta[req:req + 1])[:, :, heads],
                         [slot], [pos], None, 0, O.GATE_PER_KEY, FLAGS, 1.0, "bf16", spec=ospec,
                         parent=[wl.TREE])
        assert st == 0
        got = np64(wl.out[req][:, heads])
        for k in range(2):
            assert rel_l2(got[:, k], o[0, :, k]) <= TOL_BF16
        for j in range(ND):
            gs = np64(spec.temporal[0, req, j][heads])
            for k in range(2):
                assert rel_l2(gs[k], ospec["temporal"][0, 0, j, k]) <= TOL_BF16
            assert np.array_equal(np64(spec.conv[0, req, j])[ch], ospec["conv"][0, 0, j])
        O.spec_commit(pool, ospec, 0, 1, [slot], [pos], None, [ts], 256, ND, parent=[wl.TREE],
                      accept_node=[node[req]])
        for s_ in (slot, ts):
            gt = np64(wl.pools[0].temporal[0, s_][heads])
            for k in range(2):
                assert rel_l2(gt[k], pool["temporal"][0, s_, k]) <= TOL_BF16
            assert np.array_equal(np64(wl.pools[0].conv[0, s_])[ch], pool["conv"][0, s_])


def test_headline_e2e_pipeline_equals_one_call():
    """bench.py's end-to-end leg runs each request of the headline batch as
    consecutive warm-started calls on its own stream, with host copies in and
    out. Its outputs read back to the host equal the one-call prefill's, bit
    for bit (requests are independent; the fp32 state and the bf16 windows
    round-trip the pool exactly), and so do the slots and track slots it
    leaves."""
    wl = bench.make_workload("qwen35_gdn_prefill", L, DEV)
    wl.step(0)
    torch.cuda.synchronize()
    ref_out = wl.out.clone()
    ref_t = wl.pool.temporal.clone()
    ref_c = wl.pool.conv.clone()
    wl.out.zero_()
    wl.setup_e2e()
    assert len(wl.parts) > 1
    wl.step_e2e(0)
    torch.cuda.synchronize()
    assert torch.equal(wl.h_out.to(DEV), ref_out)
    assert torch.equal(wl.pool.temporal, ref_t)
    assert torch.equal(wl.pool.conv, ref_c)
