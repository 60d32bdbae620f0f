"""The C restatement of the oracle (oracle/lin_state_ref.c), which the benchmark
times as the CPU baseline, against the numpy oracle it restates: in float64 it
must give the numpy oracle's results up to summation order, in float32 within
fp32 rounding; status bits, snapshot placement and conv windows exactly; the
threaded run equal to the single-threaded one bit for bit."""

import numpy as np
import pytest

from oracle import lin_state_oracle as O
from oracle import lin_state_ref as R

FLAGS = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU


def _rel(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / (nb if nb else 1.0))


def _inputs(rng, T, H, K, V, gate_mode, additive=False):
    C = 2 * H * K + H * V
    x = rng.standard_normal((T, C))
    w = 0.5 * rng.standard_normal((C, 4))
    if gate_mode == O.GATE_PER_KEY:
        g = -np.log1p(np.exp(rng.standard_normal((T, H, K))))
    else:
        g = -np.log1p(np.exp(rng.standard_normal((T, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    if additive:
        beta = beta * 0.1
    return x, w, g, beta, C


def _pool(rng, S, H, K, V, C, sd, cd):
    p = O.make_pool(1, S, H, K, V, C, state_dtype=sd, conv_dtype=cd)
    p["temporal"][:] = O.round_to(0.1 * rng.standard_normal(p["temporal"].shape), sd)
    p["conv"][:] = O.round_to(rng.standard_normal(p["conv"].shape), cd)
    return p


def _copy(p):
    return {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}


@pytest.mark.parametrize("H,K,V", [(2, 16, 16), (2, 32, 32), (1, 128, 64)])
@pytest.mark.parametrize("gate_mode", [O.GATE_PER_HEAD, O.GATE_PER_KEY])
@pytest.mark.parametrize("sd,additive", [("f64", False), ("f32", False), ("bf16", False), ("f64", True)])
def test_prefill_matches_numpy_oracle(H, K, V, gate_mode, sd, additive):
    rng = np.random.default_rng(3)
    # request 3 has a misaligned prefix, request 4 its own slot in its track
    # list, request 5 is padding
    lengths, prefixes, warm = [130, 0, 70, 64, 5, 9], [0, 64, 128, 32, 0, 0], [0, 1, 1, 1, 0, 0]
    T = sum(lengths)
    x, w, g, beta, C = _inputs(rng, T, H, K, V, gate_mode, additive)
    cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
    slots = [1, 2, 3, 4, 11, -1]
    tracks, cu_track = [5, 6, 7, 8, 9, 10, 11], [0, 2, 4, 6, 6, 7, 7]
    flags = FLAGS | (O.FLAG_UPDATE_ADDITIVE if additive else 0)
    cd = "bf16" if sd == "bf16" else sd
    base = _pool(rng, 12, H, K, V, C, sd, cd)
    pn, pc = _copy(base), _copy(base)
    on, sn = O.prefill(pn, 0, x, w, g, beta, cu, prefixes, slots, warm, tracks, cu_track, 64,
                       gate_mode, flags, 0.5, "f32" if sd != "f64" else "f64")
    oc, sc = R.prefill(pc, 0, x, w, g, beta, cu, prefixes, slots, warm, tracks, cu_track, 64,
                       gate_mode, flags, 0.5, "f32" if sd != "f64" else "f64", precision="f64")
    assert sn == sc == (O.ST_BAD_PREFIX | O.ST_TRACK_ALIAS)
    tol = 1e-4 if sd == "bf16" else 1e-12  # bf16: a tie may round the other way
    assert _rel(oc, on) <= tol
    assert _rel(pc["temporal"], pn["temporal"]) <= tol
    assert _rel(pc["conv"], pn["conv"]) <= tol
    # float32: within fp32 rounding of the float64 result
    p32 = _copy(base)
    o32, s32 = R.prefill(p32, 0, x, w, g, beta, cu, prefixes, slots, warm, tracks, cu_track, 64,
                         gate_mode, flags, 0.5, "f32", precision="f32")
    assert s32 == sn
    assert _rel(o32, on) <= 1e-4
    assert _rel(p32["temporal"], pn["temporal"]) <= 1e-4


def test_prefill_threads_equal_one_thread():
    rng = np.random.default_rng(4)
    H, K, V = 3, 32, 32
    lengths = [200, 150, 70]
    T = sum(lengths)
    x, w, g, beta, C = _inputs(rng, T, H, K, V, O.GATE_PER_KEY)
    cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
    base = _pool(rng, 10, H, K, V, C, "f32", "f32")
    res = []
    for n in (1, 7):
        p = _copy(base)
        o, st = R.prefill(p, 0, x, w, g, beta, cu, [0, 64, 0], [1, 2, 3], [0, 1, 0],
                          [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 64, O.GATE_PER_KEY, FLAGS, 1.0, "f32",
                          precision="f32", nthreads=n)
        res.append((o, p))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1]["temporal"], res[1][1]["temporal"])
    assert np.array_equal(res[0][1]["conv"], res[1][1]["conv"])


@pytest.mark.parametrize("sd", ["f64", "bf16"])
@pytest.mark.parametrize("gate_mode", [O.GATE_PER_HEAD, O.GATE_PER_KEY])
def test_decode_verify_commit_match_numpy_oracle(sd, gate_mode):
    rng = np.random.default_rng(5)
    H, K, V, B = 2, 32, 32, 4
    C = 2 * H * K + H * V
    cd = "bf16" if sd == "bf16" else sd
    base = _pool(rng, 16, H, K, V, C, sd, cd)
    conv_w = 0.5 * rng.standard_normal((C, 4))
    slots, pos, track = [1, 3, -1, 5], [255, 10, 0, 510], [2, 4, 6, -1]
    tol = 1e-4 if sd == "bf16" else 1e-12
    # one token in place, with the interval track
    x, _, g, beta, _ = _inputs(rng, B, H, K, V, gate_mode)
    x, g, beta = x[:, None], g[:, None], beta[:, None]
    pn, pc = _copy(base), _copy(base)
    on, sn = O.decode(pn, 0, x, conv_w, g, beta, slots, pos, track, 256, gate_mode, FLAGS)
    oc, sc = R.decode(pc, 0, x, conv_w, g, beta, slots, pos, track, 256, gate_mode, FLAGS)
    assert sn == sc == 0
    assert _rel(oc, on) <= tol and _rel(pc["temporal"], pn["temporal"]) <= tol
    assert np.array_equal(pc["conv"], pn["conv"])
    assert not np.array_equal(pn["temporal"][0, 2], base["temporal"][0, 2])  # 256 was crossed
    # verify 3 drafts into a per-step buffer, then commit 2 / 3 / 0 / 1
    D = 3
    xs, _, gs, bs, _ = _inputs(rng, B * D, H, K, V, gate_mode)
    xs, gs, bs = (a.reshape((B, D) + a.shape[1:]) for a in (xs, gs, bs))
    spn = O.make_spec_buffer(1, B, D, H, K, V, C)
    spc = O.make_spec_buffer(1, B, D, H, K, V, C)
    pos2 = [p + 1 for p in pos]
    on, _ = O.decode(pn, 0, xs, conv_w, gs, bs, slots, pos2, None, 0, gate_mode, FLAGS, spec=spn)
    oc, _ = R.decode(pc, 0, xs, conv_w, gs, bs, slots, pos2, None, 0, gate_mode, FLAGS, spec=spc)
    assert _rel(oc, on) <= tol and _rel(spc["temporal"], spn["temporal"]) <= tol
    acc = [2, 3, 0, 1]
    O.spec_commit(pn, spn, 0, 1, slots, pos2, acc, track, 256, D)
    dt = R.DTYPE["f64"]
    t, c = pc["temporal"][0].astype(dt), pc["conv"][0].astype(dt)
    R.commit_arrays("f64", t, c, slots, pos2, acc, track, 256, spc["temporal"][0], spc["conv"][0])
    assert _rel(t, pn["temporal"][0]) <= tol
    assert np.array_equal(c, pn["conv"][0])


def test_copy_slots_is_a_gather():
    rng = np.random.default_rng(6)
    buf = rng.integers(0, 2 ** 16, size=(3, 10, 7, 5), dtype=np.uint16)
    src, dst = [1, 1, 4, -1, 7], [2, 3, 5, 6, 7]
    want = buf.copy()
    for s, d in zip(src, dst):
        if s >= 0 and d >= 0 and s != d:
            want[:, d] = buf[:, s]
    R.copy_slots_bytes(buf, src, dst)
    assert np.array_equal(buf, want)


def test_host_description():
    assert R.host_threads() >= 1
    assert isinstance(R.cpu_model(), str) and R.cpu_model()
