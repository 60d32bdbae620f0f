"""Pins for the CPU oracle: each check ties it to something other than itself
(an independent formulation, a closed form, an invariant the pages state, or a
number the pages print). CPU only."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import lin_state_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# Independent brute force: conv by numpy.convolve per channel, the update in
# explicit matrix form S_t = S_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
# ----------------------------------------------------------------------------

def brute_force(S0, cw0, x, w, g, beta, H, K, V, gate_mode, silu, l2, q_scale=1.0):
    C = x.shape[1]
    L = x.shape[0]
    y = np.zeros((L, C))
    for c in range(C):
        seq = np.concatenate([cw0[c], x[:, c]])
        y[:, c] = np.convolve(seq, w[c][::-1], mode="valid")
    if silu:
        y = y * (1.0 / (1.0 + np.exp(-y)))
    S = [S0[h].copy() for h in range(H)]
    outs = np.zeros((L, H, V))
    for t in range(L):
        for h in range(H):
            q = y[t, h * K:(h + 1) * K]
            k = y[t, H * K + h * K:H * K + (h + 1) * K]
            v = y[t, 2 * H * K + h * V:2 * H * K + (h + 1) * V]
            if l2:
                q = q / np.linalg.norm(np.append(q, 1e-3))  # sqrt(sum q^2 + 1e-6)
                k = k / np.linalg.norm(np.append(k, 1e-3))
            q = q * q_scale
            a = np.exp(g[t, h]) * np.ones(K) if gate_mode == O.GATE_PER_HEAD else np.exp(g[t, h])
            Dm = np.diag(a)
            b = beta[t, h]
            S[h] = S[h] @ Dm @ (np.eye(K) - b * np.outer(k, k)) + b * np.outer(v, k)
            outs[t, h] = S[h] @ q
    cw_end = np.concatenate([cw0, x.T], axis=1)[:, -3:]
    return np.stack(S), cw_end, outs


def _tiny_inputs(seed, H, K, V, L, gate_mode, warm=True):
    r = rng(seed)
    C = 2 * H * K + H * V
    x = r.standard_normal((L, C))
    w = r.standard_normal((C, 4)) * 0.5
    g = -np.log1p(np.exp(r.standard_normal((L, H) if gate_mode == 0 else (L, H, K))))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((L, H))))
    S0 = r.standard_normal((H, V, K)) * 0.3 if warm else np.zeros((H, V, K))
    cw0 = r.standard_normal((C, 3)) if warm else np.zeros((C, 3))
    return x, w, g, beta, S0, cw0


def _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, gate_mode, flags, q_scale=1.0,
                    dtype="f64"):
    C = x.shape[1]
    pool = O.make_pool(1, 4, H, K, V, C, state_dtype=dtype, conv_dtype=dtype)
    pool["temporal"][0, 1] = S0
    pool["conv"][0, 1] = cw0
    out, st = O.prefill(pool, 0, x, w, g, beta, [0, x.shape[0]], [0], [1], [1],
                        [], [0, 0], 0, gate_mode, flags, q_scale, out_dtype=dtype)
    assert st == 0
    return pool["temporal"][0, 1], pool["conv"][0, 1], out


@pytest.mark.parametrize("gate_mode", [O.GATE_PER_HEAD, O.GATE_PER_KEY])
@pytest.mark.parametrize("flags", [O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU, O.FLAG_QK_L2NORM, 0])
@pytest.mark.parametrize("K,V", [(4, 4), (8, 6)])
def test_matches_matrix_form_brute_force(gate_mode, flags, K, V):
    H, L = 2, 23
    x, w, g, beta, S0, cw0 = _tiny_inputs(1, H, K, V, L, gate_mode)
    S, cw, out = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, gate_mode, flags, 0.7)
    Sb, cwb, outb = brute_force(S0, cw0, x, w, g, beta, H, K, V, gate_mode,
                                bool(flags & O.FLAG_CONV_SILU),
                                bool(flags & O.FLAG_QK_L2NORM), 0.7)
    np.testing.assert_allclose(out, outb, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, Sb, rtol=1e-11, atol=1e-12)
    assert np.array_equal(cw, cwb)


def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = S_0 Diag(prod alpha), o_t = S_t q_t (closed form)."""
    H, K, V, L = 2, 8, 8, 17
    x, w, g, beta, S0, cw0 = _tiny_inputs(2, H, K, V, L, O.GATE_PER_KEY)
    beta[:] = 0.0
    w[:] = 0.0
    w[:, 3] = 1.0  # identity conv: q, k, v are the raw inputs
    S, _, out = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_KEY, 0)
    cum = np.cumsum(g, axis=0)  # [L][H][K]
    gam_T = np.exp(cum[-1])
    np.testing.assert_allclose(S, S0 * gam_T[:, None, :], rtol=1e-12)
    for t in [0, 5, L - 1]:
        q = x[t, :H * K].reshape(H, K)
        expect = np.einsum("hvk,hk->hv", S0 * np.exp(cum[t])[:, None, :], q)
        np.testing.assert_allclose(out[t], expect, rtol=1e-11, atol=1e-13)


def test_delta_rule_retrieval():
    """alpha = 1, beta = 1, unit k: after the token, S k = v exactly."""
    H, K, V, L = 2, 8, 5, 9
    x, w, g, beta, S0, cw0 = _tiny_inputs(3, H, K, V, L, O.GATE_PER_HEAD)
    g[:] = 0.0
    beta[:] = 1.0
    w[:] = 0.0
    w[:, 3] = 1.0
    for n in range(1, L + 1):
        S, _, _ = _run_oracle_one(S0, cw0, x[:n], w, g[:n], beta[:n], H, K, V,
                                  O.GATE_PER_HEAD, O.FLAG_QK_L2NORM)
        k = x[n - 1, H * K:2 * H * K].reshape(H, K)
        k = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
        v = x[n - 1, 2 * H * K:].reshape(H, V)
        # ||k||^2 = 1 - 1e-6 / (|k|^2 + 1e-6): retrieval holds up to that factor.
        got = np.einsum("hvk,hk->hv", S, k)
        np.testing.assert_allclose(got, v, rtol=2e-6, atol=2e-6)


def test_orthonormal_keys_sum_of_outer_products():
    """alpha = 1, beta = 1, S_0 = 0, orthonormal keys: S = sum_i v_i k_i^T."""
    H, K, V = 1, 8, 3
    r = rng(4)
    Q, _ = np.linalg.qr(r.standard_normal((K, K)))
    L = K
    C = 2 * H * K + H * V
    x = np.zeros((L, C))
    x[:, H * K:2 * H * K] = Q.T  # token i key = column i of Q (unit norm)
    x[:, 2 * H * K:] = r.standard_normal((L, V))
    x[:, :H * K] = r.standard_normal((L, K))
    w = np.zeros((C, 4))
    w[:, 3] = 1.0
    g = np.zeros((L, H))
    beta = np.ones((L, H))
    S, _, out = _run_oracle_one(np.zeros((H, V, K)), np.zeros((C, 3)), x, w, g, beta,
                                H, K, V, O.GATE_PER_HEAD, 0)
    expect = sum(np.outer(x[i, 2 * K:], Q[:, i]) for i in range(L))
    np.testing.assert_allclose(S[0], expect, atol=1e-12)


def test_scalar_head_closed_form():
    """K = V = 1: s_T = s_0 prod_j a_j (1 - b_j k_j^2) + sum_i b_i v_i k_i prod_{j>i} a_j (1 - b_j k_j^2)."""
    H, K, V, L = 3, 1, 1, 30
    x, w, g, beta, S0, cw0 = _tiny_inputs(5, H, K, V, L, O.GATE_PER_KEY)
    w[:] = 0.0
    w[:, 3] = 1.0
    S, _, _ = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_KEY, 0)
    for h in range(H):
        k = x[:, H + h]
        v = x[:, 2 * H + h]
        a = np.exp(g[:, h, 0])
        b = beta[:, h]
        f = a * (1 - b * k * k)
        total = S0[h, 0, 0] * np.prod(f)
        for i in range(L):
            total += b[i] * v[i] * k[i] * np.prod(f[i + 1:])
        np.testing.assert_allclose(S[h, 0, 0], total, rtol=1e-11)


def _ssd_quadratic_form(S0, x, g, beta, H, K, V, gate_mode):
    """The additive recurrence unrolled (the state-space / masked-attention
    duality): with b_t = sum_{r<=t} log alpha_r per key channel,
        o_t = sum_{s<=t} beta_s v_s sum_c q_tc k_sc exp(b_tc - b_sc)
              + S_0 (exp(b_t) . q_t),
        S_T = S_0 Diag(exp(b_T)) + sum_s beta_s v_s (exp(b_T - b_s) . k_s)^T.
    q, k, v are the raw inputs (identity conv, no normalisation)."""
    L = x.shape[0]
    q = x[:, :H * K].reshape(L, H, K)
    k = x[:, H * K:2 * H * K].reshape(L, H, K)
    v = x[:, 2 * H * K:].reshape(L, H, V)
    lg = np.repeat(g[:, :, None], K, axis=2) if gate_mode == O.GATE_PER_HEAD else g
    b = np.cumsum(lg, axis=0)  # [L][H][K]
    out = np.zeros((L, H, V))
    for t in range(L):
        for s_ in range(t + 1):
            w = np.einsum("hc,hc->h", q[t] * np.exp(b[t] - b[s_]), k[s_])
            out[t] += (beta[s_] * w)[:, None] * v[s_]
        out[t] += np.einsum("hvk,hk->hv", S0, np.exp(b[t]) * q[t])
    S = S0 * np.exp(b[-1])[:, None, :]
    for s_ in range(L):
        S += beta[s_][:, None, None] * v[s_][:, :, None] * (np.exp(b[-1] - b[s_]) * k[s_])[:, None, :]
    return S, out


@pytest.mark.parametrize("gate_mode", [O.GATE_PER_HEAD, O.GATE_PER_KEY])
def test_additive_matches_ssd_quadratic_form(gate_mode):
    """FLAG_UPDATE_ADDITIVE (S' = S Diag(alpha) + beta v k^T) against its
    unrolled quadratic form, warm start; the delta-rule result differs."""
    H, K, V, L = 2, 6, 5, 19
    x, w, g, beta, S0, cw0 = _tiny_inputs(11, H, K, V, L, gate_mode)
    w[:] = 0.0
    w[:, 3] = 1.0
    S, cw, out = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, gate_mode,
                                 O.FLAG_UPDATE_ADDITIVE)
    Se, oute = _ssd_quadratic_form(S0, x, g, beta, H, K, V, gate_mode)
    np.testing.assert_allclose(out, oute, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, Se, rtol=1e-11, atol=1e-12)
    Sd, _, outd = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, gate_mode, 0)
    assert not np.allclose(outd, oute, rtol=1e-3, atol=1e-3)


def test_additive_unit_decay_is_sum_of_outer_products():
    """alpha = 1, S_0 = 0, any keys: S = sum_i beta_i v_i k_i^T (no interference
    term, unlike the delta rule), through the conv and SiLU path."""
    H, K, V, L = 1, 5, 3, 9
    x, w, g, beta, _, _ = _tiny_inputs(12, H, K, V, L, O.GATE_PER_HEAD, warm=False)
    g[:] = 0.0
    S, _, _ = _run_oracle_one(np.zeros((H, V, K)), np.zeros((x.shape[1], 3)), x, w, g, beta,
                              H, K, V, O.GATE_PER_HEAD, O.FLAG_UPDATE_ADDITIVE | O.FLAG_CONV_SILU)
    C = x.shape[1]
    y = np.zeros((L, C))
    for c in range(C):
        y[:, c] = np.convolve(np.concatenate([np.zeros(3), x[:, c]]), w[c][::-1], mode="valid")
    y = y / (1.0 + np.exp(-y))
    expect = sum(beta[i, 0] * np.outer(y[i, 2 * K:], y[i, K:2 * K]) for i in range(L))
    np.testing.assert_allclose(S[0], expect, rtol=1e-12, atol=1e-13)


def test_gdn_equals_kda_with_broadcast_gate():
    H, K, V, L = 2, 6, 6, 15
    x, w, g, beta, S0, cw0 = _tiny_inputs(6, H, K, V, L, O.GATE_PER_HEAD)
    f = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU
    a = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_HEAD, f)
    b = _run_oracle_one(S0, cw0, x, w, np.repeat(g[:, :, None], K, 2), beta, H, K, V,
                        O.GATE_PER_KEY, f)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_conv_identity_and_window():
    """w = e_3 gives y = x; the conv state after a run is the last 3 inputs,
    bit for bit, including runs shorter than 3 tokens."""
    H, K, V = 1, 4, 4
    for L in [1, 2, 3, 7]:
        x, w, g, beta, S0, cw0 = _tiny_inputs(7 + L, H, K, V, L, O.GATE_PER_HEAD)
        w[:] = 0.0
        w[:, 3] = 1.0
        _, cw, _ = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_HEAD, 0)
        window = np.concatenate([cw0, x.T], axis=1)[:, -3:]
        assert np.array_equal(cw, window)
    # A random w matches numpy.convolve through the q channel path:
    # with alpha = 1, beta = 0, S_0 = I-like, o = S_0 q gives q back.
    H, K, V, L = 1, 4, 4, 12
    x, w, g, beta, S0, cw0 = _tiny_inputs(20, H, K, V, L, O.GATE_PER_HEAD)
    g[:] = 0.0
    beta[:] = 0.0
    S0 = np.eye(4)[None]
    _, _, out = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_HEAD, 0)
    for c in range(K):
        seq = np.concatenate([cw0[c], x[:, c]])
        np.testing.assert_allclose(out[:, 0, c], np.convolve(seq, w[c][::-1], "valid"),
                                   rtol=1e-13, atol=1e-14)


def _tiny_pool_run(x, w, g, beta, lengths, prefixes, slots, warm, tracks, cu_track,
                   stride, H, K, V, dtype="f64", pool=None, gate=O.GATE_PER_HEAD,
                   chunk_align=64):
    C = x.shape[1]
    if pool is None:
        pool = O.make_pool(1, 16, H, K, V, C, state_dtype=dtype, conv_dtype=dtype)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    out, st = O.prefill(pool, 0, x, w, g, beta, cu, prefixes, slots, warm, tracks,
                        cu_track, stride, gate, O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU,
                        1.0, dtype, chunk_align=chunk_align)
    assert st == 0
    return pool, out


def test_warm_start_from_checkpoint_equals_cold_run():
    """Qwen3.5 Linear-State Prefix Cache 2.2: a checkpoint at a chunk boundary
    is an exact snapshot; continuing from it reproduces the cold run."""
    H, K, V, T, b = 2, 8, 8, 200, 128
    x, w, g, beta, _, _ = _tiny_inputs(30, H, K, V, T, O.GATE_PER_KEY)
    pool, out_cold = _tiny_pool_run(x, w, g, beta, [T], [0], [1], [0], [5, 6], [0, 2],
                                    64, H, K, V, gate=O.GATE_PER_KEY)
    # boundaries 64 -> slot 5, 128 -> slot 6
    S_cold, cw_cold = pool["temporal"][0, 1].copy(), pool["conv"][0, 1].copy()
    pool["temporal"][0, 2] = pool["temporal"][0, 6]
    pool["conv"][0, 2] = pool["conv"][0, 6]
    pool, out_warm = _tiny_pool_run(x[b:], w, g[b:], beta[b:], [T - b], [b], [2], [1],
                                    [], [0, 0], 64, H, K, V, pool=pool, gate=O.GATE_PER_KEY)
    assert np.array_equal(out_warm, out_cold[b:])
    assert np.array_equal(pool["temporal"][0, 2], S_cold)
    assert np.array_equal(pool["conv"][0, 2], cw_cold)


def test_deepest_checkpoint_suffices():
    """Restoring the deepest checkpoint (b2) equals restoring an earlier one
    (b1) and running b1..b2 (Qwen3.5 Linear-State Prefix Cache 2.2)."""
    H, K, V, T = 1, 8, 8, 256
    x, w, g, beta, _, _ = _tiny_inputs(31, H, K, V, T, O.GATE_PER_HEAD)
    pool, _ = _tiny_pool_run(x, w, g, beta, [T], [0], [1], [0], [5, 6, 7, 8], [0, 4],
                             64, H, K, V)
    b1, b2 = 64, 192
    # path 1: from the checkpoint at b2 (slot 7)
    pool["temporal"][0, 2] = pool["temporal"][0, 7]
    pool["conv"][0, 2] = pool["conv"][0, 7]
    pool, o1 = _tiny_pool_run(x[b2:], w, g[b2:], beta[b2:], [T - b2], [b2], [2], [1],
                              [], [0, 0], 64, H, K, V, pool=pool)
    # path 2: from b1 (slot 5), run to b2, then on to T
    pool["temporal"][0, 3] = pool["temporal"][0, 5]
    pool["conv"][0, 3] = pool["conv"][0, 5]
    pool, _ = _tiny_pool_run(x[b1:b2], w, g[b1:b2], beta[b1:b2], [b2 - b1], [b1], [3], [1],
                             [], [0, 0], 64, H, K, V, pool=pool)
    pool, o2 = _tiny_pool_run(x[b2:], w, g[b2:], beta[b2:], [T - b2], [b2], [3], [1],
                              [], [0, 0], 64, H, K, V, pool=pool)
    assert np.array_equal(o1, o2)
    assert np.array_equal(pool["temporal"][0, 2], pool["temporal"][0, 3])


def test_placement_long_request_1200():
    gold = _load("placement_examples.json")["long_request"]
    A, B, C, D = (gold["slots"][k] for k in "ABCD")
    H, K, V, T = 1, 4, 4, 1200
    x, w, g, beta, _, _ = _tiny_inputs(32, H, K, V, T, O.GATE_PER_HEAD)
    Cc = x.shape[1]
    pool = O.make_pool(1, 8, H, K, V, Cc, state_dtype="f64", conv_dtype="f64", fill=-7.0)
    track_list = [B, C]
    nxt = 0
    pos = 0
    for n in gold["calls"]:
        lst = track_list[nxt:] + track_list[:nxt]  # host-side ping-pong rotation
        _tiny_pool_run(x[pos:pos + n], w, g[pos:pos + n], beta[pos:pos + n], [n], [pos],
                       [A], [1 if pos else 0], lst, [0, 2], gold["chunk"], H, K, V,
                       pool=pool)
        if (pos + n) // gold["chunk"] > pos // gold["chunk"]:
            nxt ^= 1
        pos += n
    O.copy_slots(pool, [A], [D], 0, 1)
    for name, ntok in gold["expect"].items():
        Sb, cwb, _ = brute_force(np.zeros((H, V, K)), np.zeros((Cc, 3)), x[:ntok], w,
                                 g[:ntok], beta[:ntok], H, K, V, O.GATE_PER_HEAD, True, True)
        s = gold["slots"][name]
        np.testing.assert_allclose(pool["temporal"][0, s], Sb, rtol=1e-10, atol=1e-12)
        assert np.array_equal(pool["conv"][0, s], cwb)
    assert np.array_equal(pool["temporal"][0, D], pool["temporal"][0, A])


def test_placement_toy_chunked_prefill():
    gold = _load("placement_examples.json")["toy_chunked"]
    H, K, V, T = 1, 4, 4, 8
    x, w, g, beta, _, _ = _tiny_inputs(33, H, K, V, T, O.GATE_PER_HEAD)
    Cc = x.shape[1]
    pool = O.make_pool(1, 128, H, K, V, Cc, state_dtype="f64", conv_dtype="f64")
    pos = 0
    for n, ts in zip(gold["calls"], gold["track_slot_per_call"]):
        _tiny_pool_run(x[pos:pos + n], w, g[pos:pos + n], beta[pos:pos + n], [n], [pos],
                       [1], [1 if pos else 0], [ts], [0, 1], gold["chunk"], H, K, V,
                       pool=pool, chunk_align=gold["chunk"])
        pos += n
    for s, ntok in gold["expect_tokens_in_state"].items():
        Sb, _, _ = brute_force(np.zeros((H, V, K)), np.zeros((Cc, 3)), x[:ntok], w,
                               g[:ntok], beta[:ntok], H, K, V, O.GATE_PER_HEAD, True, True)
        np.testing.assert_allclose(pool["temporal"][0, int(s)], Sb, rtol=1e-10, atol=1e-12)


def test_short_request_no_track():
    gold = _load("placement_examples.json")["short_request"]
    H, K, V, T = 1, 4, 4, gold["length"]
    x, w, g, beta, _, _ = _tiny_inputs(34, H, K, V, T, O.GATE_PER_HEAD)
    pool = O.make_pool(1, 8, H, K, V, x.shape[1], state_dtype="f64", conv_dtype="f64",
                       fill=-3.0)
    _tiny_pool_run(x, w, g, beta, [T], [0], [1], [0], [2, 3], [0, 2], gold["chunk"],
                   H, K, V, pool=pool)
    assert np.all(pool["temporal"][0, 2:4] == -3.0)
    assert np.all(pool["conv"][0, 2:4] == -3.0)


def test_decode_track_positions_match_page_example():
    gold = _load("decode_track_interval.json")
    H, K, V = 1, 4, 4
    C = 2 * H * K + H * V
    pool = O.make_pool(1, 4, H, K, V, C, state_dtype="f32", conv_dtype="f32")
    r = rng(40)
    w = r.standard_normal((C, 4)) * 0.5
    hits = []
    pos = gold["prompt_len"]
    n_steps = gold["decode_tokens_processed"][-1] + 10
    for step in range(1, n_steps + 1):
        pool["temporal"][0, 2] = np.nan
        x = r.standard_normal((1, 1, C))
        g = -np.log1p(np.exp(r.standard_normal((1, 1, H))))
        b = np.full((1, 1, H), 0.5)
        O.decode(pool, 0, x, w, g, b, [1], [pos], [2], gold["interval"], O.GATE_PER_HEAD,
                 O.FLAG_QK_L2NORM)
        if not np.isnan(pool["temporal"][0, 2]).any():
            hits.append(step)
            assert np.array_equal(pool["temporal"][0, 2], pool["temporal"][0, 1])
        pos += 1
    assert hits == gold["decode_tokens_processed"]
    assert [gold["prompt_len"] + h for h in hits] == gold["checkpoint_total_lengths"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spec_commit_equals_sequential_decode(dtype):
    """MambaRadixCache page 9.4: the accepted path is a linear chain, so after
    commit the slot equals running the accepted tokens one by one; 8.4:
    main_state = buffer[accepted step]. Track crossing 256 (8.6)."""
    H, K, V, D = 2, 8, 8, 4
    C = 2 * H * K + H * V
    r = rng(41)
    w = r.standard_normal((C, 4)) * 0.5
    S0 = O.round_to(r.standard_normal((H, V, K)) * 0.2, dtype)
    c0 = O.round_to(r.standard_normal((C, 3)), dtype)
    x = O.round_to(r.standard_normal((1, D, C)), dtype)
    g = -np.log1p(np.exp(r.standard_normal((1, D, H, K))))
    b = 1 / (1 + np.exp(-r.standard_normal((1, D, H))))
    f = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU
    for pos in [100, 254]:
        for acc in range(0, D + 1):
            pa = O.make_pool(1, 6, H, K, V, C, state_dtype=dtype, conv_dtype=dtype, fill=-1)
            pa["temporal"][0, 1] = S0
            pa["conv"][0, 1] = c0
            pb = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pa.items()}
            spec = O.make_spec_buffer(1, 1, D, H, K, V, C)
            out_v, st = O.decode(pa, 0, x, w, g, b, [1], [pos], [3], 256, O.GATE_PER_KEY,
                                 f, spec=spec)
            assert st == 0
            assert np.array_equal(pa["temporal"][0, 1], S0)  # verify leaves the slot
            O.spec_commit(pa, spec, 0, 1, [1], [pos], [acc], [3], 256, D)
            for j in range(acc):
                out_s, _ = O.decode(pb, 0, x[:, j:j + 1], w, g[:, j:j + 1], b[:, j:j + 1],
                                    [1], [pos + j], [3], 256, O.GATE_PER_KEY, f)
                assert np.array_equal(out_s[0, 0], out_v[0, j])
            assert np.array_equal(pa["temporal"][0, 1], pb["temporal"][0, 1])
            assert np.array_equal(pa["conv"][0, 1], pb["conv"][0, 1])
            assert np.array_equal(pa["temporal"][0, 3], pb["temporal"][0, 3])
            if pos == 254 and acc >= 2:
                assert np.array_equal(pa["temporal"][0, 3], spec["temporal"][0, 0, 1])
            else:
                assert np.all(pa["temporal"][0, 3] == -1)


@pytest.mark.parametrize("gate_mode", [O.GATE_PER_HEAD, O.GATE_PER_KEY])
def test_verify_outputs_is_a_prefill_of_the_drafts(gate_mode):
    """A verify that keeps no per-step states (Kimi-K3 notes "ReplaySSM";
    MambaRadixCache page 9.2 - 9.10) carries the state unrounded across its
    drafts: on a bf16 pool its outputs equal those of a prefill of the same
    tokens from the slot (which carries the state unrounded inside the call,
    storing nothing); with unrounded storage they equal the per-step verify's
    outputs (whose per-token rounding is then the identity), and with bf16
    storage they differ from them only by that rounding. The pool is left
    as it was."""
    H, K, V, D = 2, 8, 6, 5
    C = 2 * H * K + H * V
    r = rng(43)
    w = r.standard_normal((C, 4)) * 0.5
    x = O.round_to(r.standard_normal((2, D, C)), "bf16")
    g = -np.log1p(np.exp(r.standard_normal((2, D, H) if gate_mode == O.GATE_PER_HEAD else (2, D, H, K))))
    b = 1 / (1 + np.exp(-r.standard_normal((2, D, H))))
    f = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU
    for dtype in ("bf16", "f64"):
        pool = O.make_pool(1, 5, H, K, V, C, state_dtype=dtype, conv_dtype=dtype)
        pool["temporal"][0, 1:3] = O.round_to(r.standard_normal((2, H, V, K)) * 0.2, dtype)
        pool["conv"][0, 1:3] = O.round_to(r.standard_normal((2, C, 3)), dtype)
        before = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pool.items()}
        out, st = O.verify_outputs(pool, 0, x, w, g, b, [1, 2], gate_mode, f)
        assert st == 0
        assert np.array_equal(pool["temporal"], before["temporal"])
        assert np.array_equal(pool["conv"], before["conv"])
        for req in range(2):
            pp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in before.items()}
            op, _ = O.prefill(pp, 0, x[req], w, g[req], b[req], [0, D], [0], [1 + req], [1], [],
                              [0, 0], 0, gate_mode, f)
            assert np.array_equal(op, out[req])
        pv = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in before.items()}
        spec = O.make_spec_buffer(1, 2, D, H, K, V, C)
        ov, _ = O.decode(pv, 0, x, w, g, b, [1, 2], [0, 0], None, 0, gate_mode, f, spec=spec)
        if dtype == "f64":
            assert np.array_equal(ov, out)
        else:
            assert not np.array_equal(ov, out)
            assert np.linalg.norm(ov - out) <= 2e-2 * np.linalg.norm(out)


# a draft tree in the shape of the MambaRadixCache page's example (9.6): two
# roots, children of both, a grandchild; parent index per draft, -1 = the slot
TREE_PARENT = [-1, -1, 0, 0, 1, 2, 2, 5]


def _tree_setup(seed, dtype, D):
    H, K, V = 2, 8, 8
    C = 2 * H * K + H * V
    r = rng(seed)
    w = r.standard_normal((C, 4)) * 0.5
    S0 = O.round_to(r.standard_normal((H, V, K)) * 0.2, dtype)
    c0 = O.round_to(r.standard_normal((C, 3)), dtype)
    x = O.round_to(r.standard_normal((1, D, C)), dtype)
    g = -np.log1p(np.exp(r.standard_normal((1, D, H, K))))
    b = 1 / (1 + np.exp(-r.standard_normal((1, D, H))))
    pool = O.make_pool(1, 6, H, K, V, C, state_dtype=dtype, conv_dtype=dtype, fill=-1)
    pool["temporal"][0, 1] = S0
    pool["conv"][0, 1] = c0
    return H, K, V, C, w, x, g, b, pool


def _path(parent, node):
    p = []
    while node >= 0:
        p.insert(0, node)
        node = parent[node]
    return p


@pytest.mark.parametrize("dtype", ["f64", "bf16"])
def test_tree_verify_paths_equal_linear_chains(dtype):
    """MambaRadixCache page 8.3 / 9.6: each draft of a tree starts from its
    parent's state (retrieve_parent_token). Every node's output and state
    equal the linear chain run along its root-to-node path, and a chain given
    as parents (j - 1) equals the plain verify exactly."""
    D = len(TREE_PARENT)
    H, K, V, C, w, x, g, b, pool = _tree_setup(61, dtype, D)
    f = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU
    spec = O.make_spec_buffer(1, 1, D, H, K, V, C)
    out_t, st = O.decode(pool, 0, x, w, g, b, [1], [0], None, 0, O.GATE_PER_KEY, f, spec=spec,
                         parent=[TREE_PARENT])
    assert st == 0
    for node in range(D):
        path = _path(TREE_PARENT, node)
        pc = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pool.items()}
        sc = O.make_spec_buffer(1, 1, len(path), H, K, V, C)
        if len(path) == 1:
            out_c, _ = O.decode(pc, 0, x[:, path], w, g[:, path], b[:, path], [1], [0], None, 0,
                                O.GATE_PER_KEY, f)
            # a single decode writes the slot: compare against it
            assert np.array_equal(pc["temporal"][0, 1], spec["temporal"][0, 0, node])
        else:
            out_c, _ = O.decode(pc, 0, x[:, path], w, g[:, path], b[:, path], [1], [0], None, 0,
                                O.GATE_PER_KEY, f, spec=sc)
            assert np.array_equal(sc["temporal"][0, 0, -1], spec["temporal"][0, 0, node])
            assert np.array_equal(sc["conv"][0, 0, -1], spec["conv"][0, 0, node])
        assert np.array_equal(out_c[0, -1], out_t[0, node])
    # a chain written as parents is the plain verify
    chain = [[j - 1 for j in range(D)]]
    s1, s2 = O.make_spec_buffer(1, 1, D, H, K, V, C), O.make_spec_buffer(1, 1, D, H, K, V, C)
    o1, _ = O.decode(pool, 0, x, w, g, b, [1], [0], None, 0, O.GATE_PER_KEY, f, spec=s1, parent=chain)
    o2, _ = O.decode(pool, 0, x, w, g, b, [1], [0], None, 0, O.GATE_PER_KEY, f, spec=s2)
    assert np.array_equal(o1, o2) and np.array_equal(s1["temporal"], s2["temporal"])


def test_tree_commit_equals_chain_commit_and_rejects_bad_trees():
    """The accepted path of a tree is a linear chain (MambaRadixCache page
    9.9): committing node a equals committing a chain verify of a's path with
    accept_len = its depth, boundary snapshots included; a parent outside
    [-1, j) or an accepted node outside [-1, n_draft) is rejected."""
    D = len(TREE_PARENT)
    H, K, V, C, w, x, g, b, pool = _tree_setup(62, "bf16", D)
    f = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU
    for pos in [100, 254, 255]:
        for node in [-1, 0, 3, 4, 7]:
            pa = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pool.items()}
            spec = O.make_spec_buffer(1, 1, D, H, K, V, C)
            O.decode(pa, 0, x, w, g, b, [1], [pos], None, 0, O.GATE_PER_KEY, f, spec=spec,
                     parent=[TREE_PARENT])
            st = O.spec_commit(pa, spec, 0, 1, [1], [pos], None, [3], 256, D, parent=[TREE_PARENT],
                               accept_node=[node])
            assert st == 0
            path = _path(TREE_PARENT, node)
            pb = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pool.items()}
            if path:
                sc = O.make_spec_buffer(1, 1, max(2, len(path)), H, K, V, C)
                xp = x[:, path + path[-1:]] if len(path) == 1 else x[:, path]
                gp = g[:, path + path[-1:]] if len(path) == 1 else g[:, path]
                bp = b[:, path + path[-1:]] if len(path) == 1 else b[:, path]
                O.decode(pb, 0, xp, w, gp, bp, [1], [pos], None, 0, O.GATE_PER_KEY, f, spec=sc)
                O.spec_commit(pb, sc, 0, 1, [1], [pos], [len(path)], [3], 256, sc["temporal"].shape[2])
            for k in ("temporal", "conv"):
                assert np.array_equal(pa[k], pb[k]), (pos, node, k)
    bad = [-1, 0, 2, 0, 1, 2, 2, 5]  # draft 2's parent is itself
    st = O.decode(pool, 0, x, w, g, b, [1], [0], None, 0, O.GATE_PER_KEY, f,
                  spec=O.make_spec_buffer(1, 1, D, H, K, V, C), parent=[bad])[1]
    assert st == O.ST_BAD_TREE
    st = O.spec_commit(pool, O.make_spec_buffer(1, 1, D, H, K, V, C), 0, 1, [1], [0], None, None, 0,
                       D, parent=[TREE_PARENT], accept_node=[D])
    assert st == O.ST_BAD_TREE


def test_copy_slots_is_a_gather():
    r = rng(50)
    pool = O.make_pool(3, 10, 2, 4, 4, 24)
    pool["temporal"][:] = r.standard_normal(pool["temporal"].shape)
    pool["conv"][:] = r.standard_normal(pool["conv"].shape)
    before = {k: pool[k].copy() for k in ("temporal", "conv")}
    src, dst = [2, 2, 7, -1, 5], [3, 4, 1, 6, 5]
    assert O.copy_slots(pool, src, dst, 1, 3) == 0
    for k in ("temporal", "conv"):
        exp = before[k].copy()
        exp[1:3, [3, 4, 1]] = before[k][1:3, [2, 2, 7]]
        assert np.array_equal(pool[k], exp)
    # aliasing under VALIDATE: dst 3 also a src
    st = O.copy_slots(pool, [3, 8], [9, 3], 0, 3, O.FLAG_VALIDATE)
    assert st & O.ST_COPY_ALIAS
    assert O.copy_slots(pool, [0], [10], 0, 3) & O.ST_BAD_SLOT


def test_restore_semantics():
    """Qwen3.5 Linear-State Prefix Cache 6.4: RESTORED -> 1, COLD_START -> 0,
    no restore request -> untouched; -1 live id is padding (6.1 defaults)."""
    r = rng(51)
    pool = O.make_pool(2, 8, 1, 4, 4, 12)
    pool["temporal"][:] = r.standard_normal(pool["temporal"].shape)
    pool["conv"][:] = r.standard_normal(pool["conv"].shape)
    before = pool["temporal"].copy()
    ops = [(1, 1, 5), (2, 1, -1), (3, 0, 6), (-1, 1, 5), (4, 1, 99)]
    his = np.array([7, 7, 7, 7, 7], np.int64)
    O.restore(pool, ops, his)
    assert his.tolist() == [1, 0, 7, 7, 0]
    assert np.array_equal(pool["temporal"][:, 1], before[:, 5])
    assert np.array_equal(pool["temporal"][:, 2], before[:, 2])
    assert np.array_equal(pool["temporal"][:, 3], before[:, 3])


def test_slot_bytes_match_page_figures():
    gold = _load("state_sizes.json")
    k3 = gold["kimi_k3_tp8"]
    ssm = O.slot_bytes(k3["num_layers"], k3["num_heads"], k3["head_k"], k3["head_v"], 0, 4, 2, 2)
    conv = O.slot_bytes(k3["num_layers"], 0, 0, 0, k3["conv_channels"], 4, 2, 2)
    assert ssm == k3["ssm_bytes_per_slot"] == eval(k3["ssm_bytes_per_slot_formula"])
    assert conv == k3["conv_bytes_per_slot"] == eval(k3["conv_bytes_per_slot_formula"])
    assert round(ssm / 2**20, 1) == k3["ssm_mb_printed"]
    assert round(conv / 2**20, 2) == k3["conv_mb_printed"]
    assert round((round(ssm / 2**20, 1) + round(conv / 2**20, 2)) * 8, 1) == k3["tp8_total_mb_printed"]
    qn = gold["qwen3_next_layer"]
    layer = O.slot_bytes(1, qn["num_heads"], qn["head_k"], qn["head_v"], 0, 4, qn["state_esize"], 2)
    assert layer / 2**20 == qn["ssm_mb_printed"]
    assert 32 * layer / 2**20 == qn["fork_mb_printed_32_layers"]
    al = gold["allocation_log"]
    for dt, es in (("fp32", 4), ("bf16", 2)):
        n = al[dt]["max_mamba_cache_size"] + 1  # size + 1 slots are allocated
        ssm_b = n * O.slot_bytes(69, 12, 128, 128, 0, 4, es, 2)
        conv_b = n * O.slot_bytes(69, 0, 0, 0, 4608, 4, es, 2)
        assert round(ssm_b / 2**30, 2) == al[dt]["ssm_gb_printed"]
        assert round(conv_b / 2**30, 2) == al[dt]["conv_gb_printed"]


def test_bf16_rounding_matches_torch():
    x = rng(60).standard_normal(100000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, np.float32([1.00390625, 1.01171875, -1.00390625, 0.0, 1e-39])])
    ours = O.round_to(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


# ----------------------------------------------------------------------------
# Planted mistakes: each mutant of the update must be caught by the brute force.
# ----------------------------------------------------------------------------

def _mutant(kind):
    real = O.token_step

    def step(S, cw, x_t, conv_w, g_t, beta_t, H, K, V, gate_mode, flags, q_scale):
        if kind == "no_decay_in_delta":
            alpha = np.exp(g_t)[:, None] * np.ones((H, K)) if gate_mode == 0 else np.exp(g_t)
            S_new, cw_new, _ = real(S, cw, x_t, conv_w, g_t, beta_t, H, K, V, gate_mode,
                                    flags, q_scale)
            y = conv_w[:, 3] * x_t + (conv_w[:, :3] * cw).sum(1)
            if flags & O.FLAG_CONV_SILU:
                y = y / (1 + np.exp(-y))
            k = y[H * K:2 * H * K].reshape(H, K)
            v = y[2 * H * K:].reshape(H, V)
            q = y[:H * K].reshape(H, K)
            if flags & O.FLAG_QK_L2NORM:
                k = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
                q = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6)
            d = beta_t[:, None] * (v - np.einsum("hvk,hk->hv", S, k))
            S2 = S * alpha[:, None, :] + d[:, :, None] * k[:, None, :]
            return S2, cw_new, np.einsum("hvk,hk->hv", S2, q * q_scale)
        if kind == "output_before_update":
            S_new, cw_new, _ = real(S, cw, x_t, conv_w, g_t, beta_t, H, K, V, gate_mode,
                                    flags, q_scale)
            _, _, o_prev = real(S, cw, x_t, conv_w, g_t, beta_t * 0, H, K, V, gate_mode,
                                flags, q_scale)
            return S_new, cw_new, o_prev
        if kind == "conv_taps_reversed":
            return real(S, cw, x_t, conv_w[:, ::-1], g_t, beta_t, H, K, V, gate_mode,
                        flags, q_scale)
        raise ValueError(kind)
    return step


@pytest.mark.parametrize("kind", ["no_decay_in_delta", "output_before_update",
                                  "conv_taps_reversed"])
def test_brute_force_catches_planted_mistake(kind, monkeypatch):
    H, K, V, L = 2, 4, 4, 12
    x, w, g, beta, S0, cw0 = _tiny_inputs(70, H, K, V, L, O.GATE_PER_KEY)
    monkeypatch.setattr(O, "token_step", _mutant(kind))
    S, _, out = _run_oracle_one(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_KEY,
                                O.FLAG_QK_L2NORM)
    Sb, _, outb = brute_force(S0, cw0, x, w, g, beta, H, K, V, O.GATE_PER_KEY, False, True)
    assert not np.allclose(out, outb, rtol=1e-6, atol=1e-8)
