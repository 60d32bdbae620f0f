"""The seeded input generators (workloads/) on the CPU: the same seed and
name give the same tensor, different names independent ones, and each recipe
stays in the ranges the workloads are specified with."""

import torch

import workloads as W


def test_streams_are_seeded_and_independent():
    a = W.randn((4096,), 7, "x")
    assert torch.equal(a, W.randn((4096,), 7, "x"))
    b = W.randn((4096,), 7, "y")
    c = W.randn((4096,), 8, "x")
    for other in (b, c):
        corr = float(torch.corrcoef(torch.stack([a, other]))[0, 1])
        assert abs(corr) < 0.06, corr
    assert abs(float(a.mean())) < 0.06 and abs(float(a.std()) - 1.0) < 0.05


def test_gate_recipes():
    g = W.gate_log_decay_uniform((20000,), 0, "gu")
    assert float(g.min()) >= -0.1 and float(g.max()) <= 0.0
    s = W.gate_log_decay_softplus((20000,), 0, "gs")
    assert float(s.max()) < 0.0  # alpha = exp(g) in (0, 1)
    # -softplus(z), z ~ N(0, 1): the median is -softplus(0) = -log 2
    assert abs(float(s.median()) + 0.6931) < 0.03
    b = W.beta_sigmoid((20000,), 0, "b")
    assert float(b.min()) > 0.0 and float(b.max()) < 1.0 and abs(float(b.median()) - 0.5) < 0.02


def test_ssd_gates_recipe():
    """dt = softplus(N(0,1) - 3) per (token, head), A = -U[1, 16] per head,
    g = dt A, beta = dt."""
    T, H = 20000, 8
    g, beta = W.ssd_gates((T, H), 0, "ssd")
    assert g.shape == beta.shape == (T, H)
    assert float(beta.min()) > 0.0
    # median of softplus(z - 3) is softplus(-3) = log(1 + e^-3)
    assert abs(float(beta.median()) - 0.048587) < 0.004
    A = g / beta  # the per-head rate, the same in every row
    assert torch.allclose(A, A[:1].expand_as(A), rtol=1e-5)
    assert float(A.min()) >= -16.0 and float(A.max()) <= -1.0


def test_kimi_k3_lengths_and_prefixes():
    L, P = W.kp_lengths(0)
    assert len(L) == len(P) == 32
    assert all(1024 <= l <= 16384 for l in L)
    for r, (l, p) in enumerate(zip(L, P)):
        if r < 16:
            assert p % 64 == 0 and 64 <= p < l
        else:
            assert p == 0
    assert (L, P) == W.kp_lengths(0)


def test_prefill_batch_shapes():
    dims = W.LayerDims(num_heads=3, head_k=16, head_v=16)
    b = W.make_prefill_batch(dims, [100, 70, 5], W.GATE_PER_KEY, dtype=torch.bfloat16, seed=1,
                             prefixes=[64, 0, 128], warm=[1, 0, 1], tag="wl")
    assert b.x.shape == (175, dims.conv_channels) and b.x.dtype == torch.bfloat16
    assert dims.conv_channels == 2 * 3 * 16 + 3 * 16
    assert b.conv_w.shape == (dims.conv_channels, 4)
    assert b.g.shape == (175, 3, 16) and b.g.dtype == torch.float32
    assert b.beta.shape == (175, 3)
    assert b.cu_seqlens.tolist() == [0, 100, 170, 175]
    assert b.prefix_len.tolist() == [64, 0, 128]
    assert b.has_initial_state.tolist() == [1, 0, 1]
    h = W.make_prefill_batch(dims, [40], W.GATE_PER_HEAD, seed=1, gate="ssd", tag="wl2")
    assert h.g.shape == (40, 3) and float(h.g.max()) < 0.0 and float(h.beta.min()) > 0.0


def test_slot_bytes_of_the_named_shapes():
    """Kimi-K3 TP8 shard: 12 x 128 x 128 bf16 state + [4608][3] bf16 window per
    layer-slot; Qwen3.5-style GDN: 32 x 128 x 128 fp32 state per layer."""
    assert W.KIMI_K3_TP8.conv_channels == 4608
    assert W.state_bytes(W.KIMI_K3_TP8, 2, 2) == 393216 + 27648
    assert W.QWEN35_GDN.conv_channels == 12288
    assert W.state_bytes(W.QWEN35_GDN, 4, 2) == 32 * 128 * 128 * 4 + 12288 * 3 * 2
