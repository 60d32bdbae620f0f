"""The end-to-end leg's call plan (bench.plan_e2e_pieces), checked on the CPU
with the oracle: a request run as its planned consecutive calls, each warm
from the state the call before left in the slot (the pages' chunked prefill
across calls), gives the same outputs, slot and track slots as one call. With
fp64 storage nothing is rounded between calls, so the two agree exactly; this
pins the plan's prefixes, warm flags and rotated track lists."""

import copy

import numpy as np
import pytest
import torch

import bench
import workloads as W
from oracle import lin_state_oracle as O

FLAGS = O.FLAG_QK_L2NORM | O.FLAG_CONV_SILU


def _np(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("cuts", [bench.PrefillWorkload.E2E_CUTS, (0.5,), (0.25, 0.5, 0.75),
                                  (0.1, 0.3, 0.6, 0.9)])
def test_planned_calls_equal_one_call(cuts):
    H, K = 2, 16
    dims = W.LayerDims(num_heads=H, head_k=K, head_v=K)
    lengths, prefixes, warm = [300, 130, 512], [0, 64, 128], [0, 1, 1]
    b = W.make_prefill_batch(dims, lengths, W.GATE_PER_KEY, dtype=torch.float32, seed=3,
                             prefixes=prefixes, warm=warm, tag="e2eplan")
    C = dims.conv_channels
    pool0 = O.make_pool(1, 16, H, K, K, C, state_dtype="f64", conv_dtype="f64")
    rng = np.random.default_rng(3)
    pool0["temporal"][:] = rng.standard_normal(pool0["temporal"].shape) * 0.1
    pool0["conv"][:] = rng.standard_normal(pool0["conv"].shape)
    slots = [1, 2, 3]
    # per request: a ping-pong pair, one slot, five slots cycled
    tracks, cu_track = [4, 5, 6, 7, 8, 9, 10, 11], [0, 2, 3, 8]
    stride = 64
    x, w, g, beta = _np(b.x), _np(b.conv_w), _np(b.g), _np(b.beta)
    cu = b.cu_seqlens.tolist()

    one = copy.deepcopy(pool0)
    o_one, st = O.prefill(one, 0, x, w, g, beta, cu, prefixes, slots, warm, tracks, cu_track,
                          stride, O.GATE_PER_KEY, FLAGS, 1.0, "f64")
    assert st == 0

    plan = bench.plan_e2e_pieces(cu, prefixes, warm, tracks, cu_track, stride, cuts)
    # every token is covered once, each call is 64-aligned and starts where
    # the request's previous call ended
    covered = sorted((p["t0"], p["t1"]) for p in plan)
    assert covered[0][0] == 0 and covered[-1][1] == cu[-1]
    assert all(a[1] == c[0] for a, c in zip(covered, covered[1:]))
    assert all(p["prefix"] % 64 == 0 for p in plan)
    assert [p["index"] for p in plan] == sorted(p["index"] for p in plan)

    pieces = copy.deepcopy(pool0)
    o_pieces = np.full_like(o_one, np.nan)
    for p in plan:
        r, t0, t1 = p["request"], p["t0"], p["t1"]
        rot = p["tracks"]
        o, st = O.prefill(pieces, 0, x[t0:t1], w, g[t0:t1], beta[t0:t1], [0, t1 - t0],
                          [p["prefix"]], [slots[r]], [p["warm"]], rot, [0, len(rot)], stride,
                          O.GATE_PER_KEY, FLAGS, 1.0, "f64")
        assert st == 0
        o_pieces[t0:t1] = o
    assert np.array_equal(o_pieces, o_one)
    assert np.array_equal(pieces["temporal"], one["temporal"])
    assert np.array_equal(pieces["conv"], one["conv"])


def test_plan_rotates_track_lists_by_the_boundaries_before_each_call():
    """A request with prefix 64, 512 tokens, stride 64 and a 3-slot list: its
    boundaries 128, 192, ..., 576 are the request's boundaries 0..7, so the
    call starting at token 256 (absolute 320) has 4 boundaries before it and
    its list starts at slot list[4 mod 3]."""
    plan = bench.plan_e2e_pieces([0, 512], [64], [1], [20, 21, 22], [0, 3], 64, (0.5,))
    assert [(p["t0"], p["t1"], p["prefix"], p["warm"], p["tracks"]) for p in plan] == [
        (0, 256, 64, 1, [20, 21, 22]),
        (256, 512, 320, 1, [21, 22, 20]),
    ]
