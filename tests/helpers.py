"""Shared helpers for the parity tests: run the library (through the C ABI
binding) and the CPU oracle on the same seeded inputs and compare."""

from __future__ import annotations

import numpy as np
import torch

DT_NAME = {torch.float32: "f32", torch.bfloat16: "bf16"}

# Parity bars: rel-L2 per (request, head) tensor.
TOL_F32 = 1e-3   # fp32 state and fp32 outputs
TOL_BF16 = 2e-2  # bf16 inputs and bf16 state


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def oracle_pool(pool) -> dict:
    return {"temporal": np64(pool.temporal), "conv": np64(pool.conv),
            "state_dtype": DT_NAME[pool.temporal.dtype], "conv_dtype": DT_NAME[pool.conv.dtype]}


def max_rel_per_head(gpu: np.ndarray, ref: np.ndarray, head_axis: int) -> float:
    """Max over heads of rel-L2 (head_axis indexes heads)."""
    worst = 0.0
    for h in range(gpu.shape[head_axis]):
        worst = max(worst, rel_l2(np.take(gpu, h, head_axis), np.take(ref, h, head_axis)))
    return worst


def compare_outputs(out_gpu, out_ref, cu_seqlens, tol, skip=()):
    """Per (request, head) rel-L2 of outputs [T][H][V]."""
    o = np64(out_gpu)
    worst = 0.0
    for r in range(len(cu_seqlens) - 1):
        if r in skip:
            continue
        a, b = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        if b > a:
            worst = max(worst, max_rel_per_head(o[a:b], out_ref[a:b], 1))
    assert worst <= tol, f"outputs rel-L2 {worst:.3e} > {tol}"
    return worst


def compare_slots(pool, opool, slots, tol, layer=0):
    """States per (slot, head) within tol; conv windows bit-exact."""
    t = np64(pool.temporal[layer])
    c = np64(pool.conv[layer])
    worst = 0.0
    for s in slots:
        worst = max(worst, max_rel_per_head(t[s], opool["temporal"][layer, s], 0))
        assert np.array_equal(c[s], opool["conv"][layer, s]), f"conv window of slot {s} differs"
    assert worst <= tol, f"state rel-L2 {worst:.3e} > {tol}"
    return worst


def fill_pool(pool, seed, std=0.05):
    import workloads as W
    t = W.randn(pool.temporal.shape, seed, "pool.t", std=std)
    c = W.randn(pool.conv.shape, seed, "pool.c")
    pool.temporal.copy_(t.to(pool.temporal.dtype))
    pool.conv.copy_(c.to(pool.conv.dtype))
