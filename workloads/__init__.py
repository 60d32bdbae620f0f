"""Seeded synthetic inputs for the gated delta-rule state path.

This module only draws random numbers and lays them out in the shapes the
library and the oracle consume. It holds none of the method's arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.

Shapes follow the pages' workloads:

* Kimi-K3 notes ("企业官网建设流程全解析", section on the Linear state size):
  one TP8 shard has 12 KDA heads, K = V = 128, conv state [3, 4608], 69 layers.
* Qwen3.5 Linear-State Prefix Cache (section 1): GDN layers with 32 heads.
* Ping-Pong page (parameters): chunk 64, track interval 256, two track slots.

Every tensor is drawn from its own torch.Generator seeded from (seed, name),
so a tensor does not change when another one is added or resized.
"""

from __future__ import annotations

import dataclasses
import hashlib
from typing import List, Optional

import torch

# Gate modes (scalar decay per head = GDN, per key channel = KDA).
GATE_PER_HEAD = 0
GATE_PER_KEY = 1


def _gen(seed: int, name: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def randn(shape, seed, name, device="cpu", dtype=torch.float32, std=1.0):
    g = _gen(seed, name, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def rand(shape, seed, name, device="cpu", lo=0.0, hi=1.0):
    g = _gen(seed, name, device)
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def randint(lo, hi, shape, seed, name):
    """Integers uniform in [lo, hi] (inclusive), drawn on the CPU."""
    g = _gen(seed, name, "cpu")
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int64)


def randperm(n, seed, name):
    g = _gen(seed, name, "cpu")
    return torch.randperm(n, generator=g)


@dataclasses.dataclass
class LayerDims:
    num_heads: int
    head_k: int
    head_v: int
    conv_width: int = 4

    @property
    def conv_channels(self) -> int:
        # q | k | v projection channels feed the short conv (Kimi-K3 notes:
        # conv state [3, Q_local + K_local + V_local]).
        return 2 * self.num_heads * self.head_k + self.num_heads * self.head_v


# Named workload shapes.
TINY_GDN = LayerDims(num_heads=2, head_k=16, head_v=16)
QWEN35_GDN = LayerDims(num_heads=32, head_k=128, head_v=128)
KIMI_K3_TP8 = LayerDims(num_heads=12, head_k=128, head_v=128)
# a Mamba2-style SSD layer with head dim 64 and state size 128 (d_inner 4096):
# in this pool's layout 64 heads of 128 key (B, C) and 64 value (x) channels
MAMBA2_HD64 = LayerDims(num_heads=64, head_k=128, head_v=64)


def gate_log_decay_softplus(shape, seed, name, device="cpu"):
    """log(alpha) for alpha = exp(-softplus(z)), z ~ N(0, 1): g = -softplus(z)."""
    z = randn(shape, seed, name, device)
    return -torch.nn.functional.softplus(z)


def gate_log_decay_uniform(shape, seed, name, device="cpu", lo=-0.1, hi=0.0):
    """Scalar per-head log-decay uniform in [lo, hi]."""
    return rand(shape, seed, name, device, lo, hi)


def beta_sigmoid(shape, seed, name, device="cpu"):
    return torch.sigmoid(randn(shape, seed, name, device))


def ssd_gates(shape, seed, name, device="cpu"):
    """Inputs of the additive (Mamba2 SSD) form: a step size dt = softplus(z - 3),
    z ~ N(0, 1) (median about 0.05) per (token, head), and a per-head rate
    A = -U[1, 16] over the last axis of `shape`. Returns (g, beta) =
    (dt * A, dt): the log-decay and the input scale."""
    dt = torch.nn.functional.softplus(randn(shape, seed, f"{name}.dt", device) - 3.0)
    A = -rand((shape[-1],), seed, f"{name}.A", device, 1.0, 16.0)
    return dt * A, dt


def l2_normalise_heads(x: torch.Tensor, dims: LayerDims) -> torch.Tensor:
    """Normalise the q and k channel groups of x [..., C] per head (input recipe
    of the tiny workload: q, k drawn N(0,1) then L2-normalised per head)."""
    H, K = dims.num_heads, dims.head_k
    out = x.clone()
    for part in range(2):
        sl = out[..., part * H * K:(part + 1) * H * K]
        shp = sl.shape[:-1] + (H, K)
        v = sl.reshape(shp)
        v = v / v.norm(dim=-1, keepdim=True)
        out[..., part * H * K:(part + 1) * H * K] = v.reshape(sl.shape)
    return out


@dataclasses.dataclass
class PrefillBatch:
    dims: LayerDims
    gate_mode: int
    x: torch.Tensor            # [T][C] pre-conv q|k|v inputs
    conv_w: torch.Tensor       # [C][4]
    g: torch.Tensor            # [T][H] or [T][H][K], fp32 log-decay
    beta: torch.Tensor         # [T][H] fp32
    cu_seqlens: torch.Tensor   # [B+1] int32
    prefix_len: torch.Tensor   # [B] int32
    has_initial_state: torch.Tensor  # [B] int64

    @property
    def batch(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])


def make_prefill_batch(dims: LayerDims, lengths: List[int], gate_mode: int,
                       dtype=torch.bfloat16, seed: int = 0, device="cpu",
                       gate: str = "softplus", prefixes: Optional[List[int]] = None,
                       warm: Optional[List[int]] = None, tag: str = "prefill",
                       qk_prenorm: bool = False, conv_std: float = 0.5
                       ) -> PrefillBatch:
    """Varlen prefill inputs. x ~ N(0,1); conv weights ~ N(0, conv_std^2);
    g per the gate recipe; beta = sigmoid(N(0,1)), except gate "ssd": g and
    beta from ssd_gates (per-head gates only)."""
    B = len(lengths)
    T = int(sum(lengths))
    H, K = dims.num_heads, dims.head_k
    C = dims.conv_channels
    x = randn((T, C), seed, f"{tag}.x", device)
    if qk_prenorm:
        x = l2_normalise_heads(x, dims)
    x = x.to(dtype)
    conv_w = randn((C, dims.conv_width), seed, f"{tag}.conv_w", device,
                   std=conv_std).to(dtype)
    gshape = (T, H) if gate_mode == GATE_PER_HEAD else (T, H, K)
    if gate == "ssd":
        assert gate_mode == GATE_PER_HEAD
        g, beta = ssd_gates((T, H), seed, f"{tag}.ssd", device)
    else:
        if gate == "softplus":
            g = gate_log_decay_softplus(gshape, seed, f"{tag}.g", device)
        else:
            g = gate_log_decay_uniform(gshape, seed, f"{tag}.g", device)
        beta = beta_sigmoid((T, H), seed, f"{tag}.beta", device)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    pre = torch.tensor(prefixes if prefixes is not None else [0] * B, dtype=torch.int32)
    hs = torch.tensor(warm if warm is not None else [0] * B, dtype=torch.int64)
    return PrefillBatch(dims, gate_mode, x, conv_w, g, beta, cu.to(device),
                        pre.to(device), hs.to(device))


def make_decode_inputs(dims: LayerDims, batch: int, n_draft: int, gate_mode: int,
                       dtype=torch.bfloat16, seed: int = 0, device="cpu",
                       tag: str = "decode", step: int = 0, gate: str = "softplus"):
    """One decode step's inputs for `batch` requests x `n_draft` tokens
    (gate "ssd": g and beta from ssd_gates, per-head gates only)."""
    H, K = dims.num_heads, dims.head_k
    C = dims.conv_channels
    t = f"{tag}.{step}"
    x = randn((batch, n_draft, C), seed, f"{t}.x", device).to(dtype)
    if gate == "ssd":
        assert gate_mode == GATE_PER_HEAD
        g, beta = ssd_gates((batch, n_draft, H), seed, f"{t}.ssd", device)
        return x, g, beta
    gshape = (batch, n_draft, H) if gate_mode == GATE_PER_HEAD else (batch, n_draft, H, K)
    g = gate_log_decay_softplus(gshape, seed, f"{t}.g", device)
    beta = beta_sigmoid((batch, n_draft, H), seed, f"{t}.beta", device)
    return x, g, beta


def state_bytes(dims: LayerDims, state_esize: int, conv_esize: int) -> int:
    """Bytes of one layer-slot (temporal + conv state)."""
    return (dims.num_heads * dims.head_v * dims.head_k * state_esize
            + dims.conv_channels * (dims.conv_width - 1) * conv_esize)


def kp_lengths(seed: int = 0, n: int = 32, lo: int = 1024, hi: int = 16384):
    """Kimi-K3 varlen prefill recipe: L_r ~ U{lo..hi}; requests 0..n/2-1 warm
    with prefix P_r = 64 * U{1..floor((L_r-1)/64)}, the rest cold."""
    L = randint(lo, hi, (n,), seed, "kp.len").tolist()
    pre = []
    for r, Lr in enumerate(L):
        if r < n // 2:
            m = max(1, (Lr - 1) // 64)
            u = int(randint(1, m, (1,), seed, f"kp.pre.{r}")[0])
            pre.append(64 * u)
        else:
            pre.append(0)
    return L, pre
