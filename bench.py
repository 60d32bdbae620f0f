"""Benchmark of the GB300 state path on seeded synthetic workloads.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--only qwen35_gdn_prefill,...]

Prints ONE JSON line. The headline (`value`) is the Qwen3.5-style GDN prefill:
one linear layer, 32 heads, K = V = 128, conv over 3 x 4096 channels, bf16
inputs, fp32 state and outputs, 8 requests x 4096 tokens, cold start,
snapshots every 64 tokens into ping-pong track slots -- in tokens per second.
Each timed step is one lin_state_prefill call over the whole batch, with inputs
already resident in HBM (they are larger than L2). The other workloads of the
path (Kimi-K3 KDA varlen prefill, KDA decode, speculative verify + commit, slot
copies, a 131,072-token single-request prefill) are measured the same way and
reported under "workloads".

Multi-GPU (torchrun): every rank runs the same workload on its own GPU with
no collective on the data path (requests and their slots are independent),
so the aggregate is the sum over ranks ("scaling": "weak"); time is the max
over ranks.

--impl reference times the oracle's plain C restatement (float32, every
host thread) on a bounded sample of the same workload; each workload line
also carries that CPU baseline on a sample of its own inputs.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "GDN/KDA prefill tok/s, decode req-steps/s, slot-copy GB/s vs HBM roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class Workload:
    name = ""
    unit = ""
    kernel = ""          # the dominant kernel's name (for the roofline block)
    launches_per_step = 1
    kern_events = None   # when a dict, step() appends (start, end) events around each timed launch, by tag
    # the step's other timed launches: tag -> (kernel name, algorithmic bytes per launch)
    other_launches = {}

    def units_per_step(self) -> float: ...
    def algo_bytes_per_step(self) -> float: ...
    def kernel_bytes_per_launch(self) -> float:
        return self.algo_bytes_per_step()
    def step(self, i: int) -> None: ...

    def _k_begin(self, tag="main"):
        if self.kern_events is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            self.kern_events.setdefault(tag, []).append([e, None])

    def _k_end(self, tag="main"):
        if self.kern_events is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            self.kern_events[tag][-1][1] = e


def prefill_algo_bytes(dims, lengths, prefixes, warm, gate_mode, es_io, es_out, es_state,
                       track_stride):
    """Algorithmic bytes of one prefill launch and its snapshot count: per
    token x, g, beta in and the output out; one state block (state and conv
    window) per snapshot, per final write-back and per warm start; the conv
    taps once. The conv window is stored in the input dtype."""
    H, K, V, C = dims.num_heads, dims.head_k, dims.head_v, dims.conv_channels
    per_tok = C * es_io + (H * K if gate_mode == W.GATE_PER_KEY else H) * 4 + H * 4 + H * V * es_out
    state_b = H * V * K * es_state + C * 3 * es_io
    n_snap = sum(((p + l) // track_stride - p // track_stride) for p, l in zip(prefixes, lengths))
    n_init = sum(1 for w in warm if w)
    T = sum(lengths)
    return T * per_tok + (n_snap + len(lengths) + n_init) * state_b + C * 4 * es_io, n_snap


class PrefillWorkload(Workload):
    def __init__(self, L, dev, name, dims, lengths, prefixes, warm, gate_mode, io_dtype,
                 out_dtype, state_dtype, track_stride, tracks_per_req, gate, seed=0, flags=None):
        self.L, self.dev, self.name = L, dev, name
        self.unit = "tok/s"
        self.kernel = "prefill"
        b = W.make_prefill_batch(dims, lengths, gate_mode, dtype=io_dtype, seed=seed,
                                 device=dev, gate=gate, prefixes=prefixes, warm=warm,
                                 tag=name)
        self.b = b
        B = len(lengths)
        self.B = B
        if tracks_per_req == "all":
            n_tr = [((p + l) // track_stride - p // track_stride) for p, l in zip(prefixes, lengths)]
        else:
            n_tr = [tracks_per_req] * B
        n_slots = 1 + B + sum(n_tr)
        self.pool = L.StatePool(1, n_slots, dims.num_heads, dims.head_k, state_dtype=state_dtype,
                                conv_dtype=io_dtype, device=dev, head_v=dims.head_v)
        if any(warm):
            g = torch.Generator(device=dev)
            g.manual_seed(seed + 17)
            self.pool.temporal.normal_(0.0, 0.05, generator=g)
            self.pool.conv.normal_(0.0, 1.0, generator=g)
        self.slot = torch.arange(1, 1 + B, dtype=torch.int32, device=dev)
        self.track = torch.arange(1 + B, n_slots, dtype=torch.int32, device=dev)
        cu = [0]
        for n in n_tr:
            cu.append(cu[-1] + n)
        self.cu_track = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.out = torch.empty((b.total_tokens, dims.num_heads, dims.head_v), dtype=out_dtype,
                               device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.track_stride = track_stride
        self.kw = dict(layer=0, x=b.x, conv_w=b.conv_w, g=b.g, beta=b.beta, out=self.out,
                       cu_seqlens=b.cu_seqlens, prefix_len=b.prefix_len, slot=self.slot,
                       has_initial_state=b.has_initial_state, track_slots=self.track,
                       cu_track=self.cu_track, track_stride=track_stride, gate_mode=gate_mode,
                       flags=L.LIN_QK_L2NORM | L.LIN_CONV_SILU if flags is None else flags,
                       status=self.status)
        need = L.lin_state_prefill_workspace(self.pool, **self.kw)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.kernel_kind = L.lin_state_prefill_kernel(self.pool, **self.kw)
        self.kernel = "prefill_chunked" if self.kernel_kind == L.LIN_KERNEL_CHUNKED else "prefill_recurrent"
        # launches per call: the chunked kernel, plus the longest-first order of
        # a varlen batch; a batch with more (request, head) chains than SMs takes
        # the wrap-around plan instead of the order (its buffers are the
        # workspace beyond what the one-piece schedule asks for); a request in
        # segments takes the offset / transition launch, the scan (more than
        # two segments) and the final launch; per-key gates add the
        # token-by-token rerun launch behind the chunked one (its CTAs return at
        # once unless their pair left the chunk's factored decay range) and the
        # rerun flags in the workspace
        if self.kernel_kind == L.LIN_KERNEL_CHUNKED:
            kda = gate_mode == W.GATE_PER_KEY
            kw1 = dict(self.kw, flags=self.kw["flags"] | L.LIN_PREFILL_ONE_PIECE)
            need1 = L.lin_state_prefill_workspace(self.pool, **kw1)
            self.wrap = need > need1
            ow = (B * 4 + 255) // 256 * 256 if 1 < B <= 4096 else 0
            rw = ((B * dims.num_heads + 31) // 32 * 4 + 255) // 256 * 256 if kda else 0
            seg_bytes = need1 - ow - rw
            if self.wrap:
                self.launches_per_step = 2
            elif seg_bytes > 0:
                nseg = seg_bytes // (2 * dims.num_heads * dims.head_k * dims.head_k * 4)
                self.launches_per_step = (1 if ow else 0) + 2 + (1 if nseg > 2 else 0)
            else:
                self.launches_per_step = 1 + (1 if ow else 0)
            self.launches_per_step += 1 if kda else 0
        self.tokens = b.total_tokens
        self.bytes, self.n_snap = prefill_algo_bytes(
            dims, lengths, prefixes, warm, gate_mode, b.x.element_size(), self.out.element_size(),
            self.pool.temporal.element_size(), track_stride)

    def units_per_step(self):
        return self.tokens

    def algo_bytes_per_step(self):
        return self.bytes

    def step(self, i):
        self._k_begin()
        self.L.lin_state_prefill(self.pool, workspace=self.ws, **self.kw)
        self._k_end()

    # e2e: the public call with host inputs (pinned) and the outputs read back.
    # The batch is pipelined over streams: one copies inputs in, one per request
    # runs that request's calls as soon as their inputs have landed, one copies
    # outputs out, so the host link (about 0.2 TB/s each way, 0.34 TB/s both
    # ways together with large copies) stays busy while the GPU computes. Each
    # request runs as calls over consecutive 64-aligned token ranges cut at
    # E2E_CUTS of its length, each warm from the state the one before left in
    # the slot (the pages' chunked prefill), with its track list rotated so
    # every boundary lands where the one-call run puts it. The small first
    # pieces start the computation and the output copies early, the small last
    # pieces keep the tail after the last input copy short; pieces go in order
    # of their index, then request. The gates and betas of the whole step
    # (8 MB) go in one copy ahead of the first piece: two small copies per piece
    # cost the link more than their bytes. Requests are independent and a state
    # round-trips the pool exactly (fp32 state, bf16 windows that are copies of
    # bf16 inputs), so the outputs and slots equal the one-call run's bit for bit.
    E2E_CUTS = (0.125, 0.5, 0.875)

    def setup_e2e(self):
        b, L, dev = self.b, self.L, self.dev
        cu = b.cu_seqlens.cpu().tolist()
        cut = self.cu_track.cpu().tolist()
        pre = b.prefix_len.cpu().tolist()
        warm = b.has_initial_state.cpu().tolist()
        tracks = self.track.cpu().tolist()
        stride = self.track_stride
        self.h_in = [t.cpu().pin_memory() for t in (b.x, b.g, b.beta)]
        self.d_in = [b.x, b.g, b.beta]
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        i32 = lambda v: torch.tensor(v, dtype=torch.int32, device=dev)
        streams = [torch.cuda.Stream() for _ in range(self.B)]
        self.parts = []
        for pc in plan_e2e_pieces(cu, pre, warm, tracks, cut, stride, self.E2E_CUTS):
            r, t0, t1, rot = pc["request"], pc["t0"], pc["t1"], pc["tracks"]
            kw = dict(self.kw)
            kw.update(x=b.x[t0:t1], g=b.g[t0:t1], beta=b.beta[t0:t1], out=self.out[t0:t1],
                      cu_seqlens=i32([0, t1 - t0]), prefix_len=i32([pc["prefix"]]),
                      slot=self.slot[r:r + 1].contiguous(),
                      has_initial_state=torch.tensor([pc["warm"]], dtype=torch.int64, device=dev),
                      track_slots=i32(rot) if rot else None,
                      cu_track=i32([0, len(rot)]) if rot else None)
            self.parts.append(dict(kw=kw, h_in=self.h_in[0][t0:t1], d_in=self.d_in[0][t0:t1],
                                   h_out=self.h_out[t0:t1], d_out=self.out[t0:t1],
                                   stream=streams[r], ev_c=None, ev_d=None))
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        return (sum(t.numel() * t.element_size() for t in self.h_in),
                self.out.numel() * self.out.element_size())

    def step_e2e(self, i):
        cur = torch.cuda.current_stream()
        start = cur.record_event()
        self.s_in.wait_event(start)
        with torch.cuda.stream(self.s_in):  # the step's gates and betas
            for h, d in zip(self.h_in[1:], self.d_in[1:]):
                d.copy_(h, non_blocking=True)
        for pt in self.parts:
            # a piece's input buffers are free once its previous call has run
            if pt["ev_c"] is not None:
                self.s_in.wait_event(pt["ev_c"])
            with torch.cuda.stream(self.s_in):
                pt["d_in"].copy_(pt["h_in"], non_blocking=True)
                ev_in = self.s_in.record_event()
            s = pt["stream"]
            s.wait_event(ev_in)
            if pt["ev_d"] is not None:  # its outputs of the previous step are read back
                s.wait_event(pt["ev_d"])
            with torch.cuda.stream(s):
                # one request per call: noalloc runs it in one piece (a lone
                # request would otherwise go in segments, made for a request
                # that leaves SMs idle; here the requests fill the GPU together)
                self.L.lin_state_prefill_noalloc(self.pool, **pt["kw"])
                pt["ev_c"] = s.record_event()
            self.s_out.wait_event(pt["ev_c"])
            with torch.cuda.stream(self.s_out):
                pt["h_out"].copy_(pt["d_out"], non_blocking=True)
                pt["ev_d"] = self.s_out.record_event()
        for pt in self.parts:
            cur.wait_stream(pt["stream"])
        cur.wait_stream(self.s_in)
        cur.wait_stream(self.s_out)

    def describe(self):
        return {"batch": self.B, "tokens": self.tokens, "snapshots": self.n_snap,
                "kernel": self.kernel}


def plan_e2e_pieces(cu_seqlens, prefix_len, has_initial_state, track_slots, cu_track,
                    track_stride, cut_fractions):
    """The calls of the end-to-end leg. Request r's tokens [cu[r], cu[r+1]) are
    cut at the 64-aligned fractions `cut_fractions` of its length into
    consecutive calls; a call starts from the request's own initial state if
    it is the first, else warm from the state the call before left in the
    slot (its prefix then covers the tokens before it). Each call's track list
    is request r's list rotated by the boundaries that lie before the call, so
    boundary j of the request lands in list[j mod n] as in the one-call run.
    Returns dicts (index, request, t0, t1, prefix, warm, tracks), ordered by
    index within the request, then request."""
    pieces = []
    for r in range(len(cu_seqlens) - 1):
        n = cu_seqlens[r + 1] - cu_seqlens[r]
        cuts = sorted({0, n} | {int(n * f) // 64 * 64 for f in cut_fractions})
        tr = list(track_slots[cu_track[r]:cu_track[r + 1]]) if cu_track is not None else []
        p0 = prefix_len[r]
        for k, (o0, o1) in enumerate(zip(cuts[:-1], cuts[1:])):
            if o1 <= o0:
                continue
            # boundaries before this call, counted within the whole request
            j0 = ((p0 + o0) // track_stride - p0 // track_stride) if track_stride else 0
            rot = [tr[(j0 + q) % len(tr)] for q in range(len(tr))] if tr else []
            pieces.append({"index": k, "request": r, "t0": cu_seqlens[r] + o0,
                           "t1": cu_seqlens[r] + o1, "prefix": p0 + o0,
                           "warm": has_initial_state[r] if o0 == 0 else 1, "tracks": rot})
    pieces.sort(key=lambda e: (e["index"], e["request"]))
    return pieces


def decode_algo_bytes(dims, batch, n_draft, replay=False, track_interval=256):
    """Algorithmic bytes of a decode step and of its dominant launch, bf16
    state, conv window and inputs, per-key gates: (step bytes, launch bytes).
    One token: state and window read and written, the token's x, g, beta and
    output, and the track copy amortised over the interval. Verify of D drafts
    (chain or tree): the slot's state and window read once, every draft's
    state and window written, the drafts' inputs and outputs; the commit reads
    and writes one state. A tree node's read-back of its parent's state is not
    counted. Replay form: the verify reads the state and writes outputs only;
    the commit reads and writes the state and reads the inputs of the accepted
    tokens, (D + 1) / 2 on average."""
    H, K, V = dims.num_heads, dims.head_k, dims.head_v
    st = W.state_bytes(dims, 2, 2)
    o_b = H * V * 2
    x_b = dims.conv_channels * 2 + H * K * 4 + H * 4 + o_b
    B, D = batch, n_draft
    if D == 1:
        b = B * (2 * st + x_b + st / float(track_interval))
        return b, b
    if replay:
        verify = B * (st + D * x_b)
        return verify + B * (2 * st + (D + 1) / 2.0 * (x_b - o_b)), verify
    verify = B * (st + D * st + D * x_b)
    return verify + B * (2 * st), verify


class DecodeWorkload(Workload):
    """KDA decode: pool of 2000 slots x 1 layer (12 x 128 x 128 bf16 temporal,
    [4608][3] bf16 conv), 256 requests on distinct random slots, one token per
    step, interval 256 with per-request track slots; the pool is rotated over 4
    replicas so the per-step working set does not stay in L2."""

    # the draft tree of the tree-verify workload: the MambaRadixCache page's
    # shape (9.6), two roots and depth 4, for every request
    TREE = [-1, -1, 0, 0, 1, 2, 2, 5]

    def __init__(self, L, dev, n_draft=1, replicas=4, seed=0, replay=False, tree=False):
        self.L, self.dev = L, dev
        self.n_draft = n_draft
        self.replay = replay
        self.tree = tree
        self.name = ("kda_decode" if n_draft == 1 else
                     f"kda_tree_verify{n_draft}_commit" if tree else
                     f"kda_spec_verify{n_draft}_replay" if replay else f"kda_spec_verify{n_draft}_commit")
        self.unit = "req-steps/s" if n_draft == 1 else "verify-rounds/s"
        self.kernel = "decode"
        dims = W.KIMI_K3_TP8
        self.dims = dims
        B, S = 256, 2000
        self.B = B
        self.pools = []
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 3)
        for _ in range(replicas):
            p = L.StatePool(1, S, 12, 128, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                            device=dev)
            p.temporal.normal_(0.0, 0.05, generator=g)
            p.conv.normal_(0.0, 1.0, generator=g)
            self.pools.append(p)
        perm = W.randperm(S, seed, "kd.slots")
        self.slot = perm[:B].to(torch.int32).to(dev)
        self.track = perm[B:2 * B].to(torch.int32).to(dev)
        self.pos0 = W.randint(1024, 16384, (B,), seed, "kd.pos").to(torch.int32).to(dev)
        # positions advance by one per pass over the replicas; prepared up front
        self.pos_by_pass = [self.pos0 + k for k in range(64)]
        self.conv_w = W.randn((dims.conv_channels, 4), seed, "kd.w", dev, std=0.5).to(torch.bfloat16)
        n_in = 8
        self.inputs = [W.make_decode_inputs(dims, B, n_draft, W.GATE_PER_KEY, torch.bfloat16,
                                            seed, dev, tag=self.name, step=i) for i in range(n_in)]
        self.out = torch.empty((B, n_draft, 12, 128), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if n_draft > 1:
            if not replay:
                self.specs = [L.SpecBuffer(p, B, n_draft) for p in self.pools]
            self.acc = (W.randint(1, n_draft, (B,), seed, "kd.acc")).to(torch.int32).to(dev)
            self.launches_per_step = 2
        if tree:
            assert n_draft == len(self.TREE) and not replay
            self.parent = torch.tensor([self.TREE] * B, dtype=torch.int32, device=dev)
            node = W.randint(0, n_draft - 1, (B,), seed, "kd.node")
            self.accept_node = node.to(torch.int32).to(dev)
            depth = [0] * n_draft  # tokens on the path from a root to each node
            for j, pj in enumerate(self.TREE):
                depth[j] = 1 + (depth[pj] if pj >= 0 else 0)
            acc_tokens_tree = float(sum(depth[int(k)] for k in node))
        self.bytes, self.verify_bytes = decode_algo_bytes(dims, B, n_draft, replay)
        if n_draft > 1:
            # the commit launch: the replay of the accepted tokens into the slot,
            # or the copy of the accepted step's state and window out of the buffer
            self.other_launches = {"commit": ("decode_kernel (replay commit)" if replay else
                                              "slot_copy_kernel (commit)", self.bytes - self.verify_bytes)}
        if n_draft == 1:
            self.units = B
        else:
            self.units = 1
            self.acc_tokens = acc_tokens_tree if tree else B * (n_draft + 1) / 2.0
        self.steps_done = 0

    def units_per_step(self):
        return self.units

    def algo_bytes_per_step(self):
        return self.bytes

    def kernel_bytes_per_launch(self):
        # the dominant kernel is the decode / verify launch
        return self.verify_bytes

    def step(self, i):
        L = self.L
        r = i % len(self.pools)
        p = self.pools[r]
        x, g, beta = self.inputs[i % len(self.inputs)]
        pos = self.pos_by_pass[(i // len(self.pools)) % len(self.pos_by_pass)]
        if self.n_draft == 1:
            self._k_begin()
            L.lin_state_decode(p, layer=0, x=x, conv_w=self.conv_w, g=g, beta=beta, out=self.out,
                               slot=self.slot, pos=pos, track_slot=self.track, track_interval=256,
                               gate_mode=L.LIN_GATE_PER_KEY, status=self.status)
            self._k_end()
        elif self.replay:
            self._k_begin()
            L.lin_state_decode(p, layer=0, x=x, conv_w=self.conv_w, g=g, beta=beta, out=self.out,
                               slot=self.slot, pos=pos, gate_mode=L.LIN_GATE_PER_KEY,
                               status=self.status)
            self._k_end()
            self._k_begin("commit")
            L.lin_state_replay_commit(p, layer=0, x=x, conv_w=self.conv_w, g=g, beta=beta,
                                      slot=self.slot, pos=pos, accept_len=self.acc,
                                      track_slot=self.track, track_interval=256,
                                      gate_mode=L.LIN_GATE_PER_KEY, status=self.status)
            self._k_end("commit")
            return
        elif self.tree:
            self._k_begin()
            L.lin_state_decode(p, layer=0, x=x, conv_w=self.conv_w, g=g, beta=beta, out=self.out,
                               slot=self.slot, pos=pos, spec=self.specs[r], parent=self.parent,
                               gate_mode=L.LIN_GATE_PER_KEY, status=self.status)
            self._k_end()
            self._k_begin("commit")
            L.lin_state_spec_commit(p, spec=self.specs[r], slot=self.slot, pos=pos,
                                    n_draft=self.n_draft, track_slot=self.track, track_interval=256,
                                    parent=self.parent, accept_node=self.accept_node,
                                    status=self.status)
            self._k_end("commit")
        else:
            self._k_begin()
            L.lin_state_decode(p, layer=0, x=x, conv_w=self.conv_w, g=g, beta=beta, out=self.out,
                               slot=self.slot, pos=pos, spec=self.specs[r],
                               gate_mode=L.LIN_GATE_PER_KEY, status=self.status)
            self._k_end()
            self._k_begin("commit")
            L.lin_state_spec_commit(p, spec=self.specs[r], slot=self.slot, pos=pos,
                                    accept_len=self.acc, n_draft=self.n_draft,
                                    track_slot=self.track, track_interval=256, status=self.status)
            self._k_end("commit")

    def describe(self):
        d = {"batch": self.B, "n_draft": self.n_draft, "pool_slots": 2000,
             "replicas": len(self.pools)}
        if self.tree:
            d["parent"] = self.TREE
        return d


class CopyWorkload(Workload):
    """Checkpoint fork/restore copies: Kimi-K3 slots over 69 layers (12 x 128 x 128
    bf16 + [4608][3] bf16 per layer, 29,039,616 B per slot) in a 128-slot pool
    (3.7 GB), batches of 64 src -> dst pairs: a random half of the slots are the
    destinations, the other half the sources, each used once, so every batch
    reads and writes 64 distinct slots and nothing is read from L2."""

    def __init__(self, L, dev, seed=0, n_batches=8, layers=69):
        self.L, self.dev = L, dev
        self.layers = layers
        self.name = f"slot_copy_kimi_k3_{layers}l"
        self.unit = "GB/s"
        self.kernel = "slot_copy"
        self.n_slots = 128
        self.pool = L.StatePool(layers, self.n_slots, 12, 128, state_dtype=torch.bfloat16,
                                conv_dtype=torch.bfloat16, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 5)
        self.pool.temporal.view(torch.int16).random_(generator=g)
        self.pool.conv.view(torch.int16).random_(generator=g)
        self.pairs = []
        for k in range(n_batches):
            perm = W.randperm(self.n_slots, seed, f"cp.batch{k}")
            dst, src = perm[:64], perm[64:128]
            self.pairs.append((src.to(torch.int32).to(dev), dst.to(torch.int32).to(dev)))
        self.slot_bytes = L.lin_state_slot_bytes(self.pool)
        self.bytes = 2.0 * 64 * self.slot_bytes
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def units_per_step(self):
        return self.bytes / 1e9  # GB moved (read + write)

    def algo_bytes_per_step(self):
        return self.bytes

    def step(self, i):
        s, d = self.pairs[i % len(self.pairs)]
        self._k_begin()
        self.L.lin_state_copy_slots(self.pool, s, d, status=self.status)
        self._k_end()

    def describe(self):
        return {"pairs": 64, "layers": self.layers, "pool_slots": self.n_slots, "slot_bytes": self.slot_bytes}


def make_workload(name, L, dev):
    if name == "qwen35_gdn_prefill":
        return PrefillWorkload(L, dev, name, W.QWEN35_GDN, [4096] * 8, [0] * 8, [0] * 8,
                               W.GATE_PER_HEAD, torch.bfloat16, torch.float32, torch.float32,
                               64, 2, "uniform")
    if name == "kimi_k3_kda_varlen_prefill":
        Ls, Ps = W.kp_lengths(0)
        ext = [l - p for l, p in zip(Ls, Ps)]
        return PrefillWorkload(L, dev, name, W.KIMI_K3_TP8, ext, Ps, [1 if p else 0 for p in Ps],
                               W.GATE_PER_KEY, torch.bfloat16, torch.bfloat16, torch.bfloat16,
                               256, 2, "softplus")
    if name == "kda_long_prefill_131k":
        return PrefillWorkload(L, dev, name, W.KIMI_K3_TP8, [131072], [0], [0], W.GATE_PER_KEY,
                               torch.bfloat16, torch.bfloat16, torch.bfloat16, 64, "all",
                               "softplus")
    if name == "mamba2_ssd_prefill":
        return PrefillWorkload(L, dev, name, W.QWEN35_GDN, [4096] * 8, [0] * 8, [0] * 8,
                               W.GATE_PER_HEAD, torch.bfloat16, torch.float32, torch.float32,
                               64, 2, "ssd", flags=L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE)
    if name == "mamba2_ssd_prefill_hd64":
        return PrefillWorkload(L, dev, name, W.MAMBA2_HD64, [4096] * 8, [0] * 8, [0] * 8,
                               W.GATE_PER_HEAD, torch.bfloat16, torch.float32, torch.float32,
                               64, 2, "ssd", flags=L.LIN_CONV_SILU | L.LIN_UPDATE_ADDITIVE)
    if name == "kda_recurrent_prefill":
        return PrefillWorkload(L, dev, name, W.KIMI_K3_TP8, [2048] * 32, [0] * 32, [0] * 32,
                               W.GATE_PER_KEY, torch.bfloat16, torch.bfloat16, torch.bfloat16,
                               256, 2, "softplus",
                               flags=L.LIN_QK_L2NORM | L.LIN_CONV_SILU | L.LIN_PREFILL_RECURRENT)
    if name == "kda_decode":
        return DecodeWorkload(L, dev, 1)
    if name == "kda_spec_verify4_commit":
        return DecodeWorkload(L, dev, 4)
    if name == "kda_spec_verify4_replay":
        return DecodeWorkload(L, dev, 4, replay=True)
    if name == "kda_tree_verify8_commit":
        return DecodeWorkload(L, dev, 8, tree=True)
    if name == "slot_copy_kimi_k3_69l":
        return CopyWorkload(L, dev)
    if name == "slot_copy_kimi_k3_8l":
        # the same copies over 8 layers (a 0.43 GB pool): the case profiled
        # with every ncu section; the 69-layer pool (3.7 GB) is captured for
        # its DRAM counters and duration only
        return CopyWorkload(L, dev, layers=8)
    raise ValueError(name)


HEADLINE = "qwen35_gdn_prefill"
DEFAULT_EXTRA = ["kimi_k3_kda_varlen_prefill", "kda_decode", "kda_spec_verify4_commit",
                 "kda_spec_verify4_replay", "kda_tree_verify8_commit",
                 "slot_copy_kimi_k3_69l", "kda_long_prefill_131k", "mamba2_ssd_prefill",
                 "mamba2_ssd_prefill_hd64", "kda_recurrent_prefill"]

CONFIG_TEXT = {
    "qwen35_gdn_prefill": "Qwen3.5-style GDN prefill: 1 linear layer, 32 heads, K=V=128, conv 4 over "
                          "3x4096 channels, bf16 q/k/v inputs, fp32 state and outputs, scalar "
                          "log-decay U[-0.1,0], 8 requests x 4096 tokens, chunk 64, cold start, "
                          "snapshot every 64 into ping-pong track slots",
    "kimi_k3_kda_varlen_prefill": "Kimi-K3 TP8-shard KDA varlen prefill: 12 heads, K=V=128, per-key "
                                  "decay, bf16 inputs/state/outputs, 32 requests L~U[1k,16k], half "
                                  "warm at a 64-multiple prefix, snapshots every 256 (ping-pong)",
    "kda_decode": "KDA decode: 2000-slot pool, 256 requests, 12x128x128 bf16 state + [4608][3] conv, "
                  "1 token per step, track interval 256, 4 pool replicas",
    "kda_spec_verify4_commit": "KDA speculative verify of 4 drafts + commit of U{1..4} accepted, "
                               "256 requests, per-step states in a spec buffer",
    "kda_tree_verify8_commit": "KDA draft-tree verify of 8 drafts (two roots, depth 4: parents "
                               "-1,-1,0,0,1,2,2,5) into a spec buffer + commit of a random accepted "
                               "node, 256 requests",
    "kda_spec_verify4_replay": "KDA speculative verify of 4 drafts (outputs only) + replay commit of "
                               "U{1..4} accepted tokens into the slot, 256 requests, no per-step buffer",
    "slot_copy_kimi_k3_8l": "checkpoint fork/restore copy: Kimi-K3 slot over 8 layers (3,366,912 B), 64 "
                            "random src->dst pairs per batch over a 128-slot pool, every slot used once "
                            "(the case profiled with every ncu section)",
    "slot_copy_kimi_k3_69l": "checkpoint fork/restore copy: Kimi-K3 slot over 69 layers (29,039,616 B), "
                             "64 random src->dst pairs per batch over a 128-slot pool (3.7 GB), every "
                             "slot used once",
    "mamba2_ssd_prefill": "Mamba2-style SSD prefill (additive update, no delta correction): 32 heads, "
                          "headdim = d_state = 128, conv 4 + SiLU over x|B|C, no q/k norm, "
                          "dt = softplus(N(0,1)-3), A = -U[1,16] per head, bf16 inputs, fp32 state "
                          "and outputs, 8 requests x 4096 tokens, snapshot every 64 (ping-pong)",
    "mamba2_ssd_prefill_hd64": "Mamba2-style SSD prefill with head dim 64 and state size 128 (additive "
                               "update): 64 heads of 128 key (B, C) and 64 value (x) channels, conv 4 + "
                               "SiLU over x|B|C, no q/k norm, dt = softplus(N(0,1)-3), A = -U[1,16] per "
                               "head, bf16 inputs, fp32 state and outputs, 8 requests x 4096 tokens, "
                               "snapshot every 64 (ping-pong)",
    "kda_long_prefill_131k": "single-request KDA prefill, 131072 tokens, 12 heads, bf16, cold, "
                             "snapshots every 64 into 2048 distinct track slots",
    "kda_recurrent_prefill": "KDA prefill on the token-by-token kernel (LIN_PREFILL_RECURRENT, the kernel "
                             "that also reruns pairs whose decay leaves the chunk's range): Kimi-K3 TP8 "
                             "shard, 12 heads, K=V=128, bf16, 32 requests x 2048 tokens, cold, snapshots "
                             "every 256 (ping-pong)",
}


def flush_l2(buf):
    buf.add_(1)


def time_steps(wl, steps, warmup, stream, flush=None):
    """Returns (total_ms over `steps`, per-step ms list, per-launch ms lists of
    the timed launches by tag, "main" the dominant kernel). The timed steps are queued behind a short device-side
    sleep so the host enqueues them ahead of the GPU: no step waits on the
    host, and the events measure device time only."""
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    wl.kern_events = {}
    torch.cuda._sleep(int(min(steps, 200) * 300e3))  # ~0.15 ms of host enqueue time per step at 2 GHz
    t0.record(stream)
    for i in range(steps):
        if flush is not None:
            flush()
        evs[i][0].record(stream)
        wl.step(warmup + i)
        evs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in evs]
    kern = {tag: [a.elapsed_time(b) for a, b in ev] for tag, ev in wl.kern_events.items()}
    wl.kern_events = None
    return t0.elapsed_time(t1), per, kern


def reduce_over_ranks(rank_ms, units_per_rank, world, device):
    """Whole-job figures of a step that every rank ran on its own replica:
    the time is the slowest rank's (all-reduce MAX), the work is the sum over
    ranks. Returns (ms, units per second)."""
    if world > 1:
        t = torch.tensor([rank_ms], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        rank_ms = float(t.item())
    return rank_ms, units_per_rank * world / (rank_ms / 1e3)


def run_workload(name, L, dev, steps, warmup, peaks, stream, dist_info, e2e=False, cpu=False):
    wl = make_workload(name, L, dev)
    # decode rotates 4 pool replicas: a replica's 108 MB working set is never
    # L2-resident when it comes back, so no flush is needed (a written flush
    # buffer would leave dirty lines for the timed kernel to write back)
    need_flush = False
    flush_buf = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev) if need_flush else None
    total_ms, per, kern = time_steps(wl, steps, warmup, stream,
                                     (lambda: flush_l2(flush_buf)) if need_flush else None)
    kern_ms = statistics.mean(kern["main"])
    rank_ms, value = reduce_over_ranks(statistics.mean(per), wl.units_per_step(), dist_info["world"], dev)
    units = wl.units_per_step() * dist_info["world"]
    achieved = wl.kernel_bytes_per_launch() / (kern_ms / 1e3) / 1e9
    res = {"value": value, "unit": wl.unit, "ms_per_step": rank_ms,
           "roofline": {"bound": "hbm", "kernel": wl.kernel, "achieved": achieved,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(name),
                        "algo_bytes_per_launch": wl.kernel_bytes_per_launch(),
                        "kernel_ms": kern_ms},
           "config": {"workload": CONFIG_TEXT[name], **wl.describe()},
           "gpu_launches": wl.launches_per_step * steps}
    if wl.other_launches:
        # the step's other launches, each against the same peak
        res["other_launches"] = {}
        for tag, (kname, kbytes) in wl.other_launches.items():
            ms = statistics.mean(kern[tag])
            ach = kbytes / (ms / 1e3) / 1e9
            res["other_launches"][tag] = {"kernel": kname, "kernel_ms": ms, "algo_bytes_per_launch": kbytes,
                                          "achieved": ach, "frac": ach / peaks["hbm_gbs"]}
    if hasattr(wl, "acc_tokens"):
        res["accepted_tok_s"] = wl.acc_tokens * dist_info["world"] / (rank_ms / 1e3)
    if e2e and hasattr(wl, "setup_e2e"):
        bi, bo = wl.setup_e2e()
        for i in range(2):
            wl.step_e2e(i)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            wl.step_e2e(i)
        t1.record(stream)
        torch.cuda.synchronize()
        e_ms, e_val = reduce_over_ranks(t0.elapsed_time(t1) / steps, wl.units_per_step(),
                                        dist_info["world"], dev)
        res["e2e"] = {"value": e_val, "unit": wl.unit,
                      "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e_ms}
    if cpu and name in CPU_LEGS:
        res["cpu_baseline"] = CPU_LEGS[name](wl)
    del wl
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# DRAM traffic of the dominant kernels, from one ncu capture each
# ---------------------------------------------------------------------------
ROOT = os.path.dirname(os.path.abspath(__file__))


def _code_only(src):
    """C / C++ / CUDA source without its comments and with each line's
    whitespace collapsed (string and character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    lines = (" ".join(line.split()) for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


# The source files each kernel family is built from (besides the shared
# headers, the ABI layer and the C header, which count for all of them).
KERNEL_SOURCES = {
    "chunked": ["chunked_prefill.cu", "umma.cuh"],
    "token": ["token_kernels.cu"],
    "verify_chunk": ["verify_chunk.cu"],
    "copy": ["copy_kernels.cu"],
}
SHARED_SOURCES = ["common.cuh", "internal.h", "api.cu"]


def library_source_hash(family=None):
    """Digest of the CUDA library sources, comments and whitespace left out:
    of one kernel family's files plus the shared ones, or of every source
    (family None). A traffic figure is reported only while the code of the
    kernel it was measured on is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_state_chunked_gb300", "csrc")
    if family is None:
        names = [f for f in sorted(os.listdir(csrc)) if f.endswith((".cu", ".cuh", ".h"))]
    else:
        names = sorted(KERNEL_SOURCES[family] + SHARED_SOURCES)
    files = [os.path.join(csrc, f) for f in names]
    files.append(os.path.join(ROOT, "include", "lin_state.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of the workload's
    dominant kernel, from the capture table profiles/dram_traffic.json, or None
    when there is no row or the row's kernel family has changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rows = json.load(fh).get("rows", [])
    for row in rows:
        if row.get("workload") == workload and row.get("library_source") == library_source_hash(row.get("family")):
            return int(row["traffic_per_launch"])
    return None


# ---------------------------------------------------------------------------
# CPU baseline: the C restatement of the oracle (oracle/lin_state_ref.c) in
# float32 on every host thread, on a bounded sample of each workload's own
# inputs. A baseline beside the GPU figures, not a target.
# ---------------------------------------------------------------------------
def _host_f32(t):
    import numpy as np
    return np.ascontiguousarray(t.detach().to(torch.float32).cpu().numpy())


def _rname(dtype):
    return "bf16" if dtype == torch.bfloat16 else "f32"


def _cpu_result(value, unit, sample, seconds):
    from oracle import lin_state_ref as R
    return {"value": value, "unit": unit, "cores": R.host_threads(), "cpu_model": R.cpu_model(),
            "kind": "oracle", "precision": "f32",
            "sample": f"{sample}; C restatement of the oracle, float32, {R.host_threads()} threads, "
                      f"{seconds:.2f} s"}


def cpu_prefill(wl, max_tokens):
    """Requests of the prefill workload in batch order (the first request cut
    at max_tokens if it alone is longer) until max_tokens extend tokens, all
    heads, with the workload's snapshots, dtypes and flags."""
    import numpy as np
    from oracle import lin_state_ref as R
    b = wl.b
    cu = b.cu_seqlens.tolist()
    n = 0
    while n < wl.B and cu[n + 1] - cu[0] <= max_tokens:
        n += 1
    if n == 0:  # one request longer than the sample: its first max_tokens tokens
        n, cu_s = 1, [0, max_tokens]
    else:
        cu_s = cu[:n + 1]
    T = cu_s[-1]
    x, g, beta = (_host_f32(t[:T]) for t in (b.x, b.g, b.beta))
    cw = _host_f32(b.conv_w)
    ctr = wl.cu_track.tolist()[:n + 1]
    # the sample's live and track slots, gathered into a compact host pool
    slots, tracks = wl.slot.tolist()[:n], wl.track.tolist()[:ctr[-1]]
    used = sorted(set(slots) | set(t for t in tracks if t >= 0))
    remap = {s_: i for i, s_ in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=wl.pool.temporal.device)
    temporal = _host_f32(wl.pool.temporal[0].index_select(0, idx))
    conv = _host_f32(wl.pool.conv[0].index_select(0, idx))
    out = np.zeros((T,) + tuple(wl.out.shape[1:]), np.float32)
    args = (temporal, conv, x, cw, g, beta, cu_s, b.prefix_len.tolist()[:n], [remap[s_] for s_ in slots],
            b.has_initial_state.tolist()[:n], [remap[t] if t >= 0 else -1 for t in tracks], ctr,
            wl.track_stride, b.gate_mode,
            wl.kw["flags"], 1.0, out, _rname(wl.pool.temporal.dtype), _rname(wl.pool.conv.dtype),
            _rname(wl.out.dtype))
    t0 = time.perf_counter()
    st = R.prefill_arrays("f32", *args)
    dt = time.perf_counter() - t0
    assert st == 0, st
    return _cpu_result(T / dt, "tok/s", f"{n} request(s), {T} tokens x {b.dims.num_heads} heads of the "
                       f"workload", dt)


def cpu_decode(wl, rounds):
    """`rounds` steps of the decode / verify workload on all 256 requests, its
    slots gathered into a compact host pool (live slots, then track slots)."""
    import numpy as np
    from oracle import lin_state_ref as R
    B = wl.B
    slots, tracks = wl.slot.tolist(), wl.track.tolist()
    idx = torch.tensor(slots + tracks, dtype=torch.long, device=wl.pools[0].temporal.device)
    temporal = _host_f32(wl.pools[0].temporal[0].index_select(0, idx))
    conv = _host_f32(wl.pools[0].conv[0].index_select(0, idx))
    cs, ct = list(range(B)), list(range(B, 2 * B))
    cw = _host_f32(wl.conv_w)
    ins = [tuple(_host_f32(t) for t in wl.inputs[k % len(wl.inputs)]) for k in range(rounds)]
    D = wl.n_draft
    out = np.zeros((B, D, 12, 128), np.float32)
    spec_t = spec_c = None
    if D > 1 and not wl.replay:
        spec_t = np.zeros((B, D, 12, 128, 128), np.float32)
        spec_c = np.zeros((B, D, wl.dims.conv_channels, 3), np.float32)
    acc = wl.acc.tolist() if D > 1 else None
    pos0 = wl.pos0.tolist()
    flags = 3  # L2 norm + SiLU, as the workload
    t0 = time.perf_counter()
    for k in range(rounds):
        x, g, beta = ins[k]
        pos = [p + k for p in pos0]
        if D == 1:
            st = R.decode_arrays("f32", temporal, conv, x, cw, g, beta, cs, pos, ct, 256, 1, flags,
                                 1.0, out, "bf16", "bf16", "bf16")
        elif not wl.replay:
            st = R.decode_arrays("f32", temporal, conv, x, cw, g, beta, cs, pos, None, 0, 1, flags,
                                 1.0, out, "bf16", "bf16", "bf16", spec_t, spec_c)
            R.commit_arrays("f32", temporal, conv, cs, pos, acc, ct, 256, spec_t, spec_c)
        else:
            # verify with outputs only, then the accepted tokens again into the slot
            st = R.decode_arrays("f32", temporal, conv, x, cw, g, beta, cs, pos, None, 0, 1, flags,
                                 1.0, out, "bf16", "bf16", "bf16")
            o1 = np.zeros((B, 1, 12, 128), np.float32)
            for j in range(D):
                sl = [s if acc[r] > j else -1 for r, s in enumerate(cs)]
                R.decode_arrays("f32", temporal, conv, np.ascontiguousarray(x[:, j:j + 1]), cw,
                                np.ascontiguousarray(g[:, j:j + 1]),
                                np.ascontiguousarray(beta[:, j:j + 1]), sl,
                                [p + j for p in pos], ct, 256, 1, flags, 1.0, o1, "bf16", "bf16",
                                "bf16")
        assert st == 0, st
    dt = time.perf_counter() - t0
    what = "steps" if D == 1 else "verify rounds"
    unit_val = (B * rounds / dt) if D == 1 else (rounds / dt)
    return _cpu_result(unit_val, wl.unit, f"{rounds} {what} of all {B} requests x 12 heads", dt)


def cpu_copy(wl, pairs_per_batch=16, batches=3):
    """Slot copies of the copy workload's batches (the first `pairs_per_batch`
    pairs of each) as a threaded memcpy gather over a compact host pool of the
    same 69-layer slot layout."""
    import numpy as np
    from oracle import lin_state_ref as R
    H, K, C = 12, 128, W.KIMI_K3_TP8.conv_channels
    nslot = 2 * pairs_per_batch
    t_host = np.zeros((wl.layers, nslot, H * K * K), np.uint16)
    c_host = np.zeros((wl.layers, nslot, C * 3), np.uint16)
    src = list(range(pairs_per_batch))
    dst = list(range(pairs_per_batch, nslot))
    R.copy_slots_bytes(t_host, src, dst)  # first touch of every page
    R.copy_slots_bytes(c_host, src, dst)
    t0 = time.perf_counter()
    for _ in range(batches):
        R.copy_slots_bytes(t_host, src, dst)
        R.copy_slots_bytes(c_host, src, dst)
    dt = time.perf_counter() - t0
    moved = 2.0 * batches * pairs_per_batch * wl.slot_bytes
    return _cpu_result(moved / dt / 1e9, "GB/s", f"{batches} batches of {pairs_per_batch} slot copies "
                       f"over {wl.layers} layers (29,039,616 B per slot), read + write counted", dt)


CPU_LEGS = {
    "qwen35_gdn_prefill": lambda wl: cpu_prefill(wl, 16384),
    "mamba2_ssd_prefill": lambda wl: cpu_prefill(wl, 16384),
    "mamba2_ssd_prefill_hd64": lambda wl: cpu_prefill(wl, 8192),
    "kimi_k3_kda_varlen_prefill": lambda wl: cpu_prefill(wl, 40000),
    "kda_long_prefill_131k": lambda wl: cpu_prefill(wl, 24576),
    "kda_recurrent_prefill": lambda wl: cpu_prefill(wl, 16384),
    "kda_decode": lambda wl: cpu_decode(wl, 8),
    "kda_spec_verify4_commit": lambda wl: cpu_decode(wl, 3),
    "kda_spec_verify4_replay": lambda wl: cpu_decode(wl, 3),
    "slot_copy_kimi_k3_69l": cpu_copy,
    "slot_copy_kimi_k3_8l": cpu_copy,
}


def reference_arm(args, dist_info):
    """The oracle as the reference arm: the C restatement in float32 on every
    host thread, one 4096-token request of the headline workload (all 32
    heads) per step."""
    if dist_info["rank"] != 0:
        return
    import numpy as np
    from oracle import lin_state_ref as R
    steps = max(1, args.steps)
    dims = W.QWEN35_GDN
    b = W.make_prefill_batch(dims, [4096], W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=0,
                             gate="uniform", tag=f"{HEADLINE}.ref")
    x, cw, g, beta = (_host_f32(t) for t in (b.x, b.conv_w, b.g, b.beta))
    temporal = np.zeros((4, 32, 128, 128), np.float32)
    conv = np.zeros((4, dims.conv_channels, 3), np.float32)
    out = np.zeros((4096, 32, 128), np.float32)

    def one():
        t0 = time.perf_counter()
        R.prefill_arrays("f32", temporal, conv, x, cw, g, beta, [0, 4096], [0], [1], [0], [2, 3],
                         [0, 2], 64, W.GATE_PER_HEAD, 3, 1.0, out, "f32", "bf16", "f32")
        return time.perf_counter() - t0

    for _ in range(max(0, min(args.warmup, 1))):
        one()
    times = [one() for _ in range(steps)]
    dt = statistics.median(times)
    v = 4096 / dt
    cb = _cpu_result(v, "tok/s", "one 4096-token request of the headline workload (32 heads) per step",
                     sum(times))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": CONFIG_TEXT[HEADLINE], "sample": cb["sample"]},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", default="")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_info = {"world": world, "rank": rank}

    if args.impl == "reference":
        reference_arm(args, dist_info)
        return

    import linear_attention_state_chunked_gb300 as L
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    names = [HEADLINE] + ([] if args.no_extra else DEFAULT_EXTRA)
    if args.only:
        names = args.only.split(",")

    results = {}
    clocks = None
    for i, n in enumerate(names):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # each workload's CPU baseline runs after its GPU legs (the headline's
        # after its end-to-end leg: host allocations made before that leg
        # slowed its host-device copies), on rank 0 of a single-GPU run
        cpu = rank == 0 and world == 1 and not args.no_cpu
        if i == 0:
            with ClockSampler(local) as cs:
                results[n] = run_workload(n, L, dev, args.steps, args.warmup, peaks, stream,
                                          dist_info, e2e=True, cpu=cpu)
            clocks = cs.summary()
        else:
            results[n] = run_workload(n, L, dev, max(3, args.steps), args.warmup, peaks, stream,
                                      dist_info, cpu=cpu)
    if world > 1:
        torch.distributed.barrier()
    head = results[names[0]]
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32",
                "data": "synthetic",
                "config": {**head["config"], "parallelism": f"replicas{world}",
                           "arithmetic": "fp32 state and accumulation; tensor-core operands fp16 "
                                         "with hi/lo splits (GDN) or bf16 (KDA); bf16 inputs",
                           "l2": "inputs larger than L2 (x alone is 805 MB); decode and verify rotate "
                                 "4 pool replicas (432 MB touched per rotation) so no step finds its "
                                 "state in L2"},
                "roofline": {**head["roofline"], "peak_source": peaks["source"]},
                **({"other_launches": head["other_launches"]} if "other_launches" in head else {}),
                "cpu_baseline": head.get("cpu_baseline"),
                "e2e": head.get("e2e"),
                "gpu_launches": head["gpu_launches"],
                "clocks": clocks,
                "workloads": {n: {k: v for k, v in r.items() if k != "config"} | {"config": r["config"]}
                              for n, r in results.items() if n != names[0]}}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
