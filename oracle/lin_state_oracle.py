"""CPU oracle of the gated delta-rule state path: plain, slow, fp64.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module. The library (the CUDA kernels and
their Python binding) never imports it and shares no code with it.

What it computes, token by token and in the order the pages state it:

* Short causal conv of width 4 over the q|k|v projection inputs; the conv
  state is the last 3 inputs ([channels, kernel-1]).
  -- Kimi-K3 notes ("企业官网建设流程全解析"), "Conv state" and
     "Linear的kv cache大小具体计算逻辑" (conv state [3, Q+K+V]).
* The KDA / GDN update
      S' = S Diag(alpha) + d k^T,   d = beta (v - (S Diag(alpha)) k),
  with alpha a vector over the key channels (KDA) or one scalar per head
  (GDN), followed by the output o = S' q.
  -- Kimi-K3 notes, "Speculative decoding" (the recurrent update) and the
     "g" ring paragraph (GDN g is one scalar per head, KDA g has 128 values).
* Additive (Mamba2 SSD) form, with FLAG_UPDATE_ADDITIVE: the same state,
  pool and tracking, but the update is the plain state-space recurrence
      S' = S Diag(alpha) + beta v k^T
  (no delta correction). The pages write it as S_new = A x S_old + B x x
  with activations (hidden_states, dt, B, C); in this layout alpha =
  exp(dt A) per head, beta = dt, k = B, v = x, q = C.
  -- MambaRadixCache page section 9.3 ("什么是输入激活值").
* Warm or cold start from a slot: has_initial_state = 1 loads the slot,
  0 starts from zero.
  -- Qwen3.5 Linear-State Prefix Cache, section 5.1 step 5 and section 6.4.
* Snapshots of (temporal, conv) into track slots at every absolute position
  that is a multiple of the track stride, cycling through the request's list.
  -- Ping-Pong page, "状态追踪机制" and the 1200-token long-request flow;
     MambaRadixCache page section 3.4 (ping-pong track buffer).
* Decode track at every total length that is a multiple of the interval.
  -- Kimi-K3 notes, "--mamba-track-interval" (prompt 1000 -> 1024, 1280, 1536).
* Speculative verify into a per-step buffer with the main slot untouched,
  then commit main = buffer[accepted - 1].
  -- MambaRadixCache page sections 8.3, 8.4, 8.6.
* A verify that keeps no per-step states writes only the drafts' outputs,
  carrying the state unrounded across the drafts (nothing is stored between
  them); its commit re-runs the accepted prefix.
  -- Kimi-K3 notes, "ReplaySSM"; MambaRadixCache page sections 9.2 - 9.10.
* Slot copies (fork / COW) and restore with has_initial_state.
  -- MambaRadixCache page section 3.2 (copy_from);
     Qwen3.5 Linear-State Prefix Cache sections 6.1, 6.4.

Readings taken where the pages are silent (listed with reasons in the design
notes): temporal layout [H][V][K]; conv state [C][3] with [c][0] the oldest
input; conv tap w[c][3] multiplies the current token; no conv bias; optional
SiLU after the conv; q and k L2-normalised per head with eps = 1e-6 inside the
square root; q scaled by q_scale after normalisation; the state is rounded to
the pool's storage dtype only where it is written to memory (prefill) or after
every token (decode and verify, which read and write the pool per token); a
verify without per-step states stores nothing between drafts, so it carries
the state unrounded, as a prefill does.

Storage dtypes: "f32", "bf16", or "f64" (no rounding; used by the pins).
"""

from __future__ import annotations

import numpy as np

GATE_PER_HEAD = 0
GATE_PER_KEY = 1

FLAG_QK_L2NORM = 1
FLAG_CONV_SILU = 2
FLAG_VALIDATE = 4
FLAG_UPDATE_ADDITIVE = 32

# Device status bits, as the library documents them.
ST_BAD_SLOT = 1
ST_BAD_PREFIX = 2
ST_TRACK_ALIAS = 4
ST_BAD_SEQLEN = 8
ST_COPY_ALIAS = 16
ST_BAD_ACCEPT = 64
ST_BAD_TREE = 256  # a draft's parent outside [-1, j), or an accepted node outside [-1, n_draft)

L2_EPS = 1e-6


# ----------------------------------------------------------------------------
# Rounding into storage dtypes (round to nearest, ties to even).
# ----------------------------------------------------------------------------

def round_to(x, dtype: str):
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        # bfloat16: 8 significant bits, exponent range of float32.
        m, e = np.frexp(x)
        q = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
        tiny = np.abs(x) < 2.0 ** -126
        q = np.where(tiny, np.rint(np.ldexp(x, 133)) * 2.0 ** -133, q)
        return q
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# Pool: temporal [layer][slot][H][V][K], conv [layer][slot][C][W-1].
# ----------------------------------------------------------------------------

def make_pool(num_layers, num_slots, H, K, V, C, W=4, state_dtype="f32",
              conv_dtype="f32", fill=0.0):
    return {
        "temporal": np.full((num_layers, num_slots, H, V, K), fill, np.float64),
        "conv": np.full((num_layers, num_slots, C, W - 1), fill, np.float64),
        "state_dtype": state_dtype,
        "conv_dtype": conv_dtype,
    }


def slot_bytes(num_layers, H, K, V, C, W, state_esize, conv_esize):
    """Bytes of one slot over all layers: temporal [H][V][K] plus conv
    [C][W-1] per layer (MambaRadixCache page section 1.3: one slot holds the
    conv and temporal state of every linear layer)."""
    return num_layers * (H * V * K * state_esize + C * (W - 1) * conv_esize)


# ----------------------------------------------------------------------------
# One token of one request: conv, activation, split, normalisation, update.
# ----------------------------------------------------------------------------

def _silu(y):
    return y / (1.0 + np.exp(-y))


def token_step(S, cw, x_t, conv_w, g_t, beta_t, H, K, V, gate_mode, flags, q_scale):
    """Advance one token.

    S      [H][V][K] state before the token
    cw     [C][3]    conv window: the last 3 inputs, cw[:, 0] the oldest
    x_t    [C]       this token's q|k|v projection input
    conv_w [C][4]    conv taps; conv_w[:, 3] multiplies the current input
    g_t    [H] (GDN) or [H][K] (KDA): log alpha
    beta_t [H]
    Returns (S_new, cw_new, o [H][V]).
    """
    # Short conv over (3 stored inputs, current input).
    y = (conv_w[:, 0] * cw[:, 0] + conv_w[:, 1] * cw[:, 1]
         + conv_w[:, 2] * cw[:, 2] + conv_w[:, 3] * x_t)
    cw_new = np.stack([cw[:, 1], cw[:, 2], x_t], axis=1)
    if flags & FLAG_CONV_SILU:
        y = _silu(y)
    q = y[:H * K].reshape(H, K).copy()
    k = y[H * K:2 * H * K].reshape(H, K).copy()
    v = y[2 * H * K:].reshape(H, V)
    if flags & FLAG_QK_L2NORM:
        q = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + L2_EPS)
        k = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + L2_EPS)
    q = q * q_scale

    # alpha: one scalar per head (GDN) or one value per key channel (KDA).
    if gate_mode == GATE_PER_HEAD:
        alpha = np.exp(g_t)[:, None] * np.ones((H, K))
    else:
        alpha = np.exp(g_t)
    # S Diag(alpha): column c of S (key channel c) scaled by alpha[c].
    S_dec = S * alpha[:, None, :]
    # d = beta (v - (S Diag(alpha)) k); the additive form drops the prediction
    if flags & FLAG_UPDATE_ADDITIVE:
        d = beta_t[:, None] * v
    else:
        pred = np.einsum("hvk,hk->hv", S_dec, k)
        d = beta_t[:, None] * (v - pred)
    # S' = S Diag(alpha) + d k^T
    S_new = S_dec + d[:, :, None] * k[:, None, :]
    # o = S' q
    o = np.einsum("hvk,hk->hv", S_new, q)
    return S_new, cw_new, o


def _in_range(s, n):
    return 0 <= s < n


# ----------------------------------------------------------------------------
# Prefill over a varlen batch.
# ----------------------------------------------------------------------------

def prefill(pool, layer, x, conv_w, g, beta, cu_seqlens, prefix_len, slot,
            has_initial_state, track_slots, cu_track, track_stride, gate_mode,
            flags, q_scale=1.0, out_dtype="f32", H=None, K=None, V=None,
            chunk_align=64, out=None):
    """Process each request's extend tokens from its slot state.

    x [T][C], g [T][H] or [T][H][K], beta [T][H]; cu_seqlens [B+1];
    prefix_len[r] = tokens already in the state (absolute position of the
    first extend token); has_initial_state[r] 1 = warm from slot[r], 0 = cold;
    track_slots[cu_track[r]:cu_track[r+1]] = the request's track list.
    Returns (out [T][H][V] as float64 values of out_dtype, status bits).
    The pool is updated in place.
    """
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    if H is None:
        H, V, K = temporal.shape[2], temporal.shape[3], temporal.shape[4]
    T = x.shape[0]
    if out is None:
        out = np.zeros((T, H, V), np.float64)
    status = 0
    B = len(slot)
    for r in range(B):
        s = int(slot[r])
        if s < 0:
            continue  # padding entry (slot ids below zero are no-ops)
        if not _in_range(s, num_slots):
            status |= ST_BAD_SLOT
            continue
        bos, eos = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        if bos < 0 or eos < bos or eos > T:
            status |= ST_BAD_SEQLEN
            continue
        P = int(prefix_len[r])
        if P < 0 or P % chunk_align != 0:
            status |= ST_BAD_PREFIX
            continue
        tracks = [int(t) for t in track_slots[int(cu_track[r]):int(cu_track[r + 1])]]
        if any(t >= num_slots for t in tracks):
            status |= ST_BAD_SLOT
            continue
        if any(t == s for t in tracks):
            status |= ST_TRACK_ALIAS
            continue

        if int(has_initial_state[r]):
            S = temporal[layer, s].copy()
            cw = conv[layer, s].copy()
        else:
            S = np.zeros((H, V, K))
            cw = np.zeros_like(conv[layer, s])
        j = 0
        for i in range(eos - bos):
            t = bos + i
            S, cw, o = token_step(S, cw, x[t], conv_w, g[t], beta[t], H, K, V,
                                  gate_mode, flags, q_scale)
            out[t] = round_to(o, out_dtype)
            p = P + i + 1  # tokens now folded into S
            if track_stride > 0 and tracks and p % track_stride == 0:
                dst = tracks[j % len(tracks)]
                if dst >= 0:
                    temporal[layer, dst] = round_to(S, pool["state_dtype"])
                    conv[layer, dst] = round_to(cw, pool["conv_dtype"])
                j += 1
        temporal[layer, s] = round_to(S, pool["state_dtype"])
        conv[layer, s] = round_to(cw, pool["conv_dtype"])
    return out, status


# ----------------------------------------------------------------------------
# Decode: one token per request in place, or n_draft tokens into a buffer.
# ----------------------------------------------------------------------------

def make_spec_buffer(num_layers, batch, n_draft, H, K, V, C, W=4, fill=0.0):
    return {
        "temporal": np.full((num_layers, batch, n_draft, H, V, K), fill, np.float64),
        "conv": np.full((num_layers, batch, n_draft, C, W - 1), fill, np.float64),
    }


def decode(pool, layer, x, conv_w, g, beta, slot, pos, track_slot,
           track_interval, gate_mode, flags, q_scale=1.0, out_dtype="f32",
           spec=None, out=None, parent=None):
    """x [B][D][C]; g [B][D][H] or [B][D][H][K]; beta [B][D][H].

    D == 1: the slot is read, advanced one token and written back; when the
    state then covers a multiple of track_interval tokens it is also copied
    into track_slot[r].
    D > 1 (verify): D tokens run from the slot state; the state after step j
    goes to spec[layer][r][j]; the slot is not modified. With parent
    [B][D] (a draft tree, MambaRadixCache page 8.3 and 9.6,
    retrieve_parent_token): draft j starts from the state and conv window
    after draft parent[r][j] (-1: the slot's), so a chain is parent[j] = j-1;
    a parent outside [-1, j) skips the request with ST_BAD_TREE.
    The state is rounded to the pool's dtype after every token, as a decode
    that reads and writes the pool per token would.
    """
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    H, V, K = temporal.shape[2], temporal.shape[3], temporal.shape[4]
    B, D = x.shape[0], x.shape[1]
    if out is None:
        out = np.zeros((B, D, H, V), np.float64)
    sd, cd = pool["state_dtype"], pool["conv_dtype"]
    status = 0
    for r in range(B):
        s = int(slot[r])
        if s < 0:
            continue
        if not _in_range(s, num_slots):
            status |= ST_BAD_SLOT
            continue
        ts = int(track_slot[r]) if track_slot is not None else -1
        if ts >= num_slots:
            status |= ST_BAD_SLOT
            continue
        if ts == s:
            status |= ST_TRACK_ALIAS
            continue
        if parent is not None and D > 1 and any(
                not (-1 <= int(parent[r][j]) < j) for j in range(D)):
            status |= ST_BAD_TREE
            continue
        S = temporal[layer, s].copy()
        cw = conv[layer, s].copy()
        for j in range(D):
            if parent is not None and D > 1:
                pj = int(parent[r][j])
                if pj < 0:
                    S, cw = temporal[layer, s].copy(), conv[layer, s].copy()
                else:
                    S = spec["temporal"][layer, r, pj].copy()
                    cw = spec["conv"][layer, r, pj].copy()
            S, cw, o = token_step(S, cw, x[r, j], conv_w, g[r, j], beta[r, j],
                                  H, K, V, gate_mode, flags, q_scale)
            S = round_to(S, sd)
            cw = round_to(cw, cd)
            out[r, j] = round_to(o, out_dtype)
            if D == 1:
                temporal[layer, s] = S
                conv[layer, s] = cw
                n = int(pos[r]) + 1
                if ts >= 0 and track_interval > 0 and n % track_interval == 0:
                    temporal[layer, ts] = S
                    conv[layer, ts] = cw
            else:
                spec["temporal"][layer, r, j] = S
                spec["conv"][layer, r, j] = cw
    return out, status


def verify_outputs(pool, layer, x, conv_w, g, beta, slot, gate_mode, flags, q_scale=1.0,
                   out_dtype="f32", out=None):
    """Outputs of a verify that keeps no per-step states: the replay form of
    speculative decoding (Kimi-K3 notes, "ReplaySSM"; MambaRadixCache page
    9.2 - 9.10), whose commit re-runs the accepted prefix later.

    x [B][D][C]; g [B][D][H] or [B][D][H][K]; beta [B][D][H]. The D drafts of
    request r run in order from the state and window in slot[r]. Nothing is
    stored between drafts, so the state is carried unrounded across them, as
    inside a prefill call (only the outputs are written, rounded to
    out_dtype). The pool is not modified. Returns (out [B][D][H][V], status).
    """
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    H, V, K = temporal.shape[2], temporal.shape[3], temporal.shape[4]
    B, D = x.shape[0], x.shape[1]
    if out is None:
        out = np.zeros((B, D, H, V), np.float64)
    status = 0
    for r in range(B):
        s = int(slot[r])
        if s < 0:
            continue
        if not _in_range(s, num_slots):
            status |= ST_BAD_SLOT
            continue
        S = temporal[layer, s].copy()
        cw = conv[layer, s].copy()
        for j in range(D):
            S, cw, o = token_step(S, cw, x[r, j], conv_w, g[r, j], beta[r, j],
                                  H, K, V, gate_mode, flags, q_scale)
            out[r, j] = round_to(o, out_dtype)
    return out, status


def spec_commit(pool, spec, layer_begin, layer_end, slot, pos, accept_len,
                track_slot, track_interval, n_draft, parent=None, accept_node=None):
    """main[slot] = buffer[accepted - 1] for every layer in the range; when the
    accepted tokens cross a multiple of track_interval, the state at that
    boundary (the largest one crossed) also goes to track_slot.
    accept_len == 0 leaves everything unchanged.
    A draft tree (parent [B][D], accept_node [B]): the accepted path ends at
    node accept_node[r] (-1: nothing accepted) and runs back through its
    parents to the root; its length plays the part of accept_len, and the
    node at depth n - pos on it holds the boundary state."""
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    status = 0
    for r in range(len(slot)):
        s = int(slot[r])
        if s < 0:
            continue
        if not _in_range(s, num_slots):
            status |= ST_BAD_SLOT
            continue
        if parent is not None:
            node = int(accept_node[r])
            if node < -1 or node >= n_draft:
                status |= ST_BAD_TREE
                continue
            path = []  # root first
            while node >= 0:
                path.insert(0, node)
                node = int(parent[r][node])
            a = len(path)
        else:
            a = int(accept_len[r])
            path = list(range(a)) if 0 <= a <= n_draft else []
        if a < 0 or a > n_draft:
            status |= ST_BAD_ACCEPT
            continue
        if a == 0:
            continue
        ts = int(track_slot[r]) if track_slot is not None else -1
        if ts >= num_slots:
            status |= ST_BAD_SLOT
            continue
        if ts == s:
            status |= ST_TRACK_ALIAS
            continue
        p = int(pos[r])
        boundary = None
        if ts >= 0 and track_interval > 0:
            n = ((p + a) // track_interval) * track_interval
            if n > p:
                boundary = n
        for layer in range(layer_begin, layer_end):
            temporal[layer, s] = spec["temporal"][layer, r, path[a - 1]]
            conv[layer, s] = spec["conv"][layer, r, path[a - 1]]
            if boundary is not None:
                temporal[layer, ts] = spec["temporal"][layer, r, path[boundary - p - 1]]
                conv[layer, ts] = spec["conv"][layer, r, path[boundary - p - 1]]
    return status


# ----------------------------------------------------------------------------
# Slot copies and restore.
# ----------------------------------------------------------------------------

def copy_slots(pool, src, dst, layer_begin, layer_end, flags=0):
    """conv[l][dst] = conv[l][src]; temporal[l][dst] = temporal[l][src] for
    every pair and every layer in the range (MambaRadixCache page 3.2).
    Negative ids are padding. With FLAG_VALIDATE a pair whose dst is another
    pair's dst or src is skipped and ST_COPY_ALIAS is raised."""
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    n = len(src)
    status = 0
    skip = [False] * n
    for i in range(n):
        s, d = int(src[i]), int(dst[i])
        if s < 0 or d < 0:
            skip[i] = True
            continue
        if not (_in_range(s, num_slots) and _in_range(d, num_slots)):
            status |= ST_BAD_SLOT
            skip[i] = True
            continue
        if flags & FLAG_VALIDATE:
            for j in range(n):
                if j != i and (int(dst[j]) == d or int(src[j]) == d):
                    status |= ST_COPY_ALIAS
                    skip[i] = True
                    break
    # Reads all happen before writes for a valid (non-aliasing) batch.
    snap = [(temporal[layer_begin:layer_end, int(src[i])].copy(),
             conv[layer_begin:layer_end, int(src[i])].copy())
            if not skip[i] else None for i in range(n)]
    for i in range(n):
        if skip[i]:
            continue
        d = int(dst[i])
        temporal[layer_begin:layer_end, d] = snap[i][0]
        conv[layer_begin:layer_end, d] = snap[i][1]
    return status


def restore(pool, ops, has_initial_state):
    """Qwen3.5 Linear-State Prefix Cache, sections 6.1 and 6.4: for each op
    (linear_state_id, restore_requested, restore_src_slot_id):
      requested and the source resolves -> copy src into the live slot across
                                           all layers, has_initial_state = 1
      requested and the source is missing or out of range -> 0 (cold start)
      not requested -> has_initial_state left as it was.
    A negative live id is padding."""
    temporal, conv = pool["temporal"], pool["conv"]
    num_slots = temporal.shape[1]
    status = 0
    for i, (live, requested, src) in enumerate(ops):
        live, requested, src = int(live), int(requested), int(src)
        if live < 0:
            continue
        if not _in_range(live, num_slots):
            status |= ST_BAD_SLOT
            if requested:
                has_initial_state[i] = 0
            continue
        if not requested:
            continue
        if _in_range(src, num_slots):
            temporal[:, live] = temporal[:, src].copy()
            conv[:, live] = conv[:, src].copy()
            has_initial_state[i] = 1
        else:
            has_initial_state[i] = 0
    return status
