/*
 * Plain C restatement of the oracle's token recurrence (oracle/lin_state_oracle.py),
 * for the CPU baseline timed beside the GPU path.
 *
 * TEST INFRASTRUCTURE. Only the test suite and the benchmark's CPU legs load
 * this code (through oracle/lin_state_ref.py). It shares nothing with the CUDA
 * library and the library never loads it.
 *
 * It computes, token by token and in the pages' order, what the Python oracle
 * computes (see that module's header for the passages):
 *   - the width-4 causal conv over the q|k|v projection inputs, whose last 3
 *     inputs form the conv state (Kimi-K3 notes, "Conv state");
 *   - optional SiLU, per-head L2 norms of q and k, q scale;
 *   - the update S' = S Diag(alpha) + d k^T, d = beta (v - S Diag(alpha) k),
 *     then o = S' q (Kimi-K3 notes, "Speculative decoding"); with
 *     FLAG_UPDATE_ADDITIVE, d = beta v (MambaRadixCache page 9.3);
 *   - warm or cold start (Qwen3.5 Linear-State Prefix Cache 5.1, 6.4),
 *     snapshots at multiples of the track stride into the request's cyclic
 *     track list (Ping-Pong page, chunk-boundary tracking), the final
 *     write-back, and the decode track at multiples of the interval (Kimi-K3
 *     notes, "--mamba-track-interval");
 *   - verify into a per-step buffer and the commit main = buffer[accepted-1]
 *     (MambaRadixCache page 8.3 - 8.6); batched slot copies (3.2).
 * Storage rounding (to bf16 or fp32) happens where the Python oracle rounds.
 *
 * The file is compiled twice: with REAL = double (checked against the
 * Python oracle) and REAL = float (the timed baseline). Independent
 * (request, head) pairs run on a pool of POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL double
#endif
#ifndef SUFFIX
#define SUFFIX f64
#endif
#define CAT2(a, b) a##_##b
#define CAT(a, b) CAT2(a, b)
#define NAME(f) CAT(f, SUFFIX)

typedef REAL real;
#ifdef REAL_FLOAT
#define EXP expf
#define SQRT sqrtf
#else
#define EXP exp
#define SQRT sqrt
#endif

enum { GATE_PER_HEAD = 0, GATE_PER_KEY = 1 };
enum { FLAG_QK_L2NORM = 1, FLAG_CONV_SILU = 2, FLAG_UPDATE_ADDITIVE = 32 };
enum { ST_BAD_SLOT = 1, ST_BAD_PREFIX = 2, ST_TRACK_ALIAS = 4, ST_BAD_SEQLEN = 8 };
enum { ROUND_NONE = 0, ROUND_F32 = 1, ROUND_BF16 = 2 };

/* Round to nearest, ties to even, into the storage type: bf16 keeps 8
 * significant bits with the exponent range of fp32. */
static real round_to(real x, int mode) {
  if (mode == ROUND_F32) return (real)(float)x;
#ifdef REAL_FLOAT
  if (mode == ROUND_BF16) {
    /* fp32 and bf16 share the exponent: round the 16 low mantissa bits away */
    uint32_t u;
    memcpy(&u, &x, sizeof(u));
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    float f;
    memcpy(&f, &u, sizeof(f));
    return f;
  }
#else
  if (mode == ROUND_BF16) {
    if (fabs((double)x) < ldexp(1.0, -126)) return (real)(rint(ldexp((double)x, 133)) * ldexp(1.0, -133));
    int e;
    const double m = frexp((double)x, &e);
    return (real)ldexp(rint(ldexp(m, 8)), e - 8);
  }
#endif
  return x;
}

/* ---- a pool of threads working through units 0 .. n-1 ------------------- */
typedef void (*unit_fn)(void* ctx, int64_t unit);
typedef struct {
  unit_fn fn;
  void* ctx;
  int64_t n;
  int64_t next; /* atomic */
} work_t;

static void* worker(void* p) {
  work_t* w = (work_t*)p;
  for (;;) {
    const int64_t u = __atomic_fetch_add(&w->next, 1, __ATOMIC_RELAXED);
    if (u >= w->n) break;
    w->fn(w->ctx, u);
  }
  return NULL;
}

static void run_units(unit_fn fn, void* ctx, int64_t n, int nthreads) {
  work_t w = {fn, ctx, n, 0};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  pthread_t tid[1024];
  int started = 0;
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&tid[started], NULL, worker, &w) == 0) ++started;
  worker(&w);
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
}

/* ---- one head of one token ------------------------------------------------
 * The head's channels: q [h*K, h*K+K), k [H*K + h*K, ..), v [2*H*K + h*V, ..).
 * win[3][CH] holds the last 3 inputs of those channels (win[0] the oldest),
 * CH = 2K + V in the order q | k | v. S is [V][K]. */
typedef struct {
  int H, K, V, C, gate_mode, flags;
  real q_scale;
} shape_t;

static int64_t head_channel(const shape_t* s, int h, int cl) {
  if (cl < s->K) return (int64_t)h * s->K + cl;
  if (cl < 2 * s->K) return (int64_t)s->H * s->K + (int64_t)h * s->K + (cl - s->K);
  return 2 * (int64_t)s->H * s->K + (int64_t)h * s->V + (cl - 2 * s->K);
}

/* x_t: the token's C inputs; g_t: H (per head) or H*K (per key) log-decays;
 * beta_t: H values; y: scratch [CH + K] (conv outputs, then alpha); o: [V]. */
static void head_token(const shape_t* s, int h, real* S, real* win, const real* x_t,
                       const real* conv_w, const real* g_t, const real* beta_t, real* y, real* o) {
  const int K = s->K, V = s->V, CH = 2 * K + V;
  for (int cl = 0; cl < CH; ++cl) {
    const int64_t c = head_channel(s, h, cl);
    const real xn = x_t[c];
    const real* w = conv_w + 4 * c;
    real v = w[0] * win[cl] + w[1] * win[CH + cl] + w[2] * win[2 * CH + cl] + w[3] * xn;
    win[cl] = win[CH + cl];
    win[CH + cl] = win[2 * CH + cl];
    win[2 * CH + cl] = xn;
    if (s->flags & FLAG_CONV_SILU) v = v / ((real)1 + EXP(-v));
    y[cl] = v;
  }
  real* q = y;
  real* k = y + K;
  const real* vv = y + 2 * K;
  if (s->flags & FLAG_QK_L2NORM) {
    real sq = 0, sk = 0;
    for (int c = 0; c < K; ++c) {
      sq += q[c] * q[c];
      sk += k[c] * k[c];
    }
    const real rq = (real)1 / SQRT(sq + (real)1e-6), rk = (real)1 / SQRT(sk + (real)1e-6);
    for (int c = 0; c < K; ++c) {
      q[c] *= rq;
      k[c] *= rk;
    }
  }
  for (int c = 0; c < K; ++c) q[c] *= s->q_scale;
  /* alpha = exp(g): one value per head (GDN) or per key channel (KDA) */
  real* alpha = y + CH;
  for (int c = 0; c < K; ++c) alpha[c] = EXP(s->gate_mode == GATE_PER_KEY ? g_t[(int64_t)h * K + c] : g_t[h]);
  const real beta = beta_t[h];
  for (int v = 0; v < V; ++v) {
    real* row = S + (int64_t)v * K;
    /* S Diag(alpha): key channel c of the row scaled by alpha_c */
    for (int c = 0; c < K; ++c) row[c] *= alpha[c];
    real d;
    if (s->flags & FLAG_UPDATE_ADDITIVE) {
      d = beta * vv[v];
    } else {
      real pred = 0;
      for (int c = 0; c < K; ++c) pred += row[c] * k[c];
      d = beta * (vv[v] - pred);
    }
    real out = 0;
    for (int c = 0; c < K; ++c) {
      row[c] += d * k[c];
      out += row[c] * q[c];
    }
    o[v] = out;
  }
}

/* ---- prefill ---------------------------------------------------------------- */
typedef struct {
  shape_t s;
  int num_slots, state_round, conv_round, out_round, track_stride;
  real* temporal; /* [slots][H][V][K] */
  real* conv;     /* [slots][C][3] */
  const real *x, *conv_w, *g, *beta;
  const int64_t *cu_seqlens, *prefix_len, *slot, *has_initial_state, *track_slots, *cu_track;
  real* out; /* [T][H][V] */
  const int32_t* valid; /* per request: 1 = run */
} prefill_ctx;

static void store_state(const prefill_ctx* p, int dst, int h, const real* S, const real* win) {
  const shape_t* s = &p->s;
  const int K = s->K, V = s->V, CH = 2 * K + V;
  real* t = p->temporal + ((int64_t)dst * s->H + h) * V * K;
  for (int64_t i = 0; i < (int64_t)V * K; ++i) t[i] = round_to(S[i], p->state_round);
  for (int cl = 0; cl < CH; ++cl) {
    real* c = p->conv + ((int64_t)dst * s->C + head_channel(s, h, cl)) * 3;
    for (int j = 0; j < 3; ++j) c[j] = round_to(win[j * CH + cl], p->conv_round);
  }
}

static void prefill_unit(void* ctx, int64_t u) {
  const prefill_ctx* p = (const prefill_ctx*)ctx;
  const shape_t* s = &p->s;
  const int H = s->H, K = s->K, V = s->V, CH = 2 * K + V;
  const int r = (int)(u / H), h = (int)(u % H);
  if (!p->valid[r]) return;
  const int slot = (int)p->slot[r];
  real* S = (real*)calloc((size_t)V * K, sizeof(real));
  real* win = (real*)calloc((size_t)3 * CH, sizeof(real));
  real* y = (real*)malloc(sizeof(real) * (CH + K));
  real* o = (real*)malloc(sizeof(real) * V);
  if (p->has_initial_state[r]) {
    memcpy(S, p->temporal + ((int64_t)slot * H + h) * V * K, sizeof(real) * V * K);
    for (int cl = 0; cl < CH; ++cl) {
      const real* c = p->conv + ((int64_t)slot * s->C + head_channel(s, h, cl)) * 3;
      for (int j = 0; j < 3; ++j) win[j * CH + cl] = c[j];
    }
  }
  const int64_t bos = p->cu_seqlens[r], eos = p->cu_seqlens[r + 1];
  const int64_t P = p->prefix_len[r];
  const int64_t t0 = p->cu_track ? p->cu_track[r] : 0;
  const int64_t nt = p->cu_track ? p->cu_track[r + 1] - t0 : 0;
  const int64_t gstride = s->gate_mode == GATE_PER_KEY ? (int64_t)H * K : H;
  int64_t snap = 0;
  for (int64_t t = bos; t < eos; ++t) {
    head_token(s, h, S, win, p->x + t * s->C, p->conv_w, p->g + t * gstride, p->beta + t * H, y, o);
    real* ot = p->out + (t * H + h) * V;
    for (int v = 0; v < V; ++v) ot[v] = round_to(o[v], p->out_round);
    const int64_t n = P + (t - bos) + 1;
    if (p->track_stride > 0 && nt > 0 && n % p->track_stride == 0) {
      const int64_t dst = p->track_slots[t0 + snap % nt];
      if (dst >= 0) store_state(p, (int)dst, h, S, win);
      ++snap;
    }
  }
  store_state(p, slot, h, S, win);
  free(S);
  free(win);
  free(y);
  free(o);
}

/* Returns the status bits (the Python oracle's): bad slot, bad sequence
 * bounds, misaligned prefix, a track slot out of range or equal to the live
 * slot; such requests are skipped. */
int NAME(lin_ref_prefill)(int H, int K, int V, int C, int num_slots, real* temporal, real* conv,
                          int state_round, int conv_round, const real* x, const real* conv_w,
                          const real* g, const real* beta, int B, int64_t T,
                          const int64_t* cu_seqlens, const int64_t* prefix_len, const int64_t* slot,
                          const int64_t* has_initial_state, const int64_t* track_slots,
                          const int64_t* cu_track, int track_stride, int gate_mode, int flags,
                          double q_scale, int out_round, real* out, int nthreads) {
  int status = 0;
  int32_t* valid = (int32_t*)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
  for (int r = 0; r < B; ++r) {
    const int64_t sl = slot[r];
    if (sl < 0) continue;
    if (sl >= num_slots) { status |= ST_BAD_SLOT; continue; }
    const int64_t bos = cu_seqlens[r], eos = cu_seqlens[r + 1];
    if (bos < 0 || eos < bos || eos > T) { status |= ST_BAD_SEQLEN; continue; }
    if (prefix_len[r] < 0 || prefix_len[r] % 64) { status |= ST_BAD_PREFIX; continue; }
    int bad = 0;
    if (cu_track)
      for (int64_t i = cu_track[r]; i < cu_track[r + 1]; ++i) {
        if (track_slots[i] >= num_slots) { status |= ST_BAD_SLOT; bad = 1; break; }
        if (track_slots[i] == sl) { status |= ST_TRACK_ALIAS; bad = 1; break; }
      }
    valid[r] = !bad;
  }
  prefill_ctx p = {{H, K, V, C, gate_mode, flags, (real)q_scale}, num_slots, state_round, conv_round,
                   out_round, track_stride, temporal, conv, x, conv_w, g, beta, cu_seqlens, prefix_len,
                   slot, has_initial_state, track_slots, cu_track, out, valid};
  run_units(prefill_unit, &p, (int64_t)B * H, nthreads);
  free(valid);
  return status;
}

/* ---- decode / verify -----------------------------------------------------------
 * D == 1: the slot advances one token in place; when the state then covers a
 * multiple of track_interval tokens it is also stored in track_slot[r].
 * D > 1: D tokens from the slot state, the state after step j into
 * spec[r][j] (when a spec buffer is given), the slot untouched. The state is
 * rounded to the storage dtype after every token. */
typedef struct {
  shape_t s;
  int num_slots, state_round, conv_round, out_round, D, track_interval;
  real *temporal, *conv;
  const real *x, *conv_w, *g, *beta;
  const int64_t *slot, *pos, *track_slot;
  real* out;                /* [B][D][H][V] */
  real *spec_t, *spec_c;    /* [B][D][H][V][K], [B][D][C][3] or NULL */
  const int32_t* valid;
} decode_ctx;

static void decode_unit(void* ctx, int64_t u) {
  const decode_ctx* p = (const decode_ctx*)ctx;
  const shape_t* s = &p->s;
  const int H = s->H, K = s->K, V = s->V, C = s->C, CH = 2 * K + V, D = p->D;
  const int r = (int)(u / H), h = (int)(u % H);
  if (!p->valid[r]) return;
  const int slot = (int)p->slot[r];
  real* S = (real*)malloc(sizeof(real) * V * K);
  real* win = (real*)malloc(sizeof(real) * 3 * CH);
  real* y = (real*)malloc(sizeof(real) * (CH + K));
  real* o = (real*)malloc(sizeof(real) * V);
  real* tslot = p->temporal + ((int64_t)slot * H + h) * V * K;
  memcpy(S, tslot, sizeof(real) * V * K);
  for (int cl = 0; cl < CH; ++cl) {
    const real* c = p->conv + ((int64_t)slot * C + head_channel(s, h, cl)) * 3;
    for (int j = 0; j < 3; ++j) win[j * CH + cl] = c[j];
  }
  const int64_t gstride = s->gate_mode == GATE_PER_KEY ? (int64_t)H * K : H;
  for (int j = 0; j < D; ++j) {
    const int64_t rj = (int64_t)r * D + j;
    head_token(s, h, S, win, p->x + rj * C, p->conv_w, p->g + rj * gstride, p->beta + rj * H, y, o);
    for (int64_t i = 0; i < (int64_t)V * K; ++i) S[i] = round_to(S[i], p->state_round);
    for (int i = 0; i < 3 * CH; ++i) win[i] = round_to(win[i], p->conv_round);
    real* ot = p->out + (rj * H + h) * V;
    for (int v = 0; v < V; ++v) ot[v] = round_to(o[v], p->out_round);
    int dsts[2] = {-1, -1};
    real *bt = NULL, *bc = NULL;
    if (D == 1) {
      dsts[0] = slot;
      const int64_t n = p->pos[r] + 1;
      const int64_t ts = p->track_slot ? p->track_slot[r] : -1;
      if (ts >= 0 && p->track_interval > 0 && n % p->track_interval == 0) dsts[1] = (int)ts;
    } else if (p->spec_t) {
      bt = p->spec_t + (rj * H + h) * V * K;
      bc = p->spec_c + rj * C * 3;
    }
    for (int q = 0; q < 2; ++q)
      if (dsts[q] >= 0) {
        memcpy(p->temporal + ((int64_t)dsts[q] * H + h) * V * K, S, sizeof(real) * V * K);
        for (int cl = 0; cl < CH; ++cl) {
          real* c = p->conv + ((int64_t)dsts[q] * C + head_channel(s, h, cl)) * 3;
          for (int m = 0; m < 3; ++m) c[m] = win[m * CH + cl];
        }
      }
    if (bt) {
      memcpy(bt, S, sizeof(real) * V * K);
      for (int cl = 0; cl < CH; ++cl) {
        real* c = bc + head_channel(s, h, cl) * 3;
        for (int m = 0; m < 3; ++m) c[m] = win[m * CH + cl];
      }
    }
  }
  free(S);
  free(win);
  free(y);
  free(o);
}

int NAME(lin_ref_decode)(int H, int K, int V, int C, int num_slots, real* temporal, real* conv,
                         int state_round, int conv_round, const real* x, const real* conv_w,
                         const real* g, const real* beta, int B, int D, const int64_t* slot,
                         const int64_t* pos, const int64_t* track_slot, int track_interval,
                         int gate_mode, int flags, double q_scale, int out_round, real* out,
                         real* spec_t, real* spec_c, int nthreads) {
  int status = 0;
  int32_t* valid = (int32_t*)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
  for (int r = 0; r < B; ++r) {
    const int64_t sl = slot[r];
    if (sl < 0) continue;
    if (sl >= num_slots) { status |= ST_BAD_SLOT; continue; }
    const int64_t ts = track_slot ? track_slot[r] : -1;
    if (ts >= num_slots) { status |= ST_BAD_SLOT; continue; }
    if (ts == sl) { status |= ST_TRACK_ALIAS; continue; }
    valid[r] = 1;
  }
  decode_ctx p = {{H, K, V, C, gate_mode, flags, (real)q_scale}, num_slots, state_round, conv_round,
                  out_round, D, track_interval, temporal, conv, x, conv_w, g, beta, slot, pos,
                  track_slot, out, spec_t, spec_c, valid};
  run_units(decode_unit, &p, (int64_t)B * H, nthreads);
  free(valid);
  return status;
}

/* ---- commit and slot copies -------------------------------------------------
 * Commit: for a = accept_len[r] in 1..D, slot[r] <- spec[r][a-1]; when
 * (pos, pos + a] holds a multiple of the interval, the largest such n also
 * goes to track_slot[r] from spec[r][n - pos - 1]. One layer. */
void NAME(lin_ref_commit)(int H, int K, int V, int C, real* temporal, real* conv, int B, int D,
                          const int64_t* slot, const int64_t* pos, const int64_t* accept_len,
                          const int64_t* track_slot, int track_interval, const real* spec_t,
                          const real* spec_c) {
  const int64_t tb = (int64_t)H * V * K, cb = (int64_t)C * 3;
  for (int r = 0; r < B; ++r) {
    const int64_t a = accept_len[r], sl = slot[r];
    if (sl < 0 || a < 1 || a > D) continue;
    const int64_t src = (int64_t)r * D + (a - 1);
    memcpy(temporal + sl * tb, spec_t + src * tb, sizeof(real) * tb);
    memcpy(conv + sl * cb, spec_c + src * cb, sizeof(real) * cb);
    const int64_t ts = track_slot ? track_slot[r] : -1;
    if (ts < 0 || track_interval <= 0) continue;
    const int64_t n = (pos[r] + a) / track_interval * track_interval;
    if (n > pos[r]) {
      const int64_t b = (int64_t)r * D + (n - pos[r] - 1);
      memcpy(temporal + ts * tb, spec_t + b * tb, sizeof(real) * tb);
      memcpy(conv + ts * cb, spec_c + b * cb, sizeof(real) * cb);
    }
  }
}

typedef struct {
  char* base;
  int64_t layer_stride, slot_stride, block;
  int layers;
  const int64_t *src, *dst;
} copy_ctx;

static void copy_unit(void* ctx, int64_t u) {
  const copy_ctx* p = (const copy_ctx*)ctx;
  const int64_t i = u / p->layers, l = u % p->layers;
  if (p->src[i] < 0 || p->dst[i] < 0 || p->src[i] == p->dst[i]) return;
  char* b = p->base + l * p->layer_stride;
  memcpy(b + p->dst[i] * p->slot_stride, b + p->src[i] * p->slot_stride, (size_t)p->block);
}

/* Slot copies over `layers` layers of one byte array laid out
 * [layer][slot][block]: block dst[i] <- block src[i]; a negative id skips the
 * pair (MambaRadixCache page 3.2, copy_from). Bytes, so it serves any dtype. */
void NAME(lin_ref_copy_slots)(char* base, int64_t layer_stride, int64_t slot_stride,
                              int64_t block_bytes, int layers, int n, const int64_t* src,
                              const int64_t* dst, int nthreads) {
  copy_ctx p = {base, layer_stride, slot_stride, block_bytes, layers, src, dst};
  run_units(copy_unit, &p, (int64_t)n * layers, nthreads);
}
