// Token-by-token kernels: decode (in place, with interval tracking), the
// speculative verify (per-step states into a buffer), and a recurrent prefill
// for head dims the chunked tensor-core kernel does not cover.
//
// The update is the KDA recurrence of the Kimi-K3 notes ("企业官网建设流程全解析",
// "Speculative decoding"):
//     S' = S Diag(alpha) + d k^T,   d = beta (v - (S Diag(alpha)) k),   o = S' q
// Row v of S (its K key channels) evolves on its own given (k, alpha, beta, v_v),
// so rows are spread over threads: a row is split over D/8 lanes of one warp,
// 8 consecutive key channels per lane, which makes every state load and store
// one coalesced 16-byte (bf16) or 32-byte (fp32) vector per lane. The two dot
// products of a row are reduced with xor shuffles inside those lanes.
//
// One CTA handles one (request, head). The width-4 causal conv of the head's
// q|k|v channels runs first; each conv channel is owned by one thread, which
// keeps its 3-input window in registers (Kimi-K3 notes, "Conv state").

#include "common.cuh"
#include "internal.h"

namespace lin {
namespace {

constexpr float kL2Eps = 1e-6f;

template <int D>
struct TokCfg {
  static constexpr int LPR = D / 8;  // lanes per state row
  static constexpr int NT = (D * LPR < 256) ? D * LPR : 256;
  static constexpr int RPT = D * LPR / NT;  // rows per thread
  static constexpr int RSTEP = NT / LPR;    // row stride between a thread's rows
  static constexpr int CH = 3 * D;          // conv channels of one head
  static constexpr int CPT = (CH + NT - 1) / NT;
  static_assert(NT % 32 == 0, "whole warps");
};

// Global conv channel of local channel cl (q | k | v of head h).
__device__ __forceinline__ int head_channel(int cl, int h, int H, int D) {
  if (cl < D) return h * D + cl;
  if (cl < 2 * D) return H * D + h * D + (cl - D);
  return 2 * H * D + h * D + (cl - 2 * D);
}

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-token shared scratch: post-conv q | k | v and the two norm factors.
template <int D>
struct TokSmem {
  float y[2][3 * D + 2];
};

// Conv + activation for one token: each thread does its own channels and
// keeps the window win[c][0..2] (oldest first) in registers.
template <int D>
__device__ __forceinline__ void conv_token(float (&win)[TokCfg<D>::CPT][3],
                                           const float (&w)[TokCfg<D>::CPT][4],
                                           const void* x, int64_t xrow, const int (&chan)[TokCfg<D>::CPT],
                                           int io_dtype, bool do_silu, float* ys) {
  using C = TokCfg<D>;
#pragma unroll
  for (int i = 0; i < C::CPT; ++i) {
    const int cl = threadIdx.x + i * C::NT;
    if (cl < C::CH) {
      const float xin = load_elem(x, xrow + chan[i], io_dtype);
      float y = w[i][0] * win[i][0] + w[i][1] * win[i][1] + w[i][2] * win[i][2] + w[i][3] * xin;
      win[i][0] = win[i][1];
      win[i][1] = win[i][2];
      win[i][2] = xin;
      if (do_silu) y = silu(y);
      ys[cl] = y;
    }
  }
}

// Sum of squares of q and k (first 2D entries of ys) -> 1/sqrt(ss + eps).
template <int D>
__device__ __forceinline__ void qk_norms(float* ys, bool l2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!l2) {
    if (threadIdx.x == 0) {
      ys[3 * D] = 1.f;
      ys[3 * D + 1] = 1.f;
    }
    return;
  }
  constexpr int NW = TokCfg<D>::NT / 32;
  if (NW >= 2) {
    if (warp < 2) {
      const float* v = ys + warp * D;
      float ss = 0.f;
      for (int i = lane; i < D; i += 32) ss += v[i] * v[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) ys[3 * D + warp] = rsqrtf(ss + kL2Eps);
    }
  } else {
    for (int part = 0; part < 2; ++part) {
      const float* v = ys + part * D;
      float ss = 0.f;
      for (int i = lane; i < D; i += 32) ss += v[i] * v[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) ys[3 * D + part] = rsqrtf(ss + kL2Eps);
    }
  }
}

// Update this thread's rows for one token; writes o for the rows it leads.
template <int D>
__device__ __forceinline__ void rows_update(float (&s)[TokCfg<D>::RPT][8], const float* ys,
                                            const float (&a8)[8], float beta, float q_scale,
                                            void* out, int64_t orow, int out_dtype) {
  using C = TokCfg<D>;
  const int lr = threadIdx.x % C::LPR;
  const int row0 = threadIdx.x / C::LPR;
  const float rq = ys[3 * D] * q_scale, rk = ys[3 * D + 1];
  float q8[8], k8[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    q8[e] = ys[lr * 8 + e] * rq;
    k8[e] = ys[D + lr * 8 + e] * rk;
  }
#pragma unroll
  for (int i = 0; i < C::RPT; ++i) {
    const int row = row0 + i * C::RSTEP;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s[i][e] *= a8[e];
      dot = fmaf(s[i][e], k8[e], dot);
    }
    dot = row_sum<C::LPR>(dot);
    const float u = beta * (ys[2 * D + row] - dot);
    float o = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s[i][e] = fmaf(u, k8[e], s[i][e]);
      o = fmaf(s[i][e], q8[e], o);
    }
    o = row_sum<C::LPR>(o);
    if (lr == 0) store_elem(out, orow + row, out_dtype, o);
  }
}

template <int D>
__device__ __forceinline__ void load_alpha(float (&a8)[8], const float* g, int64_t gbase,
                                           int gate_mode) {
  const int lr = threadIdx.x % TokCfg<D>::LPR;
  if (gate_mode == LIN_GATE_PER_KEY) {
#pragma unroll
    for (int e = 0; e < 8; ++e) a8[e] = expf(g[gbase + lr * 8 + e]);
  } else {
    const float a = expf(g[gbase]);
#pragma unroll
    for (int e = 0; e < 8; ++e) a8[e] = a;
  }
}

template <int D, int ST>
__device__ __forceinline__ void store_rows(char* base, const float (&s)[TokCfg<D>::RPT][8]) {
  using C = TokCfg<D>;
  const int lr = threadIdx.x % C::LPR, row0 = threadIdx.x / C::LPR;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
#pragma unroll
  for (int i = 0; i < C::RPT; ++i)
    Vec8<ST>::store(base + (int64_t(row0 + i * C::RSTEP) * D + lr * 8) * ES, s[i]);
}

template <int D, int ST>
__device__ __forceinline__ void load_rows(const char* base, float (&s)[TokCfg<D>::RPT][8]) {
  using C = TokCfg<D>;
  const int lr = threadIdx.x % C::LPR, row0 = threadIdx.x / C::LPR;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
#pragma unroll
  for (int i = 0; i < C::RPT; ++i)
    Vec8<ST>::load(base + (int64_t(row0 + i * C::RSTEP) * D + lr * 8) * ES, s[i]);
}

template <int CPT, int D>
__device__ __forceinline__ void store_window(void* conv_base, int conv_dtype, const int (&chan)[CPT],
                                             const float (&win)[CPT][3]) {
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int cl = threadIdx.x + i * blockDim.x;
    if (cl < 3 * D) {
#pragma unroll
      for (int j = 0; j < 3; ++j) store_elem(conv_base, int64_t(chan[i]) * 3 + j, conv_dtype, win[i][j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Decode / verify. One CTA per (request, head). Everything the head needs --
// its state block, the conv window and taps of its q|k|v channels, and the
// step's x (and per-key g) rows -- is staged into shared memory by bulk async
// copies on one mbarrier, issued before any other work, so loads in flight
// cost no registers and the CTA stays small. Each thread then updates its
// rows from shared memory (8 key channels per lane, D/8 lanes per row) and
// writes them straight to their destinations.
// ---------------------------------------------------------------------------
struct DecodeParams {
  lin_state_pool_t pool;
  lin_decode_args_t a;
};

constexpr uint32_t kDecWaitTries = 1u << 24;

template <int D>
struct DecCfg {
  static constexpr int LPR = D / 8;
  static constexpr int NT = (D * LPR) < 128 ? ((D * LPR) < 32 ? 32 : D * LPR) : 128;
  static constexpr int RSTEP = NT / LPR;
  static constexpr int RPT = D / RSTEP;
  static constexpr int CH = 3 * D;
  static constexpr int CPT = (CH + NT - 1) / NT;
  static_assert(RPT * RSTEP == D, "rows");
};

// Shared-memory layout of one decode CTA (byte offsets; every piece 16-aligned).
struct DecSmem {
  int state, conv, w, x, g, total;
  __host__ __device__ DecSmem(int D, int es_state, int es_conv, int es_io, int nd, bool per_key) {
    state = 0;
    conv = state + D * D * es_state;
    w = conv + 3 * D * 3 * es_conv;
    x = w + 3 * D * 4 * es_io;
    g = x + nd * 3 * D * es_io;
    total = g + (per_key ? nd * D * 4 : 0);
  }
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <int D, int ST>
__global__ void __launch_bounds__(DecCfg<D>::NT) decode_kernel(DecodeParams p) {
  using C = DecCfg<D>;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ float ysm[2][3 * D + 2];
  __shared__ uint64_t bar;
  __shared__ int abort_sh;
  const lin_state_pool_t& pool = p.pool;
  const lin_decode_args_t& a = p.a;
  const int r = blockIdx.x, h = blockIdx.y;
  const int H = pool.num_heads;
  const int ns = pool.num_slots;
  const int slot = a.slot[r];
  if (slot < 0) return;
  const bool rep = (h == 0 && threadIdx.x == 0);
  if (slot >= ns) {
    if (rep) report(a.status, LIN_ST_BAD_SLOT);
    return;
  }
  const int ts = a.track_slot ? a.track_slot[r] : -1;
  if (ts >= ns) {
    if (rep) report(a.status, LIN_ST_BAD_SLOT);
    return;
  }
  if (ts == slot) {
    if (rep) report(a.status, LIN_ST_TRACK_ALIAS);
    return;
  }
  const int ND = a.n_draft;
  const bool per_key = a.gate_mode == LIN_GATE_PER_KEY;
  const int esc = pool.conv_dtype == LIN_BF16 ? 2 : 4;
  const int esi = a.io_dtype == LIN_BF16 ? 2 : 4;
  const DecSmem L(D, ES, esc, esi, ND, per_key);
  const int64_t head_bytes = int64_t(D) * D * ES;
  char* slot_t = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                 slot * pool.temporal_slot_stride + h * head_bytes;
  char* slot_c = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                 slot * pool.conv_slot_stride;
  const int C_all = pool.conv_channels;
  const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(dsm));
  const uint32_t sbar = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    abort_sh = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sbar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sbar),
                 "r"(static_cast<uint32_t>(L.total))
                 : "memory");
    bulk_g2s(s0 + L.state, slot_t, D * D * ES, sbar);
    for (int part = 0; part < 3; ++part) {
      const int64_t ch0 = int64_t(part) * H * D + int64_t(h) * D;  // first channel of the part
      bulk_g2s(s0 + L.conv + part * D * 3 * esc, static_cast<const char*>(slot_c) + ch0 * 3 * esc,
               D * 3 * esc, sbar);
      bulk_g2s(s0 + L.w + part * D * 4 * esi, static_cast<const char*>(a.conv_w) + ch0 * 4 * esi,
               D * 4 * esi, sbar);
      for (int j = 0; j < ND; ++j) {
        const int64_t tok = int64_t(r) * ND + j;
        bulk_g2s(s0 + L.x + (j * 3 + part) * D * esi,
                 static_cast<const char*>(a.x) + (tok * C_all + ch0) * esi, D * esi, sbar);
      }
    }
    if (per_key)
      for (int j = 0; j < ND; ++j) {
        const int64_t tok = int64_t(r) * ND + j;
        bulk_g2s(s0 + L.g + j * D * 4, a.g + (tok * H + h) * D, D * 4, sbar);
      }
    bool ok = false;
    for (uint32_t it = 0; it < kDecWaitTries && !ok; ++it) {
      uint32_t done;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(done)
          : "r"(sbar)
          : "memory");
      ok = done != 0;
    }
    if (!ok) {
      abort_sh = 1;
      report(a.status, LIN_ST_TIMEOUT);
    }
  }
  __syncthreads();
  if (abort_sh) return;  // the copies were given up on; nothing is written

  const uint8_t* sconv = dsm + L.conv;
  const uint8_t* sw = dsm + L.w;
  // conv channels: local cl in [0, 3D), part = cl / D
  int chan[C::CPT];
  float win[C::CPT][3], w[C::CPT][4];
#pragma unroll
  for (int i = 0; i < C::CPT; ++i) {
    const int cl = threadIdx.x + i * C::NT;
    chan[i] = cl < C::CH ? head_channel(cl, h, H, D) : 0;
    if (cl < C::CH) {
#pragma unroll
      for (int q = 0; q < 3; ++q) win[i][q] = load_elem(sconv, cl * 3 + q, pool.conv_dtype);
#pragma unroll
      for (int q = 0; q < 4; ++q) w[i][q] = load_elem(sw, cl * 4 + q, a.io_dtype);
    }
  }
  const bool silu_on = a.flags & LIN_CONV_SILU;
  const int lr = threadIdx.x % C::LPR, row0 = threadIdx.x / C::LPR;
  for (int j = 0; j < ND; ++j) {
    float* ys = ysm[j & 1];
    const int64_t tok = int64_t(r) * ND + j;
    const uint8_t* sx = dsm + L.x + j * 3 * D * esi;
#pragma unroll
    for (int i = 0; i < C::CPT; ++i) {
      const int cl = threadIdx.x + i * C::NT;
      if (cl < C::CH) {
        const float xin = load_elem(sx, cl, a.io_dtype);
        float y = w[i][0] * win[i][0] + w[i][1] * win[i][1] + w[i][2] * win[i][2] + w[i][3] * xin;
        win[i][0] = win[i][1];
        win[i][1] = win[i][2];
        win[i][2] = xin;
#pragma unroll
        for (int q = 0; q < 3; ++q) win[i][q] = round_to_dtype(win[i][q], pool.conv_dtype);
        ys[cl] = silu_on ? silu(y) : y;
      }
    }
    __syncthreads();
    {
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      constexpr int NWp = C::NT / 32;
      for (int part = (NWp >= 2 ? warp : 0); part < 2; part += (NWp >= 2 ? 2 : 1)) {
        if (NWp >= 2 && warp >= 2) break;
        float ss = 0.f;
        for (int i = lane; i < D; i += 32) ss += ys[part * D + i] * ys[part * D + i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) ys[3 * D + part] = (a.flags & LIN_QK_L2NORM) ? rsqrtf(ss + kL2Eps) : 1.f;
      }
    }
    __syncthreads();
    float a8[8];
    if (per_key) {
      const float* sg = reinterpret_cast<const float*>(dsm + L.g) + j * D + lr * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) a8[e] = expf(sg[e]);
    } else {
      const float av = expf(a.g[tok * H + h]);
#pragma unroll
      for (int e = 0; e < 8; ++e) a8[e] = av;
    }
    const float beta = a.beta[tok * H + h];
    const float rq = ys[3 * D] * a.q_scale, rk = ys[3 * D + 1];
    float q8[8], k8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      q8[e] = ys[lr * 8 + e] * rq;
      k8[e] = ys[D + lr * 8 + e] * rk;
    }
    char* dt;
    char* dc;
    char* tt = nullptr;
    char* tc = nullptr;
    if (ND == 1) {
      dt = slot_t;
      dc = slot_c;
      const int n = a.pos[r] + 1;
      if (ts >= 0 && a.track_interval > 0 && n % a.track_interval == 0) {
        tt = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
             ts * pool.temporal_slot_stride + h * head_bytes;
        tc = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
             ts * pool.conv_slot_stride;
      }
    } else {
      dt = static_cast<char*>(a.spec.temporal) + a.layer * a.spec.temporal_layer_stride +
           r * a.spec.temporal_req_stride + j * a.spec.temporal_step_stride + h * head_bytes;
      dc = static_cast<char*>(a.spec.conv) + a.layer * a.spec.conv_layer_stride +
           r * a.spec.conv_req_stride + j * a.spec.conv_step_stride;
    }
    uint8_t* sst = dsm + L.state;
#pragma unroll 4
    for (int i = 0; i < C::RPT; ++i) {
      const int row = row0 + i * C::RSTEP;
      const int64_t off = (int64_t(row) * D + lr * 8) * ES;
      float sv[8];
      Vec8<ST>::load(sst + off, sv);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sv[e] *= a8[e];
        dot = fmaf(sv[e], k8[e], dot);
      }
      dot = row_sum<C::LPR>(dot);
      const float u = beta * (ys[2 * D + row] - dot);
      float o = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sv[e] = fmaf(u, k8[e], sv[e]);
        o = fmaf(sv[e], q8[e], o);
      }
      o = row_sum<C::LPR>(o);
      if (lr == 0) store_elem(a.out, (tok * H + h) * D + row, a.out_dtype, o);
      Vec8<ST>::round(sv);  // the stored state is what the next token starts from
      Vec8<ST>::store(dt + off, sv);
      if (tt) Vec8<ST>::store(tt + off, sv);
      if (ND > 1) Vec8<ST>::store(sst + off, sv);
    }
    store_window<DecCfg<D>::CPT, D>(dc, pool.conv_dtype, chan, win);
    if (tc) store_window<DecCfg<D>::CPT, D>(tc, pool.conv_dtype, chan, win);
  }
}

// ---------------------------------------------------------------------------
// Recurrent prefill. grid (batch, H), block NT. State carried in fp32 for
// the whole request; rounded only where stored.
// ---------------------------------------------------------------------------
struct PrefillParams {
  lin_state_pool_t pool;
  lin_prefill_args_t a;
};

template <int D, int ST>
__global__ void __launch_bounds__(TokCfg<D>::NT) prefill_recurrent_kernel(PrefillParams p) {
  using C = TokCfg<D>;
  __shared__ TokSmem<D> sm;
  const lin_state_pool_t& pool = p.pool;
  const lin_prefill_args_t& a = p.a;
  const int r = blockIdx.x, h = blockIdx.y;
  const int H = pool.num_heads;
  const int ns = pool.num_slots;
  const bool rep = (h == 0 && threadIdx.x == 0);
  const int slot = a.slot[r];
  if (slot < 0) return;
  if (slot >= ns) {
    if (rep) report(a.status, LIN_ST_BAD_SLOT);
    return;
  }
  const int64_t bos = a.cu_seqlens[r], eos = a.cu_seqlens[r + 1];
  if (bos < 0 || eos < bos || eos > a.total_tokens) {
    if (rep) report(a.status, LIN_ST_BAD_SEQLEN);
    return;
  }
  const int P = a.prefix_len[r];
  if (P < 0 || (P & 63)) {
    if (rep) report(a.status, LIN_ST_BAD_PREFIX);
    return;
  }
  int t0 = 0, nt = 0;
  if (a.track_stride > 0 && a.cu_track) {
    t0 = a.cu_track[r];
    nt = a.cu_track[r + 1] - t0;
    for (int i = 0; i < nt; ++i) {
      const int t = a.track_slots[t0 + i];
      if (t >= ns) {
        if (rep) report(a.status, LIN_ST_BAD_SLOT);
        return;
      }
      if (t == slot) {
        if (rep) report(a.status, LIN_ST_TRACK_ALIAS);
        return;
      }
    }
  }
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
  const int64_t head_bytes = int64_t(D) * D * ES;
  char* slot_t = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                 slot * pool.temporal_slot_stride + h * head_bytes;
  char* slot_c = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                 slot * pool.conv_slot_stride;
  const bool warm = a.has_initial_state[r] != 0;

  float s[C::RPT][8];
  if (warm) {
    load_rows<D, ST>(slot_t, s);
  } else {
#pragma unroll
    for (int i = 0; i < C::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) s[i][e] = 0.f;
  }
  const int C_all = pool.conv_channels;
  int chan[C::CPT];
  float win[C::CPT][3], w[C::CPT][4];
#pragma unroll
  for (int i = 0; i < C::CPT; ++i) {
    const int cl = threadIdx.x + i * C::NT;
    chan[i] = cl < C::CH ? head_channel(cl, h, H, D) : 0;
#pragma unroll
    for (int j = 0; j < 3; ++j)
      win[i][j] = (warm && cl < C::CH) ? load_elem(slot_c, int64_t(chan[i]) * 3 + j, pool.conv_dtype) : 0.f;
    if (cl < C::CH) {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[i][j] = load_elem(a.conv_w, int64_t(chan[i]) * 4 + j, a.io_dtype);
    }
  }

  int snap = 0;
  for (int64_t t = bos; t < eos; ++t) {
    float* ys = sm.y[(t - bos) & 1];
    conv_token<D>(win, w, a.x, t * C_all, chan, a.io_dtype, a.flags & LIN_CONV_SILU, ys);
    __syncthreads();
    qk_norms<D>(ys, a.flags & LIN_QK_L2NORM);
    __syncthreads();
    float a8[8];
    const int64_t gbase = a.gate_mode == LIN_GATE_PER_KEY ? (t * H + h) * D : t * H + h;
    load_alpha<D>(a8, a.g, gbase, a.gate_mode);
    rows_update<D>(s, ys, a8, a.beta[t * H + h], a.q_scale, a.out, (t * H + h) * D, a.out_dtype);
    const int64_t n = P + (t - bos) + 1;
    if (nt > 0 && n % a.track_stride == 0) {
      const int dst = a.track_slots[t0 + (snap % nt)];
      ++snap;
      if (dst >= 0) {
        char* tt = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                   dst * pool.temporal_slot_stride + h * head_bytes;
        char* tc = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                   dst * pool.conv_slot_stride;
        store_rows<D, ST>(tt, s);
        store_window<TokCfg<D>::CPT, D>(tc, pool.conv_dtype, chan, win);
      }
    }
  }
  store_rows<D, ST>(slot_t, s);
  store_window<TokCfg<D>::CPT, D>(slot_c, pool.conv_dtype, chan, win);
}

template <int D, int ST>
cudaError_t decode_launch(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                          cudaStream_t stream) {
  DecodeParams p{pool, a};
  const DecSmem L(D, ST == LIN_BF16 ? 2 : 4, dtype_size(pool.conv_dtype), dtype_size(a.io_dtype),
                  a.n_draft, a.gate_mode == LIN_GATE_PER_KEY);
  if (L.total > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, ST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return e;
  decode_kernel<D, ST><<<dim3(a.batch, pool.num_heads), DecCfg<D>::NT, L.total, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int ST>
cudaError_t prefill_launch(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                           cudaStream_t stream) {
  PrefillParams p{pool, a};
  prefill_recurrent_kernel<D, ST><<<dim3(a.batch, pool.num_heads), TokCfg<D>::NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

#define LIN_DISPATCH_D_ST(FN, D, ST, ...)                                   \
  do {                                                                      \
    const bool bf = (ST) == LIN_BF16;                                       \
    switch (D) {                                                            \
      case 16: return bf ? FN<16, LIN_BF16>(__VA_ARGS__) : FN<16, LIN_F32>(__VA_ARGS__);    \
      case 32: return bf ? FN<32, LIN_BF16>(__VA_ARGS__) : FN<32, LIN_F32>(__VA_ARGS__);    \
      case 64: return bf ? FN<64, LIN_BF16>(__VA_ARGS__) : FN<64, LIN_F32>(__VA_ARGS__);    \
      case 128: return bf ? FN<128, LIN_BF16>(__VA_ARGS__) : FN<128, LIN_F32>(__VA_ARGS__); \
      default: return cudaErrorInvalidValue;                                \
    }                                                                       \
  } while (0)

cudaError_t launch_decode(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                          cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  LIN_DISPATCH_D_ST(decode_launch, pool.head_k, pool.state_dtype, pool, a, stream);
}

cudaError_t launch_prefill_recurrent(const lin_state_pool_t& pool,
                                     const lin_prefill_args_t& a, cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  LIN_DISPATCH_D_ST(prefill_launch, pool.head_k, pool.state_dtype, pool, a, stream);
}

}  // namespace lin
