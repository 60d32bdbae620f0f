// Token-by-token kernels: decode (in place, with interval tracking), the
// speculative verify (per-step states into a buffer), and a recurrent prefill
// for head dims the chunked tensor-core kernel does not cover.
//
// The update is the KDA recurrence of the Kimi-K3 notes ("企业官网建设流程全解析",
// "Speculative decoding"):
//     S' = S Diag(alpha) + d k^T,   d = beta (v - (S Diag(alpha)) k),   o = S' q
// or, with LIN_UPDATE_ADDITIVE, the Mamba2 SSD form d = beta v of the
// MambaRadixCache page (section 9.3).
// Row v of S (its K key channels) evolves on its own given (k, alpha, beta, v_v),
// so rows are spread over threads: a row is split over D/8 lanes of one warp,
// 8 consecutive key channels per lane, which makes every state load and store
// one coalesced 16-byte (bf16) or 32-byte (fp32) vector per lane. The two dot
// products of a row are reduced with xor shuffles inside those lanes.
//
// One CTA handles one (request, head). The width-4 causal conv of the head's
// q|k|v channels runs first; each conv channel is owned by one thread, which
// keeps its 3-input window in registers (Kimi-K3 notes, "Conv state").

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace lin {
namespace {

constexpr float kL2Eps = 1e-6f;

// D: key channels per head (state row length), V: value channels (state rows).
template <int D, int V = D>
struct TokCfg {
  static constexpr int LPR = D / 8;  // lanes per state row
  static constexpr int NT = (V * LPR < 256) ? V * LPR : 256;
  static constexpr int RPT = V * LPR / NT;  // rows per thread
  static constexpr int RSTEP = NT / LPR;    // row stride between a thread's rows
  static constexpr int CH = 2 * D + V;      // conv channels of one head: q | k | v
  static constexpr int CPT = (CH + NT - 1) / NT;
  static_assert(NT % 32 == 0, "whole warps");
  static_assert(RPT * RSTEP == V, "rows");
};

// Global conv channel of local channel cl (q | k | v of head h; q and k have D
// channels per head, v has V).
__device__ __forceinline__ int head_channel(int cl, int h, int H, int D, int V) {
  if (cl < D) return h * D + cl;
  if (cl < 2 * D) return H * D + h * D + (cl - D);
  return 2 * H * D + h * V + (cl - 2 * D);
}

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-token shared scratch: post-conv q | k | v and the two norm factors.
template <int D, int V>
struct TokSmem {
  float y[2][2 * D + V];
  float part[2][(TokCfg<D, V>::NT + 31) / 32][2];  // per warp: sum of q^2, sum of k^2
};

// Conv + activation for one token: each thread does its own channels and
// keeps the window win[c][0..2] (oldest first) in registers; the token's
// inputs are already in registers too. Each warp also leaves its partial sums
// of q^2 and k^2 in part[warp] for the L2 norms.
template <int D, int V>
__device__ __forceinline__ void conv_token_in(float (&win)[TokCfg<D, V>::CPT][3],
                                              const float (&w)[TokCfg<D, V>::CPT][4],
                                              const float (&xin)[TokCfg<D, V>::CPT], bool do_silu, float* ys,
                                              float (*part)[2]) {
  using C = TokCfg<D, V>;
  float pq = 0.f, pk = 0.f;
#pragma unroll
  for (int i = 0; i < C::CPT; ++i) {
    const int cl = threadIdx.x + i * C::NT;
    if (cl < C::CH) {
      float y = w[i][0] * win[i][0] + w[i][1] * win[i][1] + w[i][2] * win[i][2] + w[i][3] * xin[i];
      win[i][0] = win[i][1];
      win[i][1] = win[i][2];
      win[i][2] = xin[i];
      if (do_silu) y = silu(y);
      ys[cl] = y;
      if (cl < D)
        pq = fmaf(y, y, pq);
      else if (cl < 2 * D)
        pk = fmaf(y, y, pk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pq += __shfl_xor_sync(0xffffffffu, pq, o);
    pk += __shfl_xor_sync(0xffffffffu, pk, o);
  }
  if ((threadIdx.x & 31) == 0) {
    part[threadIdx.x >> 5][0] = pq;
    part[threadIdx.x >> 5][1] = pk;
  }
}

// Update this thread's rows for one token and write their outputs. Both row
// dot products are taken on the decayed state, d_k = (S A) k and d_q = (S A) q,
// so o = S' q = d_q + u (k . q) needs no second pass over the updated row. The
// 2 x RPT sums of the thread's rows are reduced across the row's LPR lanes by
// one transposing butterfly: at each level a lane keeps half of its values and
// sends the other half, so sum m ends whole in lane m / (LPR / (2 RPT)).
template <int D, int V>
__device__ __forceinline__ void rows_update(float (&s)[TokCfg<D, V>::RPT][8], const float* ys,
                                            const float (&a8)[8], float beta, float dmul, float rq, float rk,
                                            void* out, int64_t orow, int out_dtype) {
  using C = TokCfg<D, V>;
  constexpr int NV = 2 * C::RPT;      // sums per thread: d_k, d_q of each row
  constexpr int VSTEP = C::LPR / NV;  // lanes per reduced sum
  static_assert(NV <= C::LPR && VSTEP * NV == C::LPR, "one reduced sum per lane group");
  const int lr = threadIdx.x % C::LPR;
  const int gbase = (threadIdx.x & 31) - lr;  // first lane of the row group
  const int row0 = threadIdx.x / C::LPR;
  float q8[8], k8[8];
  float kqp = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    q8[e] = ys[lr * 8 + e] * rq;
    k8[e] = ys[D + lr * 8 + e] * rk;
    kqp = fmaf(k8[e], q8[e], kqp);
  }
  const float kq = row_sum<C::LPR>(kqp);
  float red[NV];
#pragma unroll
  for (int i = 0; i < C::RPT; ++i) {
    float dk = 0.f, dq = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s[i][e] *= a8[e];
      dk = fmaf(s[i][e], k8[e], dk);
      dq = fmaf(s[i][e], q8[e], dq);
    }
    red[2 * i] = dk;
    red[2 * i + 1] = dq;
  }
#pragma unroll
  for (int d = C::LPR / 2, nv = NV; d > 0; d >>= 1) {
    if (nv > 1) {
      const bool up = lr & d;
      nv >>= 1;
#pragma unroll
      for (int v = 0; v < NV / 2; ++v) {
        if (v < nv) {
          const float keep = up ? red[v + nv] : red[v];
          const float send = up ? red[v] : red[v + nv];
          red[v] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
      }
    } else {
      red[0] += __shfl_xor_sync(0xffffffffu, red[0], d);
    }
  }
#pragma unroll
  for (int i = 0; i < C::RPT; ++i) {
    const int row = row0 + i * C::RSTEP;
    const float dk = __shfl_sync(0xffffffffu, red[0], gbase + 2 * i * VSTEP);
    const float u = beta * fmaf(-dmul, dk, ys[2 * D + row]);  // dmul 0: additive form
#pragma unroll
    for (int e = 0; e < 8; ++e) s[i][e] = fmaf(u, k8[e], s[i][e]);
    // the lane holding this row's d_q writes its output
    if (lr == (2 * i + 1) * VSTEP) store_elem(out, orow + row, out_dtype, fmaf(u, kq, red[0]));
  }
}

template <int D, int V, int ST>
__device__ __forceinline__ void store_rows(char* base, const float (&s)[TokCfg<D, V>::RPT][8]) {
  using C = TokCfg<D, V>;
  const int lr = threadIdx.x % C::LPR, row0 = threadIdx.x / C::LPR;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
#pragma unroll
  for (int i = 0; i < C::RPT; ++i)
    Vec8<ST>::store(base + (int64_t(row0 + i * C::RSTEP) * D + lr * 8) * ES, s[i]);
}

template <int D, int V, int ST>
__device__ __forceinline__ void load_rows(const char* base, float (&s)[TokCfg<D, V>::RPT][8]) {
  using C = TokCfg<D, V>;
  const int lr = threadIdx.x % C::LPR, row0 = threadIdx.x / C::LPR;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
#pragma unroll
  for (int i = 0; i < C::RPT; ++i)
    Vec8<ST>::load(base + (int64_t(row0 + i * C::RSTEP) * D + lr * 8) * ES, s[i]);
}

// CH: conv channels of the head; NS: threads that share them (0: the whole block).
template <int CPT, int CH, int NS = 0>
__device__ __forceinline__ void store_window(void* conv_base, int conv_dtype, const int (&chan)[CPT],
                                             const float (&win)[CPT][3]) {
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int cl = threadIdx.x + i * (NS ? NS : static_cast<int>(blockDim.x));
    if (cl < CH) {
#pragma unroll
      for (int j = 0; j < 3; ++j) store_elem(conv_base, int64_t(chan[i]) * 3 + j, conv_dtype, win[i][j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Decode / verify. The unit of work is one (request, head) item. Everything
// an item needs -- its state block, the conv window and taps of its q|k|v
// channels, and the step's x (and per-key g) rows -- is staged into shared
// memory by bulk async copies completing on one mbarrier, so loads in flight
// cost no registers. Each thread then updates its rows from shared memory
// (8 key channels per lane, D/8 lanes per row) and writes them straight to
// their destinations.
// ---------------------------------------------------------------------------
struct DecodeParams {
  lin_state_pool_t pool;
  lin_decode_args_t a;
  const int32_t* accept;  // replay commit: accepted tokens per request (NULL: decode / verify)
  // replay commit: byte offsets in dynamic shared memory of the request order
  // (int16 [batch]) and its histogram (int [n_draft + 1]); order_off 0: the
  // batch's own order
  int order_off, hist_off;
};

constexpr uint32_t kDecWaitTries = 1u << 24;

// Shared-memory layout of one decode stage (byte offsets; every piece
// 16-aligned); the producer's bulk loads fill all of it.
// Stage layout of one (request, head) item. Bytes [0, load) arrive by bulk
// copies; bg holds (beta, scalar g) per draft, fetched by the producer warp.
struct DecSmem {
  int state, conv, w, x, g, load, bg, size;
  // D key channels, V value channels per head (q | k | v: 2D + V conv channels)
  __host__ __device__ DecSmem(int D, int V, int es_state, int es_conv, int es_io, int nd, bool per_key) {
    const int CH = 2 * D + V;
    state = 0;
    conv = state + V * D * es_state;
    w = conv + CH * 3 * es_conv;
    x = w + CH * 4 * es_io;
    g = x + nd * CH * es_io;
    load = g + (per_key ? nd * D * 4 : 0);
    bg = load;
    size = bg + nd * 2 * 4;
  }
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Warp-specialised persistent form. Each CTA walks the (request, head) items
// i = blockIdx.x, blockIdx.x + gridDim.x, ... through a ring of `stages`
// shared-memory buffers (two CTAs share an SM). One producer warp looks up each
// item's slot, writes the item's metadata and issues the stage's bulk loads,
// up to `stages` items ahead. The NC consumer threads (8 warps at head 128)
// wait for a stage warp by warp, so a warp that is done with one item starts
// the conv of the next while others still update rows; the only CTA-wide
// barrier is the one that publishes the conv outputs (per token in one-token
// decode, per group of drafts in the draft modes). Each warp hands the stage
// back as soon as its own reads of it are done.
//
// Row arithmetic: with A = Diag(alpha), the output needs no second pass over
// the updated row, since  o_r = sum_c S'[r,c] q_c = (S A q)_r + u_r (k . q):
// the two reductions (S A k)_r and (S A q)_r of up to four of a thread's rows
// are summed across the row's lanes together by a transposing butterfly (each
// exchange halves the values a lane still carries), then each row's u_r is
// taken from the lane that ends up holding (S A k)_r.
// D: key channels (row length), V: value channels (rows) per head.
template <int D, int V = D>
struct DecPCfg {
  static constexpr int LPR = D / 8;  // lanes per row, 8 key channels each
  static constexpr int NC = (D * LPR) < 256 ? ((D * LPR) < 32 ? 32 : D * LPR) : 256;
  static constexpr int NCW = NC / 32;   // consumer warps
  static constexpr int NT = NC + 32;    // + one producer warp
  static constexpr int RSTEP = NC / LPR;
  static constexpr int RPT = V / RSTEP;        // rows per consumer thread
  static constexpr int RB = RPT < 4 ? RPT : 4;  // rows reduced together
  static constexpr int NV = 2 * RB;             // values reduced per lane group
  static constexpr int CH = 2 * D + V;          // conv channels of one head
  static_assert(V <= D && RPT * RSTEP == V && RPT % RB == 0, "rows");
  static_assert(NV <= LPR, "one reduced value per lane");
  static_assert(2 * D <= NC, "conv and gate threads");
};

constexpr int kDecMaxStages = 4;

struct DecMeta {
  int r, h, slot, ts, pos, acc, valid;  // acc: tokens to run (n_draft, or accepted in a replay)
};

__device__ __forceinline__ bool mbar_try(uint32_t sb, uint32_t par) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(sb), "r"(par)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t sb, uint32_t par) {
  for (uint32_t it = 0; it < kDecWaitTries; ++it)
    if (mbar_try(sb, par)) return true;
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t sb) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sb) : "memory");
}
// Named barrier over the consumer threads that also ORs a predicate across them.
__device__ __forceinline__ bool consumers_sync_or(int nthreads, bool pred) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"(pred ? 1u : 0u), "r"(nthreads)
      : "memory");
  return res != 0;
}

// MODE: kDecStates (one token in place), kDecVerify (a chain of drafts into
// the spec buffer), kDecReplay (the commit form: accepted tokens per request,
// in place, no outputs), kDecTree (verify into the spec buffer where draft j
// starts from the state after draft parent[r][j], -1: the slot's). A chain
// verify without per-step states runs as one chunk (verify_chunk.cu).
// All but the one-token mode run the drafts in groups (see the consumer loop).
enum DecMode { kDecStates = 0, kDecReplay = 2, kDecTree = 3, kDecVerify = 4 };
constexpr int kDecMaxTree = 32;  // drafts per request in a tree verify
constexpr int kDecGroup = 4;     // drafts per group in the draft modes
// Dynamic shared memory of one decode CTA: at most the opt-in limit (227 KB)
// less 1 KB for the static part; at most kDecPairSmem where two CTAs share an
// SM (228 KB per SM, 1 KB of it reserved per CTA).
constexpr int kDecMaxDynSmem = 227 * 1024 - 1024;
constexpr int kDecPairSmem = 112 * 1024;
// Floats of one group buffer: post-conv q | k | v, per-key decay factors and
// the norm partials of each conv warp, for `group` drafts.
__host__ __device__ constexpr int dec_group_floats(int D, int V, int group) {
  return (group * (2 * D + V + D + (D < 32 ? 1 : D / 32) * 3) + 3) & ~3;
}

template <int D, int V, int ST, int MODE>
__global__ void __launch_bounds__(DecPCfg<D, V>::NT, 2)
    decode_kernel(DecodeParams p, int n_items, int stage_bytes, int stages, int group) {
  using C = DecPCfg<D, V>;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
  constexpr bool BATCH = MODE != kDecStates;  // the draft modes: chains and trees
  extern __shared__ __align__(128) uint8_t dsm[];
  // per-token scratch of the one-token mode (the draft modes keep theirs in
  // the group buffers after the stages)
  __shared__ __align__(16) float ysm[BATCH ? 1 : 2][BATCH ? 4 : C::CH];  // post-conv q | k | v, by token parity
  __shared__ __align__(16) float agsm[BATCH ? 1 : 2][BATCH ? 4 : D];     // per-key decay factors
  __shared__ float normsm[BATCH ? 1 : 2][D < 32 ? 1 : D / 32][3];        // q.q, k.k, q.k partials per conv warp
  __shared__ uint64_t full[kDecMaxStages], empty[kDecMaxStages];
  __shared__ DecMeta meta[kDecMaxStages];
  __shared__ int8_t par_sm[MODE == kDecTree ? kDecMaxStages : 1][MODE == kDecTree ? kDecMaxTree : 1];
  __shared__ int8_t ord_sm[MODE == kDecTree ? kDecMaxStages : 1][MODE == kDecTree ? kDecMaxTree : 1];
  const lin_state_pool_t& pool = p.pool;
  const lin_decode_args_t& a = p.a;
  const int H = pool.num_heads;
  const int ND = a.n_draft;
  const bool per_key = a.gate_mode == LIN_GATE_PER_KEY;
  const int esc = pool.conv_dtype == LIN_BF16 ? 2 : 4;
  const int esi = a.io_dtype == LIN_BF16 ? 2 : 4;
  const DecSmem L(D, V, ES, esc, esi, ND, per_key);
  const int64_t head_bytes = int64_t(V) * D * ES;
  // global conv channel of local channel t of part pt (q, k: D per head; v: V)
  auto gchan = [&](int pt, int hh, int tt) -> int64_t {
    return pt < 2 ? int64_t(pt) * H * D + int64_t(hh) * D + tt : 2LL * H * D + int64_t(hh) * V + tt;
  };
  const int C_all = pool.conv_channels;
  const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(dsm));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return static_cast<uint32_t>(__cvta_generic_to_shared(&full[s])); };
  auto empty_bar = [&](int s) { return static_cast<uint32_t>(__cvta_generic_to_shared(&empty[s])); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      meta[s].valid = 0;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full_bar(s)) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty_bar(s)), "r"(C::NCW) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ---------------- producer warp ----------------
    int issued_n[kDecMaxStages];
#pragma unroll
    for (int s = 0; s < kDecMaxStages; ++s) issued_n[s] = -1;
    int n = 0;
    bool abort = false;
    // replay commit: the requests ordered by accepted tokens, most first (ties
    // in request order; a count outside [0, n_draft] counts as 0). Items are
    // dealt to the CTAs round-robin, so every CTA then gets about the same
    // number of token passes rather than a random sum of accept lengths.
    const int16_t* order = nullptr;
    if (MODE == kDecReplay && p.order_off > 0) {
      int16_t* ord = reinterpret_cast<int16_t*>(dsm + p.order_off);
      int* hist = reinterpret_cast<int*>(dsm + p.hist_off);
      const int nb = a.batch;
      auto acc_of = [&](int rr) {
        const int v = p.accept[rr];
        return (v < 0 || v > ND) ? 0 : v;
      };
      for (int v = lane; v <= ND; v += 32) hist[v] = 0;
      __syncwarp();
      for (int rr = lane; rr < nb; rr += 32) atomicAdd(&hist[acc_of(rr)], 1);
      __syncwarp();
      if (lane == 0) {
        int run = 0;  // requests with more accepted tokens than v come first
        for (int v = ND; v >= 0; --v) {
          const int c = hist[v];
          hist[v] = run;
          run += c;
        }
      }
      __syncwarp();
      for (int r0 = 0; r0 < nb; r0 += 32) {
        const int rr = r0 + lane;
        const int v = rr < nb ? acc_of(rr) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, v);
        const int before = __popc(peers & ((1u << lane) - 1u));
        if (rr < nb) ord[hist[v] + before] = static_cast<int16_t>(rr);
        __syncwarp();
        if (rr < nb && before == 0) hist[v] += __popc(peers);
        __syncwarp();
      }
      order = ord;
    }
    for (int base = blockIdx.x; base < n_items && !abort; base += 32 * gridDim.x) {
      // lane l looks up item base + l * gridDim.x, so 32 lookups overlap
      const int item = base + lane * gridDim.x;
      DecMeta m{0, 0, -1, -1, 0, 0, 0};
      if (item < n_items) {
        m.r = order ? order[item / H] : item / H;
        m.h = item % H;
        m.slot = a.slot[m.r];
        m.ts = a.track_slot ? a.track_slot[m.r] : -1;
        m.pos = (ND == 1 || MODE == kDecReplay) ? a.pos[m.r] : 0;
        m.acc = MODE == kDecReplay ? p.accept[m.r] : ND;
        if (m.slot >= 0) {
          if (m.slot >= pool.num_slots || m.ts >= pool.num_slots) {
            if (m.h == 0) report(a.status, LIN_ST_BAD_SLOT);
          } else if (m.ts == m.slot) {
            if (m.h == 0) report(a.status, LIN_ST_TRACK_ALIAS);
          } else if (m.acc < 0 || m.acc > ND) {
            if (m.h == 0) report(a.status, LIN_ST_BAD_ACCEPT);
          } else {
            m.valid = m.acc > 0;  // nothing accepted: nothing to load or run
            if (MODE == kDecTree) {
              for (int t = 0; t < ND; ++t) {
                const int pt = a.parent[int64_t(m.r) * ND + t];
                if (pt < -1 || pt >= t) m.valid = 0;
              }
              if (!m.valid && m.h == 0) report(a.status, LIN_ST_BAD_TREE);
            }
          }
        }
      }
      const int left = (n_items - base + gridDim.x - 1) / gridDim.x;
      const int cnt = left < 32 ? left : 32;
      for (int j = 0; j < cnt; ++j, ++n) {
        DecMeta mj;
        mj.r = __shfl_sync(0xffffffffu, m.r, j);
        mj.h = __shfl_sync(0xffffffffu, m.h, j);
        mj.slot = __shfl_sync(0xffffffffu, m.slot, j);
        mj.ts = __shfl_sync(0xffffffffu, m.ts, j);
        mj.pos = __shfl_sync(0xffffffffu, m.pos, j);
        mj.acc = __shfl_sync(0xffffffffu, m.acc, j);
        mj.valid = __shfl_sync(0xffffffffu, m.valid, j);
        const int s = n % stages;
        if (lane == 0) {
          if (n >= stages && !mbar_wait_bounded(empty_bar(s), ((n / stages) - 1) & 1)) {
            report(a.status, LIN_ST_TIMEOUT);
            abort = true;
          } else {
            meta[s] = mj;
            if (MODE == kDecTree && mj.valid)
              for (int t = 0; t < ND; ++t) par_sm[s][t] = static_cast<int8_t>(a.parent[int64_t(mj.r) * ND + t]);
            if (MODE == kDecTree && mj.valid) {
              // the order the nodes run in: depth-first preorder, each node
              // followed by its lowest-index unvisited child, so that as many
              // nodes as possible start from the state of the node run just
              // before them (parents always run before their children)
              uint32_t seen = 0u;
              int cnt = 0, cur = -1;
              for (int it = 0; it < 4 * kDecMaxTree * kDecMaxTree && cnt < ND; ++it) {
                int c = -1;
                for (int k = 0; k < ND; ++k)
                  if (!((seen >> k) & 1u) && par_sm[s][k] == cur) {
                    c = k;
                    break;
                  }
                if (c >= 0) {
                  ord_sm[s][cnt++] = static_cast<int8_t>(c);
                  seen |= 1u << c;
                  cur = c;
                } else {
                  cur = cur >= 0 ? par_sm[s][cur] : -1;  // back to the parent
                }
              }
              if (cnt < ND)  // not reached for a valid tree; index order is also valid
                for (int t = 0; t < ND; ++t) ord_sm[s][t] = static_cast<int8_t>(t);
            }
            if (mj.valid) {
              const uint32_t sf = full_bar(s);
              const uint32_t s0 = s_base + s * stage_bytes;
              const char* st = static_cast<const char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                               mj.slot * pool.temporal_slot_stride + mj.h * head_bytes;
              const char* sc = static_cast<const char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                               mj.slot * pool.conv_slot_stride;
              // the producer's own arrival comes after the (beta, g) stores below
              asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(sf),
                           "r"(static_cast<uint32_t>(L.load))
                           : "memory");
              bulk_g2s(s0 + L.state, st, V * D * ES, sf);
              for (int part = 0; part < 3; ++part) {
                const int64_t ch0 = gchan(part, mj.h, 0);
                const int nch = part < 2 ? D : V;
                bulk_g2s(s0 + L.conv + part * D * 3 * esc, sc + ch0 * 3 * esc, nch * 3 * esc, sf);
                bulk_g2s(s0 + L.w + part * D * 4 * esi, static_cast<const char*>(a.conv_w) + ch0 * 4 * esi,
                         nch * 4 * esi, sf);
                for (int t = 0; t < ND; ++t) {
                  const int64_t tok = int64_t(mj.r) * ND + t;
                  bulk_g2s(s0 + L.x + (t * C::CH + part * D) * esi,
                           static_cast<const char*>(a.x) + (tok * C_all + ch0) * esi, nch * esi, sf);
                }
              }
              if (per_key)
                for (int t = 0; t < ND; ++t) {
                  const int64_t tok = int64_t(mj.r) * ND + t;
                  bulk_g2s(s0 + L.g + t * D * 4, a.g + (tok * H + mj.h) * D, D * 4, sf);
                }
            }
          }
        }
        // (beta, scalar g) of the item's drafts into the stage, one draft per
        // lane, while the bulk copies land; then the producer's arrival
        // publishes them with the stage
        const bool stage_ok = __shfl_sync(0xffffffffu, abort ? 0 : 1, 0) != 0;
        if (stage_ok && mj.valid) {
          float* bgs = reinterpret_cast<float*>(dsm + s * stage_bytes + L.bg);
          for (int t = lane; t < ND; t += 32) {
            const int64_t tok = int64_t(mj.r) * ND + t;
            bgs[2 * t] = a.beta[tok * H + mj.h];
            bgs[2 * t + 1] = per_key ? 0.f : a.g[tok * H + mj.h];
          }
        }
        __syncwarp();
        if (lane == 0 && stage_ok) {
          mbar_arrive(full_bar(s));
          issued_n[s] = n;
        }
        abort = __shfl_sync(0xffffffffu, abort, 0);
        if (abort) break;
      }
    }
    // no bulk copy may still be landing in shared memory when the CTA exits
    if (lane == 0)
      for (int s = 0; s < stages; ++s)
        if (issued_n[s] >= 0) mbar_wait_bounded(full_bar(s), (issued_n[s] / stages) & 1);
    return;
  }

  // ---------------- consumer warps ----------------
  // Thread t < D runs the conv of key channel t of q, k and v (local channels
  // t, D + t, 2D + t); threads D..2D-1 turn the per-key gates into decay
  // factors meanwhile.
  const bool silu_on = a.flags & LIN_CONV_SILU;
  const bool l2 = a.flags & LIN_QK_L2NORM;
  const float dmul = (a.flags & LIN_UPDATE_ADDITIVE) ? 0.f : 1.f;  // 0: additive form
  constexpr bool REPLAY = MODE == kDecReplay;
  const int t = threadIdx.x;
  const int lr = lane % C::LPR;           // lane within the row group
  const int gbase = lane - lr;            // first lane of the row group
  const int row0 = t / C::LPR;            // first row of this thread
  constexpr int VSTEP = C::LPR / C::NV;   // lanes per reduced value
  constexpr int NPW = D < 32 ? 1 : D / 32;  // warps holding conv channels
  const int my_v = lr / VSTEP;            // value this lane ends up holding
  int tc = 0;                             // tokens done (parity of the scratch)
  int gc = 0;                             // draft groups done (parity of the group buffer)
  const int gfloats = dec_group_floats(D, V, group);
  float* const gbuf = reinterpret_cast<float*>(dsm + stages * stage_bytes);
  int n = 0;
  bool abort = false;
  for (int item = blockIdx.x; item < n_items && !abort; item += gridDim.x, ++n) {
    const int s = n % stages;
    // each warp waits for the stage itself
    bool got = true;
    if (lane == 0) got = mbar_wait_bounded(full_bar(s), (n / stages) & 1);
    got = __shfl_sync(0xffffffffu, got, 0);
    DecMeta m = meta[s];
    if (!got) m.valid = 0;
    uint8_t* buf = dsm + s * stage_bytes;
    char* slot_t = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                   int64_t(m.slot) * pool.temporal_slot_stride + m.h * head_bytes;
    char* slot_c = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                   int64_t(m.slot) * pool.conv_slot_stride;
    if constexpr (BATCH) {
      // Drafts in groups of `group`: the conv, gate factors and norm partials
      // of every draft of the group first (none of them depends on the state:
      // a chain carries each window to the next draft, a tree node builds its
      // window from its ancestors' inputs), one barrier, then the group's row
      // updates back to back. Group buffers alternate, so a warp starts the next group's conv
      // while others still read the previous group. Every item runs the same
      // number of groups (with no work when it is empty), so all consumers
      // meet the same barriers whatever they saw. The arithmetic is the
      // one-token path's, draft by draft.
      for (int j0 = 0; j0 < ND; j0 += group, ++gc) {
        const int gn = ND - j0 < group ? ND - j0 : group;
        int nl = m.valid ? gn : 0;  // drafts of this group that run
        if (REPLAY && nl > m.acc - j0) nl = m.acc - j0 > 0 ? m.acc - j0 : 0;
        float* gys = gbuf + (gc & 1) * gfloats;  // [group][CH] post-conv q | k | v
        float* gag = gys + group * C::CH;        // [group][D] per-key decay factors
        float* gnr = gag + group * D;            // [group][NPW][3] q.q, k.k, q.k partials
        if (t < D && nl > 0) {
          float win[3][3], w[3][4];
#pragma unroll
          for (int pt = 0; pt < 3; ++pt) {
            if (V < D && pt == 2 && t >= V) break;  // v has V channels
            const int cl = pt * D + t;
#pragma unroll
            for (int q = 0; q < 3; ++q) win[pt][q] = load_elem(buf + L.conv, cl * 3 + q, pool.conv_dtype);
#pragma unroll
            for (int q = 0; q < 4; ++q) w[pt][q] = load_elem(buf + L.w, cl * 4 + q, a.io_dtype);
          }
          for (int jj = 0; jj < nl; ++jj) {
            const int j = j0 + jj;
            const int nd = MODE == kDecTree ? ord_sm[s][j] : j;  // the draft run at position j
            const uint8_t* sx = buf + L.x + nd * C::CH * esi;
            // tree: ancestors of node nd (parent first; -1 past a root)
            int a1 = -1, a2 = -1, a3 = -1;
            if (MODE == kDecTree) {
              a1 = par_sm[s][nd];
              a2 = a1 >= 0 ? par_sm[s][a1] : -1;
              a3 = a2 >= 0 ? par_sm[s][a2] : -1;
            }
            // where the window after draft j goes (besides the next draft)
            char* dc = nullptr;
            char* tcv = nullptr;
            if (MODE == kDecVerify || MODE == kDecTree) {
              dc = static_cast<char*>(a.spec.conv) + a.layer * a.spec.conv_layer_stride +
                   m.r * a.spec.conv_req_stride + nd * a.spec.conv_step_stride;
            } else if (REPLAY) {
              if (j == m.acc - 1) dc = slot_c;
              if (m.ts >= 0 && a.track_interval > 0 && (m.pos + j + 1) % a.track_interval == 0)
                tcv = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                      int64_t(m.ts) * pool.conv_slot_stride;
            }
#pragma unroll
            for (int pt = 0; pt < 3; ++pt) {
              if (V < D && pt == 2 && t >= V) break;
              const int cl = pt * D + t;
              if (MODE == kDecTree) {
                // the window before node j: the inputs of its last three
                // ancestors, topped up from the slot's window (oldest first)
                auto xr = [&](int n) {
                  return round_to_dtype(load_elem(buf + L.x + n * C::CH * esi, cl, a.io_dtype), pool.conv_dtype);
                };
                const float s0 = load_elem(buf + L.conv, cl * 3, pool.conv_dtype);
                const float s1 = load_elem(buf + L.conv, cl * 3 + 1, pool.conv_dtype);
                const float s2 = load_elem(buf + L.conv, cl * 3 + 2, pool.conv_dtype);
                win[pt][2] = a1 >= 0 ? xr(a1) : s2;
                win[pt][1] = a2 >= 0 ? xr(a2) : (a1 >= 0 ? s2 : s1);
                win[pt][0] = a3 >= 0 ? xr(a3) : (a2 >= 0 ? s2 : (a1 >= 0 ? s1 : s0));
              }
              const float xin = load_elem(sx, cl, a.io_dtype);
              // the replay commit writes no outputs: no q (its window still moves)
              const float y = (REPLAY && pt == 0)
                                  ? 0.f
                                  : w[pt][0] * win[pt][0] + w[pt][1] * win[pt][1] + w[pt][2] * win[pt][2] +
                                        w[pt][3] * xin;
              win[pt][0] = win[pt][1];
              win[pt][1] = win[pt][2];
              win[pt][2] = round_to_dtype(xin, pool.conv_dtype);
              if (dc || tcv) {
                const int64_t ch = gchan(pt, m.h, t);
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                  if (dc) store_elem(dc, ch * 3 + q, pool.conv_dtype, win[pt][q]);
                  if (tcv) store_elem(tcv, ch * 3 + q, pool.conv_dtype, win[pt][q]);
                }
              }
              if (!(REPLAY && pt == 0)) gys[jj * C::CH + cl] = silu_on ? silu(y) : y;
            }
          }
          if (MODE != kDecTree && j0 + gn < ND) {  // the next group starts from this window
#pragma unroll
            for (int pt = 0; pt < 3; ++pt) {
              if (V < D && pt == 2 && t >= V) break;
#pragma unroll
              for (int q = 0; q < 3; ++q)
                store_elem(buf + L.conv, (pt * D + t) * 3 + q, pool.conv_dtype, win[pt][q]);
            }
          }
        } else if (per_key && t >= D && t < 2 * D) {
          const float* sg = reinterpret_cast<const float*>(buf + L.g);
          for (int jj = 0; jj < nl; ++jj) {
            const int nd = MODE == kDecTree ? ord_sm[s][j0 + jj] : j0 + jj;
            gag[jj * D + (t - D)] = expf(sg[nd * D + (t - D)]);
          }
        }
        if (warp < NPW) {
          // this warp's partial q.q, k.k, q.k of each draft (its own conv outputs)
          for (int jj = 0; jj < nl; ++jj) {
            const float yq = (t < D && !REPLAY) ? gys[jj * C::CH + t] : 0.f;
            const float yk = t < D ? gys[jj * C::CH + D + t] : 0.f;
            float pqq = yq * yq, pkk = yk * yk, pqk = yq * yk;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              if (!REPLAY) pqq += __shfl_xor_sync(0xffffffffu, pqq, o);
              pkk += __shfl_xor_sync(0xffffffffu, pkk, o);
              if (!REPLAY) pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
            }
            if (lane == 0) {
              float* nr = gnr + (jj * NPW + warp) * 3;
              nr[0] = pqq;
              nr[1] = pkk;
              nr[2] = pqk;
            }
          }
        }
        // the group's conv outputs published; also agrees on whether any
        // consumer's wait gave up
        if (consumers_sync_or(C::NC, !got)) {
          abort = true;
          break;
        }
        const float* bgs = reinterpret_cast<const float*>(buf + L.bg);
        uint8_t* sst = buf + L.state;
        for (int jj = 0; jj < nl; ++jj) {
          const int j = j0 + jj;
          const int nd = MODE == kDecTree ? ord_sm[s][j] : j;  // the draft run at position j
          const int64_t tok = int64_t(m.r) * ND + nd;
          const float* ys = gys + jj * C::CH;
          const float beta = bgs[2 * nd];
          char* dt = nullptr;
          char* tt = nullptr;
          // a tree node whose parent is not the node run before it starts from
          // the parent's state in the spec buffer (the slot's for a root);
          // each thread reads back only the rows it wrote itself
          const char* src_t = nullptr;
          if (MODE == kDecTree && j > 0) {
            const int pj = par_sm[s][nd];
            if (pj != ord_sm[s][j - 1])
              src_t = pj < 0 ? slot_t
                             : static_cast<const char*>(a.spec.temporal) + a.layer * a.spec.temporal_layer_stride +
                                   m.r * a.spec.temporal_req_stride + pj * a.spec.temporal_step_stride +
                                   m.h * head_bytes;
          }
          if (MODE == kDecVerify || MODE == kDecTree) {
            dt = static_cast<char*>(a.spec.temporal) + a.layer * a.spec.temporal_layer_stride +
                 m.r * a.spec.temporal_req_stride + nd * a.spec.temporal_step_stride + m.h * head_bytes;
          } else if (REPLAY) {
            if (j == m.acc - 1) dt = slot_t;
            if (m.ts >= 0 && a.track_interval > 0 && (m.pos + j + 1) % a.track_interval == 0)
              tt = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                   int64_t(m.ts) * pool.temporal_slot_stride + m.h * head_bytes;
          }
          float sqq = 0.f, skk = 0.f, sqk = 0.f;
#pragma unroll
          for (int pw = 0; pw < NPW; ++pw) {
            const float* nr = gnr + (jj * NPW + pw) * 3;
            sqq += nr[0];
            skk += nr[1];
            sqk += nr[2];
          }
          const float rq = (l2 ? rsqrtf(sqq + kL2Eps) : 1.f) * a.q_scale;
          const float rk = l2 ? rsqrtf(skk + kL2Eps) : 1.f;
          const float kq = sqk * rq * rk;
          uint64_t a2[4], q2[4], k2[4];
          {
            const float4* yq4 = reinterpret_cast<const float4*>(ys + lr * 8);
            const float4* yk4 = reinterpret_cast<const float4*>(ys + D + lr * 8);
            const uint64_t rq2 = f2pack(rq, rq), rk2 = f2pack(rk, rk);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float4 fk = yk4[h2];
              if (REPLAY) {
                q2[2 * h2] = q2[2 * h2 + 1] = 0ull;
              } else {
                const float4 fq = yq4[h2];
                q2[2 * h2] = fmul2(f2pack(fq.x, fq.y), rq2);
                q2[2 * h2 + 1] = fmul2(f2pack(fq.z, fq.w), rq2);
              }
              k2[2 * h2] = fmul2(f2pack(fk.x, fk.y), rk2);
              k2[2 * h2 + 1] = fmul2(f2pack(fk.z, fk.w), rk2);
            }
            if (per_key) {
              const float4* ag4 = reinterpret_cast<const float4*>(gag + jj * D + lr * 8);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const float4 fa = ag4[h2];
                a2[2 * h2] = f2pack(fa.x, fa.y);
                a2[2 * h2 + 1] = f2pack(fa.z, fa.w);
              }
            } else {
              const float av = expf(bgs[2 * nd + 1]);
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) a2[e2] = f2pack(av, av);
            }
          }
#pragma unroll
          for (int rb = 0; rb < C::RPT; rb += C::RB) {
            uint64_t sv[C::RB][4];
            float red[C::NV];
#pragma unroll
            for (int i = 0; i < C::RB; ++i) {
              const int64_t roff = (int64_t(row0 + (rb + i) * C::RSTEP) * D + lr * 8) * ES;
              if (MODE == kDecTree && src_t)
                Pair8<ST>::load(src_t + roff, sv[i]);
              else
                Pair8<ST>::load(sst + roff, sv[i]);
              uint64_t dk2 = 0ull, dq2 = 0ull;
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                sv[i][e2] = fmul2(sv[i][e2], a2[e2]);
                dk2 = ffma2(sv[i][e2], k2[e2], dk2);
                if (!REPLAY) dq2 = ffma2(sv[i][e2], q2[e2], dq2);
              }
              red[2 * i] = f2sum(dk2);
              red[2 * i + 1] = REPLAY ? 0.f : f2sum(dq2);
            }
            // transposing butterfly, as in the one-token path
#pragma unroll
            for (int d = C::LPR / 2, nv = C::NV; d > 0; d >>= 1) {
              if (nv > 1) {
                const bool up = lr & d;
                nv >>= 1;
#pragma unroll
                for (int v = 0; v < C::NV / 2; ++v) {
                  if (v < nv) {
                    const float keep = up ? red[v + nv] : red[v];
                    const float send = up ? red[v] : red[v + nv];
                    red[v] = keep + __shfl_xor_sync(0xffffffffu, send, d);
                  }
                }
              } else {
                red[0] += __shfl_xor_sync(0xffffffffu, red[0], d);
              }
            }
            float u[C::RB];
#pragma unroll
            for (int i = 0; i < C::RB; ++i) {
              const float dk = __shfl_sync(0xffffffffu, red[0], gbase + (2 * i) * VSTEP);
              u[i] = beta * fmaf(-dmul, dk, ys[2 * D + row0 + (rb + i) * C::RSTEP]);
            }
            if (!REPLAY && (my_v & 1) && (lr % VSTEP) == 0) {
              float ui = 0.f;
#pragma unroll
              for (int i = 0; i < C::RB; ++i)
                if (i == (my_v >> 1)) ui = u[i];
              const int row = row0 + (rb + (my_v >> 1)) * C::RSTEP;
              store_elem(a.out, (tok * H + m.h) * V + row, a.out_dtype, fmaf(ui, kq, red[0]));
            }
#pragma unroll
            for (int i = 0; i < C::RB; ++i) {
              const int64_t off = (int64_t(row0 + (rb + i) * C::RSTEP) * D + lr * 8) * ES;
              const uint64_t u2 = f2pack(u[i], u[i]);
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) sv[i][e2] = ffma2(u2, k2[e2], sv[i][e2]);
              if (dt) Pair8<ST>::store(dt + off, sv[i]);
              if (tt) Pair8<ST>::store(tt + off, sv[i]);
              // the next draft starts from the stored (rounded) state: the
              // store to the stage rounds as the others do
              if (ND > 1) Pair8<ST>::store(sst + off, sv[i]);
            }
          }
        }
      }
    } else {
    // one token in place (n_draft == 1): every item runs the token step (with
    // no work when it is empty), so all consumers meet the same barriers
    // whatever they saw
    for (int j = 0; j < 1; ++j, ++tc) {
      float* ys = ysm[tc & 1];
      const int64_t tok = m.r;
      const bool live = m.valid;
      float beta = 0.f, gh = 0.f;
      char* dt = nullptr;
      char* dc = nullptr;
      char* tt = nullptr;
      char* tcv = nullptr;
      float pqq = 0.f, pkk = 0.f, pqk = 0.f;
      if (live) {
        const float* bgs = reinterpret_cast<const float*>(buf + L.bg);
        beta = bgs[2 * j];
        if (!per_key) gh = bgs[2 * j + 1];
        // in place, and into the track slot when the token ends an interval
        dt = slot_t;
        dc = slot_c;
        if (m.ts >= 0 && a.track_interval > 0 && (m.pos + 1) % a.track_interval == 0) {
          tt = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
               int64_t(m.ts) * pool.temporal_slot_stride + m.h * head_bytes;
          tcv = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                int64_t(m.ts) * pool.conv_slot_stride;
        }
        if (t < D) {
          const uint8_t* sx = buf + L.x + j * C::CH * esi;
          float y3[3];
#pragma unroll
          for (int pt = 0; pt < 3; ++pt) {
            if (V < D && pt == 2 && t >= V) break;  // v has V channels
            const int cl = pt * D + t;
            float win[3], w[4];
#pragma unroll
            for (int q = 0; q < 3; ++q) win[q] = load_elem(buf + L.conv, cl * 3 + q, pool.conv_dtype);
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = load_elem(buf + L.w, cl * 4 + q, a.io_dtype);
            const float xin = load_elem(sx, cl, a.io_dtype);
            const float y = w[0] * win[0] + w[1] * win[1] + w[2] * win[2] + w[3] * xin;
            const float nw[3] = {win[1], win[2], round_to_dtype(xin, pool.conv_dtype)};
            const int64_t ch = gchan(pt, m.h, t);
#pragma unroll
            for (int q = 0; q < 3; ++q) {
              store_elem(dc, ch * 3 + q, pool.conv_dtype, nw[q]);
              if (tcv) store_elem(tcv, ch * 3 + q, pool.conv_dtype, nw[q]);
            }
            y3[pt] = silu_on ? silu(y) : y;
            ys[cl] = y3[pt];
          }
          pqq = y3[0] * y3[0];
          pkk = y3[1] * y3[1];
          pqk = y3[0] * y3[1];
        } else if (per_key && t < 2 * D) {
          const float* sg = reinterpret_cast<const float*>(buf + L.g) + j * D;
          agsm[tc & 1][t - D] = expf(sg[t - D]);
        }
        if (warp < NPW) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            pqq += __shfl_xor_sync(0xffffffffu, pqq, o);
            pkk += __shfl_xor_sync(0xffffffffu, pkk, o);
            pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
          }
          if (lane == 0) {
            normsm[tc & 1][warp][0] = pqq;
            normsm[tc & 1][warp][1] = pkk;
            normsm[tc & 1][warp][2] = pqk;
          }
        }
      }
      // conv outputs published; also agrees on whether any consumer's wait gave up
      if (consumers_sync_or(C::NC, !got)) {
        abort = true;
        break;
      }
      if (!live) continue;
      float sqq = 0.f, skk = 0.f, sqk = 0.f;
#pragma unroll
      for (int pw = 0; pw < NPW; ++pw) {
        sqq += normsm[tc & 1][pw][0];
        skk += normsm[tc & 1][pw][1];
        sqk += normsm[tc & 1][pw][2];
      }
      const float rq = (l2 ? rsqrtf(sqq + kL2Eps) : 1.f) * a.q_scale;
      const float rk = l2 ? rsqrtf(skk + kL2Eps) : 1.f;
      const float kq = sqk * rq * rk;
      // this lane's 8 key channels as 4 packed pairs
      uint64_t a2[4], q2[4], k2[4];
      {
        const float4* yq4 = reinterpret_cast<const float4*>(ys + lr * 8);
        const float4* yk4 = reinterpret_cast<const float4*>(ys + D + lr * 8);
        const uint64_t rq2 = f2pack(rq, rq), rk2 = f2pack(rk, rk);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float4 fq = yq4[h2], fk = yk4[h2];
          q2[2 * h2] = fmul2(f2pack(fq.x, fq.y), rq2);
          q2[2 * h2 + 1] = fmul2(f2pack(fq.z, fq.w), rq2);
          k2[2 * h2] = fmul2(f2pack(fk.x, fk.y), rk2);
          k2[2 * h2 + 1] = fmul2(f2pack(fk.z, fk.w), rk2);
        }
        if (per_key) {
          const float4* ag4 = reinterpret_cast<const float4*>(agsm[tc & 1] + lr * 8);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float4 fa = ag4[h2];
            a2[2 * h2] = f2pack(fa.x, fa.y);
            a2[2 * h2 + 1] = f2pack(fa.z, fa.w);
          }
        } else {
          const float av = expf(gh);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) a2[e2] = f2pack(av, av);
        }
      }
      uint8_t* sst = buf + L.state;
#pragma unroll
      for (int rb = 0; rb < C::RPT; rb += C::RB) {
        uint64_t sv[C::RB][4];
        float red[C::NV];
#pragma unroll
        for (int i = 0; i < C::RB; ++i) {
          const int row = row0 + (rb + i) * C::RSTEP;
          const int64_t roff = (int64_t(row) * D + lr * 8) * ES;
          Pair8<ST>::load(sst + roff, sv[i]);
          uint64_t dk2 = 0ull, dq2 = 0ull;
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            sv[i][e2] = fmul2(sv[i][e2], a2[e2]);
            dk2 = ffma2(sv[i][e2], k2[e2], dk2);
            dq2 = ffma2(sv[i][e2], q2[e2], dq2);
          }
          red[2 * i] = f2sum(dk2);
          red[2 * i + 1] = f2sum(dq2);
        }
        // transposing butterfly: after the exchange at distance d the lane
        // keeps the half of its values selected by (lr & d)
#pragma unroll
        for (int d = C::LPR / 2, nv = C::NV; d > 0; d >>= 1) {
          if (nv > 1) {
            const bool up = lr & d;
            nv >>= 1;
#pragma unroll
            for (int v = 0; v < C::NV / 2; ++v) {
              if (v < nv) {
                const float keep = up ? red[v + nv] : red[v];
                const float send = up ? red[v] : red[v + nv];
                red[v] = keep + __shfl_xor_sync(0xffffffffu, send, d);
              }
            }
          } else {
            red[0] += __shfl_xor_sync(0xffffffffu, red[0], d);
          }
        }
        float u[C::RB];
#pragma unroll
        for (int i = 0; i < C::RB; ++i) {
          const float dk = __shfl_sync(0xffffffffu, red[0], gbase + (2 * i) * VSTEP);
          u[i] = beta * fmaf(-dmul, dk, ys[2 * D + row0 + (rb + i) * C::RSTEP]);
        }
        if ((my_v & 1) && (lr % VSTEP) == 0) {
          float ui = 0.f;
#pragma unroll
          for (int i = 0; i < C::RB; ++i)
            if (i == (my_v >> 1)) ui = u[i];
          const int row = row0 + (rb + (my_v >> 1)) * C::RSTEP;
          store_elem(a.out, (tok * H + m.h) * V + row, a.out_dtype, fmaf(ui, kq, red[0]));
        }
#pragma unroll
        for (int i = 0; i < C::RB; ++i) {
          const int64_t off = (int64_t(row0 + (rb + i) * C::RSTEP) * D + lr * 8) * ES;
          const uint64_t u2 = f2pack(u[i], u[i]);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) sv[i][e2] = ffma2(u2, k2[e2], sv[i][e2]);
          Pair8<ST>::store(dt + off, sv[i]);
          if (tt) Pair8<ST>::store(tt + off, sv[i]);
        }
      }
    }
    }  // one-token mode
    if (abort) break;
    // this warp's reads (and, in verify, writes) of the stage are done
    __syncwarp();
    if (ND > 1) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive(empty_bar(s));
  }
}

// ---------------------------------------------------------------------------
// Recurrent prefill. grid (batch, H), block NT. State carried in fp32 for
// the whole request; rounded only where stored.
// ---------------------------------------------------------------------------
struct PrefillParams {
  lin_state_pool_t pool;
  lin_prefill_args_t a;
  const uint32_t* redo;  // when set: run only the (request, head) pairs whose bit is set
};

template <int D, int V, int ST>
__global__ void __launch_bounds__(TokCfg<D, V>::NT, 2) prefill_recurrent_kernel(PrefillParams p) {
  using C = TokCfg<D, V>;
  __shared__ TokSmem<D, V> sm;
  const lin_state_pool_t& pool = p.pool;
  const lin_prefill_args_t& a = p.a;
  const int r = blockIdx.x, h = blockIdx.y;
  const int H = pool.num_heads;
  const int ns = pool.num_slots;
  if (p.redo) {
    const int64_t idx = int64_t(r) * H + h;
    if (!((p.redo[idx >> 5] >> (idx & 31)) & 1u)) return;
  }
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
  const int64_t head_bytes = int64_t(V) * D * ES;
  char* slot_t = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                 slot * pool.temporal_slot_stride + h * head_bytes;
  char* slot_c = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                 slot * pool.conv_slot_stride;
  const bool warm = a.has_initial_state[r] != 0;

  float s[C::RPT][8];
  if (warm) {
    load_rows<D, V, ST>(slot_t, s);
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
    chan[i] = cl < C::CH ? head_channel(cl, h, H, D, V) : 0;
#pragma unroll
    for (int j = 0; j < 3; ++j)
      win[i][j] = (warm && cl < C::CH) ? load_elem(slot_c, int64_t(chan[i]) * 3 + j, pool.conv_dtype) : 0.f;
    if (cl < C::CH) {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[i][j] = load_elem(a.conv_w, int64_t(chan[i]) * 4 + j, a.io_dtype);
    }
  }

  const float dmul = (a.flags & LIN_UPDATE_ADDITIVE) ? 0.f : 1.f;
  const bool per_key = a.gate_mode == LIN_GATE_PER_KEY;
  const int lr = threadIdx.x % C::LPR;
  // a token's inputs (this thread's conv inputs, its 8 log decays or the
  // head's one, beta), loaded a token ahead so their latency hides behind
  // the current token's arithmetic
  float xn[C::CPT], gn[8], bn = 0.f;
  auto load_inputs = [&](int64_t t) {
#pragma unroll
    for (int i = 0; i < C::CPT; ++i) {
      const int cl = threadIdx.x + i * C::NT;
      xn[i] = cl < C::CH ? load_elem(a.x, t * C_all + chan[i], a.io_dtype) : 0.f;
    }
    if (per_key) {
#pragma unroll
      for (int e = 0; e < 8; ++e) gn[e] = a.g[(t * H + h) * D + lr * 8 + e];
    } else {
      gn[0] = a.g[t * H + h];
    }
    bn = a.beta[t * H + h];
  };
  if (bos < eos) load_inputs(bos);
  int snap = 0;
  for (int64_t t = bos; t < eos; ++t) {
    float xc[C::CPT], gc[8];
#pragma unroll
    for (int i = 0; i < C::CPT; ++i) xc[i] = xn[i];
#pragma unroll
    for (int e = 0; e < 8; ++e) gc[e] = gn[e];
    const float beta = bn;
    if (t + 1 < eos) load_inputs(t + 1);
    // one barrier per token: the scratch alternates between tokens, and a
    // thread reaches token t+2's conv only after every thread passed token
    // t+1's barrier, i.e. finished token t's row update
    float* ys = sm.y[(t - bos) & 1];
    float(*part)[2] = sm.part[(t - bos) & 1];
    conv_token_in<D, V>(win, w, xc, a.flags & LIN_CONV_SILU, ys, part);
    __syncthreads();
    float rq = a.q_scale, rk = 1.f;
    if (a.flags & LIN_QK_L2NORM) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int wi = 0; wi < (C::NT + 31) / 32; ++wi) {
        sq += part[wi][0];
        sk += part[wi][1];
      }
      rq = rsqrtf(sq + kL2Eps) * a.q_scale;
      rk = rsqrtf(sk + kL2Eps);
    }
    float a8[8];
    if (per_key) {
#pragma unroll
      for (int e = 0; e < 8; ++e) a8[e] = expf(gc[e]);
    } else {
      const float av = expf(gc[0]);
#pragma unroll
      for (int e = 0; e < 8; ++e) a8[e] = av;
    }
    rows_update<D, V>(s, ys, a8, beta, dmul, rq, rk, a.out, (t * H + h) * V, a.out_dtype);
    const int64_t n = P + (t - bos) + 1;
    if (nt > 0 && n % a.track_stride == 0) {
      const int dst = a.track_slots[t0 + (snap % nt)];
      ++snap;
      if (dst >= 0) {
        char* tt = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                   dst * pool.temporal_slot_stride + h * head_bytes;
        char* tc = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                   dst * pool.conv_slot_stride;
        store_rows<D, V, ST>(tt, s);
        store_window<C::CPT, C::CH>(tc, pool.conv_dtype, chan, win);
      }
    }
  }
  store_rows<D, V, ST>(slot_t, s);
  store_window<C::CPT, C::CH>(slot_c, pool.conv_dtype, chan, win);
}

// Per device: the dynamic shared memory the kernel instance was last opened
// up to, and the CTAs per SM at that size (set-up calls are not repeated on
// every launch).
struct DecodeLaunchCache {
  std::atomic<int> smem_set[kMaxDevices];
  std::atomic<int64_t> occupancy[kMaxDevices];  // (smem << 32) | CTAs per SM
};

template <int D, int V, int ST>
cudaError_t decode_launch(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                          const int32_t* accept, cudaStream_t stream) {
  const int mode = accept ? kDecReplay
                   : (a.n_draft > 1 && a.parent && a.spec.temporal) ? kDecTree
                   : a.n_draft > 1                        ? kDecVerify
                                                          : kDecStates;
  static DecodeLaunchCache caches[5];  // indexed by DecMode
  DecodeLaunchCache& cache = caches[mode];
  DecodeParams p{pool, a, accept, 0, 0};
  const int stage = decode_stage_bytes(pool, a);
  if (stage > kDecodeMaxStage) return cudaErrorInvalidValue;
  // two CTAs per SM when two stages each fit, else one CTA with two stages
  int stages = (100 * 1024) / stage;
  if (stages > kDecMaxStages) stages = kDecMaxStages;
  if (stages < 2) stages = 2;
  int smem = stages * stage;
  int group = 1;
  if (mode != kDecStates) {
    // the draft modes' two group buffers follow the stages: the largest group
    // (up to kDecGroup drafts) that keeps two CTAs per SM where the stages
    // alone would, else that fits one CTA
    const int budget = 2 * stage <= 100 * 1024 ? kDecPairSmem : kDecMaxDynSmem;
    auto gbytes = [](int g) { return 2 * dec_group_floats(D, V, g) * 4; };
    group = a.n_draft < kDecGroup ? a.n_draft : kDecGroup;
    while (group > 1 && smem + gbytes(group) > budget) --group;
    smem += gbytes(group);
    if (smem > kDecMaxDynSmem) return cudaErrorInvalidValue;
    // the replay commit's request order, where it fits the same budget
    const int obytes = ((2 * a.batch + 15) & ~15) + ((4 * (a.n_draft + 1) + 15) & ~15);
    if (mode == kDecReplay && a.batch <= 32767 && smem + obytes <= budget) {
      p.order_off = smem;
      p.hist_off = smem + ((2 * a.batch + 15) & ~15);
      smem += obytes;
    }
  }
  auto kern = mode == kDecReplay        ? decode_kernel<D, V, ST, kDecReplay>
              : mode == kDecTree        ? decode_kernel<D, V, ST, kDecTree>
              : mode == kDecVerify      ? decode_kernel<D, V, ST, kDecVerify>
                                        : decode_kernel<D, V, ST, kDecStates>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (cache.smem_set[dev].load() < smem) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
      return e;
    int cur = cache.smem_set[dev].load();
    while (cur < smem && !cache.smem_set[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  int per_sm = 0;
  const int64_t occ = cache.occupancy[dev].load();
  if ((occ >> 32) == smem && (occ & 0xffffffff) > 0) {
    per_sm = static_cast<int>(occ & 0xffffffff);
  } else {
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DecPCfg<D, V>::NT, smem)) != cudaSuccess)
      return e;
    if (per_sm < 1) per_sm = 1;
    cache.occupancy[dev].store((int64_t(smem) << 32) | per_sm);
  }
  const int items = a.batch * pool.num_heads;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidDevice;
  int grid = sms * per_sm;
  if (grid > items) grid = items;
  kern<<<grid, DecPCfg<D, V>::NT, smem, stream>>>(p, items, stage, stages, group);
  return cudaGetLastError();
}

template <int D, int V, int ST>
cudaError_t prefill_launch(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                           cudaStream_t stream, const uint32_t* redo) {
  PrefillParams p{pool, a, redo};
  prefill_recurrent_kernel<D, V, ST><<<dim3(a.batch, pool.num_heads), TokCfg<D, V>::NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// (head_k, head_v): square heads of 16..128, or 128 key channels with 64 value
// channels (the SSD-style head: state size 128, head dim 64).
#define LIN_DISPATCH_D_ST(FN, D, V, ST, ...)                                          \
  do {                                                                                \
    const bool bf = (ST) == LIN_BF16;                                                 \
    if ((D) == 128 && (V) == 64)                                                      \
      return bf ? FN<128, 64, LIN_BF16>(__VA_ARGS__) : FN<128, 64, LIN_F32>(__VA_ARGS__); \
    if ((D) != (V)) return cudaErrorInvalidValue;                                     \
    switch (D) {                                                                      \
      case 16: return bf ? FN<16, 16, LIN_BF16>(__VA_ARGS__) : FN<16, 16, LIN_F32>(__VA_ARGS__);      \
      case 32: return bf ? FN<32, 32, LIN_BF16>(__VA_ARGS__) : FN<32, 32, LIN_F32>(__VA_ARGS__);      \
      case 64: return bf ? FN<64, 64, LIN_BF16>(__VA_ARGS__) : FN<64, 64, LIN_F32>(__VA_ARGS__);      \
      case 128: return bf ? FN<128, 128, LIN_BF16>(__VA_ARGS__) : FN<128, 128, LIN_F32>(__VA_ARGS__); \
      default: return cudaErrorInvalidValue;                                          \
    }                                                                                 \
  } while (0)

int device_sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev].load();
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev].store(v);
  return v;
}

int decode_stage_bytes(const lin_state_pool_t& pool, const lin_decode_args_t& a) {
  const DecSmem L(pool.head_k, pool.head_v, dtype_size(pool.state_dtype), dtype_size(pool.conv_dtype),
                  dtype_size(a.io_dtype), a.n_draft, a.gate_mode == LIN_GATE_PER_KEY);
  return (L.size + 127) & ~127;
}

cudaError_t launch_decode(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                          const int32_t* accept, cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  LIN_DISPATCH_D_ST(decode_launch, pool.head_k, pool.head_v, pool.state_dtype, pool, a, accept, stream);
}

cudaError_t launch_prefill_recurrent(const lin_state_pool_t& pool,
                                     const lin_prefill_args_t& a, cudaStream_t stream,
                                     const uint32_t* redo) {
  if (a.batch <= 0) return cudaSuccess;
  LIN_DISPATCH_D_ST(prefill_launch, pool.head_k, pool.head_v, pool.state_dtype, pool, a, stream, redo);
}

}  // namespace lin
