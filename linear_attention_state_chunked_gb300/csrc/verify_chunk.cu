// Outputs-only speculative verify as one small chunk (sm_103a).
//
// A verify that keeps no per-step states (the replay form of speculative
// decoding: the Kimi-K3 notes' ReplaySSM, the MambaRadixCache page's deferred
// update, 9.2 - 9.10) needs only the n_draft drafts' outputs. No state is
// stored between drafts, so the state is carried exactly (fp32) from the
// slot's state S0 across the drafts, as inside a prefill call. With the
// drafts as one chunk of D tokens, b_j the cumulative log decay up to draft j
// (per key channel, or per head) and gamma_j = exp(b_j), the recurrence of
// the Kimi-K3 notes ("Speculative decoding")
//     S_j = S_{j-1} Diag(alpha_j) + beta_j (v_j - S_{j-1} Diag(alpha_j) k_j) k_j^T,
//     o_j = S_j q_j
// unrolls to (the same algebra as the chunked prefill):
//     A[t][i] = beta_t sum_c k_tc k_ic exp(b_tc - b_ic)      (i < t)
//     T       = (I + A)^-1 Diag(beta)
//     P[t][i] = sum_c q_tc k_ic exp(b_tc - b_ic)             (i <= t)
//     U       = T (V - Khat S0^T),   Khat = gamma . K
//     O       = Qhat S0^T + P U,     Qhat = gamma . Q
// so each state row v is read once and needs only 2D dot products
// (kS_j = S0[v] . khat_j, qS_j = S0[v] . qhat_j) plus D x D algebra: no
// draft-by-draft pass over the state. The additive (Mamba2 SSD) form is the
// same with A = 0 (T = Diag(beta), U = T V: no kS).
//
// One CTA of 256 threads per (request, head). The inputs arrive in shared
// memory by bulk async copies; each warp loads its 16 state rows straight into
// the registers of a tensor-core operand (issued first, so they are in flight
// while the conv, norms, gates and the D x D products run). The row products
// S0 [Khat; Qhat]^T (M = 16 rows per warp, N = 8 quantities, K = 16 key
// channels per step) run as warp-level bf16 MMAs with fp32 accumulation; the
// fp32 factors khat / qhat (and an fp32 state) enter as bf16 high / low pairs,
// 16 significant bits.

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace lin {
namespace {

constexpr int VT = 256;  // threads
constexpr uint32_t kVerWaitTries = 1u << 26;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

template <int K, int V, int ST>
struct VerCfg {
  static constexpr int CH = 2 * K + V;                 // conv channels of a head
  static constexpr int ES = ST == LIN_BF16 ? 2 : 4;
  static constexpr int SBYTES = V * K * ES;            // the state block
  static constexpr int KSTEPS = K / 16;                // MMA steps over the key channels
  static constexpr int RT = V / 16;                    // 16-row tiles of the state (one per warp)
  static_assert(RT >= 1 && RT <= VT / 32 && K % 16 == 0, "tile mapping");
};

// Dynamic shared memory: the state block and the inputs as they arrive by
// bulk copies, then fp32 arrays of the D drafts.
struct VerSmem {
  int s, win, taps, xs, gs, y, b, kh, qh, ks, qs, u, a, p, x, t, rn, bt, size;
  __host__ __device__ VerSmem(int K, int V, int ies, int ces, int D, bool kda) {
    const int CH = 2 * K + V;
    auto al = [](int v) { return (v + 15) & ~15; };
    s = 0;
    win = 0;                          // the slot's conv window of the head's channels [CH][3]
    taps = win + al(CH * 3 * ces);    // conv taps [CH][4]
    xs = taps + al(CH * 4 * ies);     // the drafts' inputs [D][CH]
    gs = xs + al(D * CH * ies);       // per-key log decay [D][K]
    y = gs + (kda ? D * K * 4 : 0);   // conv outputs [D][CH] (q, k normalised in place)
    b = y + D * CH * 4;               // cumulative log decay [D][K]
    kh = b + D * K * 4;               // gamma . k [D][K]
    qh = kh + D * K * 4;              // gamma . q [D][K]
    ks = qh + D * K * 4;              // S0 khat_j per row [D][V]
    qs = ks + D * V * 4;              // S0 qhat_j per row [D][V]
    u = qs + D * V * 4;               // U [D][V]
    a = u + D * V * 4;                // A [D][D]
    p = a + D * D * 4;                // P [D][D]
    x = p + D * D * 4;                // X = (I + A)^-1 [D][D]
    t = x + D * D * 4;                // T [D][D]
    rn = t + D * D * 4;               // 1 / norms: q then k [2][D]
    bt = rn + 2 * D * 4;              // beta [D]
    size = bt + D * 4;
  }
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait for phase 0 of an mbarrier: false when it did not complete.
__device__ __forceinline__ bool wait_phase0(uint32_t bar) {
  for (uint32_t it = 0; it < kVerWaitTries; ++it) {
    uint32_t okp;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(okp)
        : "r"(bar)
        : "memory");
    if (okp) return true;
  }
  return false;
}

// d += a b, m16n8k16, bf16 operands, fp32 accumulators (warp-level MMA)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values as a bf16 pair (x in the low half) and the pair of their
// remainders, so hi + lo holds 16 significant bits of each.
__device__ __forceinline__ void bf16_split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 f = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - f.x, y - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float ld_smem_elem(const uint8_t* base, int i, int es) {
  return es == 2 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(base)[i]) << 16)
                 : reinterpret_cast<const float*>(base)[i];
}

struct VerParams {
  lin_state_pool_t pool;
  lin_decode_args_t a;
  int resident;  // CTAs resident at once: the item one wave ahead is blockIdx.x + resident
};

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int K, int V, int ST, bool KDA>
__global__ void __launch_bounds__(VT, ST == LIN_BF16 ? 4 : 2) verify_chunk_kernel(const VerParams prm) {
  using C = VerCfg<K, V, ST>;
  extern __shared__ __align__(16) uint8_t vsm[];
  __shared__ uint64_t bar_in;
  __shared__ int ok_sh;
  const lin_state_pool_t& pool = prm.pool;
  const lin_decode_args_t& a = prm.a;
  const int H = pool.num_heads, D = a.n_draft;
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot = a.slot[r];
  if (slot < 0) return;  // padding
  if (slot >= pool.num_slots) {
    if (h == 0 && tid == 0) report(a.status, LIN_ST_BAD_SLOT);
    return;
  }
  const int ies = dtype_size(a.io_dtype), ces = dtype_size(pool.conv_dtype);
  const VerSmem L(K, V, ies, ces, D, KDA);
  float* Y = reinterpret_cast<float*>(vsm + L.y);
  float* B = reinterpret_cast<float*>(vsm + L.b);
  float* KH = reinterpret_cast<float*>(vsm + L.kh);
  float* QH = reinterpret_cast<float*>(vsm + L.qh);
  float* KS = reinterpret_cast<float*>(vsm + L.ks);
  float* QS = reinterpret_cast<float*>(vsm + L.qs);
  float* A = reinterpret_cast<float*>(vsm + L.a);
  float* Pm = reinterpret_cast<float*>(vsm + L.p);
  float* Xm = reinterpret_cast<float*>(vsm + L.x);
  float* UU = reinterpret_cast<float*>(vsm + L.u);
  float* Tm = reinterpret_cast<float*>(vsm + L.t);
  float* RN = reinterpret_cast<float*>(vsm + L.rn);
  float* BT = reinterpret_cast<float*>(vsm + L.bt);
  const float* GS = reinterpret_cast<const float*>(vsm + L.gs);

  const char* slot_t = static_cast<const char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                       slot * pool.temporal_slot_stride + int64_t(h) * C::SBYTES;
  const char* slot_c = static_cast<const char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                       slot * pool.conv_slot_stride;
  const bool additive = (a.flags & LIN_UPDATE_ADDITIVE) != 0;
  const int C_all = pool.conv_channels;

  // ---- this warp's 16 state rows (tile `warp`) as MMA operand registers.
  // Within each 16-channel step thread (g, t) takes key channels 4t .. 4t+3
  // of rows g and g + 8 as its A elements (columns 2t, 2t+1 | 2t+8, 2t+9 of
  // the fragment); the B fragments below take the same channels, so the sum
  // over the step is unchanged. Issued first: in flight during the conv.
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t abf[ST == LIN_BF16 ? C::KSTEPS : 1][4];
  float4 af[ST == LIN_BF16 ? 1 : C::KSTEPS][2];
  if (warp < C::RT) {
    const char* r0 = slot_t + int64_t(warp * 16 + g8) * K * C::ES;
    const char* r1 = r0 + int64_t(8) * K * C::ES;
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      const int off = (ks * 16 + 4 * t4) * C::ES;
      if constexpr (ST == LIN_BF16) {
        const uint2 u0 = __ldg(reinterpret_cast<const uint2*>(r0 + off));
        const uint2 u1 = __ldg(reinterpret_cast<const uint2*>(r1 + off));
        abf[ks][0] = u0.x;  // row g, channels 4t, 4t+1
        abf[ks][1] = u1.x;  // row g+8
        abf[ks][2] = u0.y;  // row g, channels 4t+2, 4t+3
        abf[ks][3] = u1.y;
      } else {
        af[ks][0] = __ldg(reinterpret_cast<const float4*>(r0 + off));
        af[ks][1] = __ldg(reinterpret_cast<const float4*>(r1 + off));
      }
    }
  }

  // ---- the inputs by bulk async copies (window, taps, the drafts' x rows and
  // per-key gates), completing on bar_in
  const uint32_t bi = smem_addr(&bar_in);
  // per part (q, k, v): the head's first channel, its first channel within the
  // head, the part's channels
  auto part_c0 = [&](int pp) { return pp == 0 ? h * K : pp == 1 ? H * K + h * K : 2 * H * K + h * V; };
  auto part_l0 = [&](int pp) { return pp * K; };
  auto part_n = [&](int pp) { return pp == 2 ? V : K; };
  if (warp == 0) {
    if (lane == 0) {
      ok_sh = 1;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bi) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      const uint32_t in_bytes = C::CH * 3 * ces + C::CH * 4 * ies + D * C::CH * ies + (KDA ? D * K * 4 : 0);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bi), "r"(in_bytes) : "memory");
    }
    __syncwarp();
    // copy q of 6 + 3D (+ D): window parts, tap parts, x rows per draft and
    // part, per-key gate rows per draft
    const int nq = 6 + 3 * D + (KDA ? D : 0);
    for (int q = lane; q < nq; q += 32) {
      if (q < 3) {
        bulk_g2s(smem_addr(vsm + L.win) + part_l0(q) * 3 * ces, slot_c + int64_t(part_c0(q)) * 3 * ces,
                 part_n(q) * 3 * ces, bi);
      } else if (q < 6) {
        const int pp = q - 3;
        bulk_g2s(smem_addr(vsm + L.taps) + part_l0(pp) * 4 * ies,
                 static_cast<const char*>(a.conv_w) + int64_t(part_c0(pp)) * 4 * ies, part_n(pp) * 4 * ies, bi);
      } else if (q < 6 + 3 * D) {
        const int j = (q - 6) / 3, pp = (q - 6) % 3;
        bulk_g2s(smem_addr(vsm + L.xs) + (j * C::CH + part_l0(pp)) * ies,
                 static_cast<const char*>(a.x) + ((int64_t(r) * D + j) * C_all + part_c0(pp)) * ies,
                 part_n(pp) * ies, bi);
      } else {
        const int j = q - 6 - 3 * D;
        bulk_g2s(smem_addr(vsm + L.gs) + j * K * 4, a.g + ((int64_t(r) * D + j) * H + h) * K, K * 4, bi);
      }
    }
  }
  // The CTAs run in waves of `resident`, each waiting first for its inputs
  // from HBM: the last warp has L2 fetch the inputs of the item one wave
  // ahead (state rows, window, the drafts' x rows and per-key gates), so that
  // CTA finds them in L2.
  if (warp == VT / 32 - 1) {
    const int nx = static_cast<int>(blockIdx.x) + prm.resident;
    if (prm.resident > 0 && nx < a.batch * H) {
      const int r1 = nx / H, h1 = nx % H;
      const int s1 = a.slot[r1];
      if (s1 >= 0 && s1 < pool.num_slots) {
        const char* t1 = static_cast<const char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                         s1 * pool.temporal_slot_stride + int64_t(h1) * C::SBYTES;
        const char* c1 = static_cast<const char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                         s1 * pool.conv_slot_stride;
        auto c0_1 = [&](int pp) { return pp == 0 ? h1 * K : pp == 1 ? H * K + h1 * K : 2 * H * K + h1 * V; };
        const int nq = 1 + 3 + 3 * D + (KDA ? D : 0);
        for (int q = lane; q < nq; q += 32) {
          if (q == 0) {
            prefetch_l2(t1, C::SBYTES);
          } else if (q < 4) {
            prefetch_l2(c1 + int64_t(c0_1(q - 1)) * 3 * ces, part_n(q - 1) * 3 * ces);
          } else if (q < 4 + 3 * D) {
            const int j = (q - 4) / 3, pp = (q - 4) % 3;
            prefetch_l2(static_cast<const char*>(a.x) + ((int64_t(r1) * D + j) * C_all + c0_1(pp)) * ies,
                        part_n(pp) * ies);
          } else {
            const int j = q - 4 - 3 * D;
            prefetch_l2(a.g + ((int64_t(r1) * D + j) * H + h1) * K, K * 4);
          }
        }
      }
    }
  }
  // per-head gates and beta: one thread per draft, loaded while the copies land
  float g_own = 0.f, b_own = 0.f;
  if (tid < D) {
    const int64_t rj = int64_t(r) * D + tid;
    if (!KDA) g_own = a.g[rj * H + h];
    b_own = a.beta[rj * H + h];
  }
  if (tid == 0 && !wait_phase0(bi)) {
    ok_sh = 0;
    report(a.status, LIN_ST_TIMEOUT);
  }
  __syncthreads();
  if (!ok_sh) {
    // the copies may still land: wait for them (bounded) before the CTA exits
    if (tid == 0) wait_phase0(bi);
    return;
  }
  if (tid < D) {
    BT[tid] = b_own;
    if (!KDA) B[tid * K] = g_own;  // summed below
  }

  // ---- conv over the D drafts (window from the slot), SiLU
  for (int cl = tid; cl < C::CH; cl += VT) {
    float w[4], win[3];
#pragma unroll
    for (int m = 0; m < 4; ++m) w[m] = ld_smem_elem(vsm + L.taps, cl * 4 + m, ies);
#pragma unroll
    for (int m = 0; m < 3; ++m) win[m] = ld_smem_elem(vsm + L.win, cl * 3 + m, ces);
    for (int j = 0; j < D; ++j) {
      const float xn = ld_smem_elem(vsm + L.xs, j * C::CH + cl, ies);
      float y = w[0] * win[0] + w[1] * win[1] + w[2] * win[2] + w[3] * xn;
      win[0] = win[1];
      win[1] = win[2];
      win[2] = xn;
      if (a.flags & LIN_CONV_SILU) y = silu(y);
      Y[j * C::CH + cl] = y;
    }
  }
  __syncthreads();
  // cumulative log decay per draft: per key channel (KDA) or per head
  for (int c = tid; c < (KDA ? K : 1); c += VT) {
    float run = 0.f;
    for (int j = 0; j < D; ++j) {
      run += KDA ? GS[j * K + c] : B[j * K];
      B[j * K + c] = run;
    }
  }
  if (!KDA) {
    __syncthreads();
    for (int i = tid; i < D * K; i += VT) B[i] = B[(i / K) * K];
  }
  __syncthreads();

  // ---- 1 / L2 norms of q and k per draft (one warp per quantity)
  for (int qd = warp; qd < 2 * D; qd += VT / 32) {
    const int j = qd >> 1, part = qd & 1;
    const float* src = Y + j * C::CH + part * K;
    float ss = 0.f;
    for (int c = lane; c < K; c += 32) ss += src[c] * src[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0)
      RN[part * D + j] = (a.flags & LIN_QK_L2NORM) ? rsqrtf(ss + 1e-6f) : 1.f;
  }
  __syncthreads();
  // normalised q (with q_scale) and k in place; gamma . q and gamma . k
  for (int i = tid; i < D * K; i += VT) {
    const int j = i / K, c = i % K;
    float* yq = Y + j * C::CH + c;
    float* yk = yq + K;
    const float qn = *yq * RN[j] * a.q_scale, kn = *yk * RN[D + j];
    *yq = qn;
    *yk = kn;
    const float gam = __expf(B[j * K + c]);
    QH[j * K + c] = qn * gam;
    KH[j * K + c] = kn * gam;
  }
  __syncthreads();

  // ---- A and P: one warp per (t, i), i <= t
  for (int pr = warp; pr < D * (D + 1) / 2; pr += VT / 32) {
    int t = 0;
    while ((t + 1) * (t + 2) / 2 <= pr) ++t;
    const int i = pr - t * (t + 1) / 2;
    const float* qt = Y + t * C::CH;
    const float* kt = qt + K;
    const float* ki = Y + i * C::CH + K;
    float sa = 0.f, sp = 0.f;
    const float dh = KDA ? 0.f : __expf(B[t * K] - B[i * K]);
    for (int c = lane; c < K; c += 32) {
      const float e = KDA ? __expf(B[t * K + c] - B[i * K + c]) : dh;
      sp += qt[c] * ki[c] * e;
      sa += kt[c] * ki[c] * e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sp += __shfl_xor_sync(0xffffffffu, sp, o);
      sa += __shfl_xor_sync(0xffffffffu, sa, o);
    }
    if (lane == 0) {
      Pm[t * D + i] = sp;
      A[t * D + i] = (i < t && !additive) ? BT[t] * sa : 0.f;
    }
  }
  __syncthreads();
  // T = (I + A)^-1 Diag(beta): column i of X = (I + A)^-1 by forward substitution
  if (tid < D) {
    const int i = tid;
    for (int t = 0; t < D; ++t) {
      float xv = (t == i) ? 1.f : 0.f;
      if (t > i) {
        float acc = 0.f;
        for (int m = i; m < t; ++m) acc = fmaf(A[t * D + m], Xm[m * D + i], acc);
        xv = -acc;
      }
      Xm[t * D + i] = xv;  // column i is this thread's alone
      Tm[t * D + i] = xv * BT[i];
    }
  }

  // ---- the row products kS_j = S0[v] . khat_j, qS_j = S0[v] . qhat_j: one
  // 16-row tile per warp, quantities in groups of 8 (N), khat then qhat (the
  // additive form needs only qhat)
  __syncthreads();  // KH, QH
  if (warp < C::RT) {
    float* KQS = KS;  // KS [D][V] then QS [D][V]: quantity n at KQS + n * V
    const int q0 = additive ? D : 0;
    for (int nt = 0; q0 + nt * 8 < 2 * D; ++nt) {
      const int n = q0 + nt * 8 + g8;  // this lane's B column
      const float* vec = n < D ? KH + n * K : (n < 2 * D ? QH + (n - D) * K : nullptr);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vec) bv = *reinterpret_cast<const float4*>(vec + ks * 16 + 4 * t4);
        uint32_t b0h, b0l, b1h, b1l;
        bf16_split2(bv.x, bv.y, b0h, b0l);
        bf16_split2(bv.z, bv.w, b1h, b1l);
        if constexpr (ST == LIN_BF16) {
          mma_bf16(d, abf[ks][0], abf[ks][1], abf[ks][2], abf[ks][3], b0h, b1h);
          mma_bf16(d, abf[ks][0], abf[ks][1], abf[ks][2], abf[ks][3], b0l, b1l);
        } else {
          uint32_t ah[4], al[4];
          bf16_split2(af[ks][0].x, af[ks][0].y, ah[0], al[0]);
          bf16_split2(af[ks][1].x, af[ks][1].y, ah[1], al[1]);
          bf16_split2(af[ks][0].z, af[ks][0].w, ah[2], al[2]);
          bf16_split2(af[ks][1].z, af[ks][1].w, ah[3], al[3]);
          mma_bf16(d, ah[0], ah[1], ah[2], ah[3], b0h, b1h);
          mma_bf16(d, ah[0], ah[1], ah[2], ah[3], b0l, b1l);
          mma_bf16(d, al[0], al[1], al[2], al[3], b0h, b1h);
        }
      }
      // d[0], d[1]: row g, quantities 2t, 2t+1 of the group; d[2], d[3]: row g+8
      const int v = warp * 16 + g8;
      const int qa = q0 + nt * 8 + 2 * t4;
      if (qa < 2 * D) {
        KQS[qa * V + v] = d[0];
        KQS[qa * V + v + 8] = d[2];
      }
      if (qa + 1 < 2 * D) {
        KQS[(qa + 1) * V + v] = d[1];
        KQS[(qa + 1) * V + v + 8] = d[3];
      }
    }
  }
  __syncthreads();

  // ---- outputs: U = T (V - kS) (U = T V in the additive form), then
  // O = qS + P U; one thread per (row v, draft)
  for (int i = tid; i < D * V; i += VT) {
    const int t = i / V, v = i % V;
    float acc = 0.f;
    for (int j = 0; j <= t; ++j) {
      const float vj = Y[j * C::CH + 2 * K + v];
      acc = fmaf(Tm[t * D + j], additive ? vj : vj - KS[j * V + v], acc);
    }
    UU[t * V + v] = acc;
  }
  __syncthreads();
  for (int i = tid; i < D * V; i += VT) {
    const int t = i / V, v = i % V;
    float o = QS[t * V + v];
    for (int m = 0; m <= t; ++m) o = fmaf(Pm[t * D + m], UU[m * V + v], o);
    store_elem(a.out, ((int64_t(r) * D + t) * H + h) * V + v, a.out_dtype, o);
  }
}

}  // namespace

int verify_chunk_smem(const lin_state_pool_t& pool, const lin_decode_args_t& a) {
  return VerSmem(pool.head_k, pool.head_v, dtype_size(a.io_dtype), dtype_size(pool.conv_dtype), a.n_draft,
                 a.gate_mode == LIN_GATE_PER_KEY)
      .size;
}

namespace {
template <int K, int V, int ST>
cudaError_t verify_chunk_launch(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                                cudaStream_t stream) {
  const int smem = verify_chunk_smem(pool, a);
  const bool kda = a.gate_mode == LIN_GATE_PER_KEY;
  auto kern = kda ? verify_chunk_kernel<K, V, ST, true> : verify_chunk_kernel<K, V, ST, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, VT, smem)) != cudaSuccess) return e;
  VerParams p{pool, a, per_sm * device_sm_count(dev)};
  kern<<<static_cast<unsigned>(a.batch) * pool.num_heads, VT, smem, stream>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_verify_chunk(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                                cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  if (a.n_draft < 2 || a.n_draft > kVerifyChunkMaxDraft) return cudaErrorInvalidValue;
  const bool bf = pool.state_dtype == LIN_BF16;
  const int K = pool.head_k, V = pool.head_v;
#define LIN_VC(KK, VV) \
  return bf ? verify_chunk_launch<KK, VV, LIN_BF16>(pool, a, stream) : verify_chunk_launch<KK, VV, LIN_F32>(pool, a, stream)
  if (K == 128 && V == 128) LIN_VC(128, 128);
  if (K == 128 && V == 64) LIN_VC(128, 64);
  if (K == 64 && V == 64) LIN_VC(64, 64);
  if (K == 32 && V == 32) LIN_VC(32, 32);
  if (K == 16 && V == 16) LIN_VC(16, 16);
#undef LIN_VC
  return cudaErrorInvalidValue;
}

}  // namespace lin
