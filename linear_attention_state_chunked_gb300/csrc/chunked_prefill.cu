// Chunked tensor-core prefill of the gated delta rule (sm_103a: tcgen05 MMAs
// with fp32 accumulators in tensor memory, TMA-staged inputs).
//
// The recurrence is the KDA / GDN update of the Kimi-K3 notes
// ("企业官网建设流程全解析", "Speculative decoding"):
//     S_t = S_{t-1} Diag(alpha_t) + d_t k_t^T,  d_t = beta_t (v_t - S_{t-1} Diag(alpha_t) k_t),
//     o_t = S_t q_t.
// The pages fix 64-token chunks aligned to absolute positions (Ping-Pong
// page, parameters: FLA_CHUNK_SIZE = 64) but give no chunked algorithm; the
// form below follows from the update by algebra. Inside a chunk starting from
// state S0, with b_t = sum_{s<=t} log alpha_s (per key channel) and
// gamma_t = exp(b_t):
//     A[t][i] = beta_t sum_c k_tc k_ic exp(b_tc - b_ic)   (i < t)
//     T       = (I + A)^-1 Diag(beta)
//     W       = T (gamma . K),   U' = T V,   U = U' - W S0^T
//     P[t][i] = sum_c q_tc k_ic exp(b_tc - b_ic)          (i <= t)
//     O       = (gamma . Q) S0^T + P U
//     S_end   = S0 Diag(gamma_last) + U^T ((gamma_last / gamma) . K)
// Since U = U' - W S0^T = T (V - Khat S0^T), the correction by the incoming
// state is applied to V before the solve's result is used: V' = V - Khat S0^T
// needs only S0 and gamma . K, so it runs next to MMA1 while the solve does,
// and W is never formed. Every product runs with V (= 128) as the MMA M
// dimension, so the state row v is TMEM lane v and all MMAs are M = 128
// (cta_group::1):
//     MMA1  [A';P'] = [K_l;Q_l] K_r^T            N = 64,  K = 128
//     MMAV  V'^T = V^T + S0 (-Khat)^T             N = 64,  K = 128 (from V^T in TMEM)
//     MMA2  U^T = V'^T T^T                        N = 64,  K = 64
// (MMA4a needs only S0 and gamma . Q, so it is issued right after MMA1 and runs
// while the solve does; MMA4b accumulates onto it.)
//     MMA4  O^T = S0 Qhat^T + U^T P^T             N = 64,  K = 128 + 64
//     MMA5  S   = S0 Diag(gamma_last) + U^T Ktil  N = 128, K = 64
// The additive (Mamba2 SSD) form S_t = S_{t-1} Diag(alpha_t) + beta_t v_t k_t^T of
// the MambaRadixCache page (section 9.3) is the same with A = 0: T = Diag(beta),
// U = T V (no solve, no MMAV).
// (KDA: K_l = k exp(b - b_ref), Q_l = q exp(b - b_ref), K_r = k exp(b_ref - b)
// with b_ref the chunk's middle row, so no exponent leaves +-(half a chunk);
// GDN: the scalar decay exp(b_t - b_i) is applied in fp32 to A' and P'.)
// The state is carried in fp32 in tensor memory across chunks and written
// (rounded to the pool dtype) at every snapshot boundary and at the end.
// Operand precision follows the pool's state dtype:
//   - fp32 pools (and every GDN pool): fp16 operands (10-bit mantissa; every
//     decay-scaled factor stays within [0, 1]) with high / low splits on the
//     products that set the error: T, V', P and U. GDN's MMA1 takes single
//     fp16 operands (its products enter A and P with fp32 decay factors); KDA's
//     MMA1 factors exp(+-(b - b_ref)) leave fp16 range, so that product takes
//     bf16 operands with a split (hi = bf16(x), lo = bf16(x - hi): 16
//     significant bits, fp32 range).
//   - KDA with a bf16 pool: bf16 operands, single products (the pool itself
//     holds 8 significant bits).
// A KDA (request, head) whose decay leaves the factored range (some key
// channel decaying by more than e^80 across half a chunk) stops before it
// writes its state back and is flagged; a token-by-token launch queued behind
// this one then reruns exactly the flagged pairs from the untouched slot.
//
// One CTA (16 warps) runs one (request, head) sequentially over its chunks.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace lin {
namespace {

constexpr int CH = 64;       // chunk length
constexpr int DH = 128;      // head dim (K = V)
constexpr int NT = 512;      // threads (16 warps)
constexpr int NW = NT / 32;
constexpr int TPW = CH / NW; // tokens per warp in the conv phase
constexpr int XR = CH + 3;   // rows of a staged x tile (3 halo rows)
constexpr uint32_t kWaitTries = 1u << 26;
// The thread that issues the TMA stores of outputs and states and owns their
// bulk groups: lane 0 of warp 1, so thread 0's wait for the next x tile runs
// beside the store issue instead of after it.
constexpr int kStoreTid = 32;

// Shared-memory map (offsets from a 1024-byte aligned base). Regions are
// reused once their previous contents have been consumed by an MMA.
constexpr uint32_t OFF_SOP = 0;                 // S0 operand, rows v, 128 x 128 16-bit
constexpr uint32_t OFF_STG = 32768;             // epilogue: state tiles for TMA stores (64 KB)
constexpr uint32_t OFF_KQ = 32768;              // [K_l; Q_l] (high part), 128 rows x 128
constexpr uint32_t OFF_TT = OFF_KQ;             //   after MMA1: T (high), 64 x 64
constexpr uint32_t OFF_TTL = OFF_KQ + 8192;     //   after MMA1: T (low part, GDN)
constexpr uint32_t OFF_PP = OFF_KQ + 16384;     //   after MMA1: P (high), 64 x 64
constexpr uint32_t OFF_PPL = OFF_KQ + 24576;    //   after MMA1: P (low part, GDN)
constexpr uint32_t OFF_KQL = 65536;             // [K; Q] low part (GDN), 128 rows x 128
constexpr int AXS = 68;                         // row stride (floats) of the fp32 A / X matrix
constexpr uint32_t OFF_AX = OFF_KQL;            //   after MMA1: fp32 A / X [64][AXS]
constexpr int XDS = 20;                         // row stride (floats) of a 16 x 16 solve block
constexpr int XBS = 16 * XDS;                   // floats per 16 x 16 solve block
constexpr int ZS = 36;                          // row stride (floats) of the 32 x 32 solve block
constexpr uint32_t OFF_XD = OFF_KQL + 64 * AXS * 4;  // after MMA1: fp32 diagonal inverses [4][16][XDS]
constexpr uint32_t OFF_YB = OFF_XD + 4 * XBS * 4;    //   after MMA1: fp32 A_10 X_00, A_32 X_22 [2][16][XDS]
constexpr uint32_t OFF_ZB = OFF_YB + 2 * XBS * 4;    //   after MMA1: fp32 A_BA X_A [32][ZS]
constexpr uint32_t OFF_OSTG = 98304;            // epilogue: output tile for a TMA store (32 KB)
constexpr uint32_t OFF_KR = 98304;              // K_r (KDA), 64 x 128
constexpr uint32_t OFF_UTL = OFF_KR;            //   after MMA2: U^T low part (split products), rows v
constexpr uint32_t OFF_KQH = 114688;            // [-gamma . K; gamma . Q], rows t and 64 + t (K-major B
                                                // of MMAV and MMA4a: one N = 128 product), 128 x 128
constexpr uint32_t OFF_VPT = OFF_KQH;           //   after MMAV: V'^T (high), rows v (K-major A of MMA2)
constexpr uint32_t OFF_UT = OFF_KQH + 16384;    //   after MMA2: U^T (high), rows v (K-major A)
constexpr uint32_t OFF_VV = 147456;             // V, rows t (read into TMEM for MMAV; MN-major A of the additive MMA2)
constexpr uint32_t OFF_KT = 163840;             // (gamma_last/gamma) . K, rows i (MN-major B)
constexpr uint32_t OFF_KRL = 180224;            // K_r low part (KDA with fp32 state), 64 x 128
constexpr uint32_t OFF_VPTL = OFF_KRL;          //   after MMA1: V'^T low part (split products), rows v
constexpr uint32_t OFF_WC = OFF_KRL + 16384;    // conv taps, fp32 [4][384] (tap-major)
constexpr uint32_t OFF_HALO = OFF_WC + 6144;    // initial conv window, fp32 [3][384]
constexpr uint32_t OFF_WTOT = OFF_HALO + 4608;  // per-warp gate sums, fp32 [16][128]
constexpr uint32_t OFF_SBETA = OFF_WTOT + 8192; // beta_t, fp32 [64]
constexpr uint32_t OFF_SB = OFF_SBETA + 256;    // GDN b_t, fp32 [64]
constexpr uint32_t OFF_GLAST = OFF_SB + 256;    // exp(b_last), fp32 [128]
constexpr uint32_t OFF_CF = OFF_GLAST + 512;    // GDN column decay factors, fp32 [64]
constexpr uint32_t OFF_WIN = OFF_CF + 256;      // last 3 inputs of chunks j even / odd, fp32 [2][3][384]
constexpr uint32_t SMEM_USED = OFF_WIN + 2 * 3 * 384 * 4;
// The next chunk's x tile (q | k | v parts of this head, 64 rows x 128 bf16
// each, row-major) lands in the V / K-tilde / K_r-low operand regions, which
// are free once a chunk's last MMA has completed.
constexpr uint32_t OFF_XT = OFF_VV;
static_assert(OFF_KT == OFF_VV + 16384 && OFF_KRL == OFF_KT + 16384, "x tile spans three regions");
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_ZB + 32 * ZS * 4 <= OFF_KR, "solve scratch inside the low-part region");

// Tensor-memory columns (all 512 of the SM; the kernel runs one CTA per SM).
constexpr uint32_t COL_S = 0;    // state, fp32, lanes v
constexpr uint32_t COL_R1 = 128; // [A';P'] -> U^T
constexpr uint32_t COL_R2 = 192; // V^T -> V'^T
constexpr uint32_t COL_RO = 256; // O^T (MMA4a is issued with MMA1)
constexpr uint32_t TMEM_COLS = 512;


// Segmented run of one long request (batch of 1). The state after a chunk is
// affine in the state before it, S' = S A_c + (U'^T K-tilde) with
// A_c = Gamma - W^T K-tilde, so a segment of chunks maps S to S M + B. Mode 1
// runs each segment from a zero state (its B; segment 0 from the request's
// own initial state, giving the true state after it), mode 2 runs segments >= 1
// from the identity with zero values (their M: rows evolve independently, and a
// zero value input drops the U' term), both writing only the fp32 state at the
// segment's end; after the scan S_{k+1} = S_k M_k + B_k, mode 3 runs every
// segment from its true initial state with outputs and snapshots. Segment 0's
// offset run starts from the true state, so it also writes its outputs and
// snapshots; the offset and transition runs share one launch.
enum SegMode { kSegOff = 0, kSegOffset = 1, kSegTransition = 2, kSegFinal = 3, kSegOffsetAndTransition = 4 };

// Wrap-around schedule of a varlen batch (McNaughton's wrap-around rule for
// preemptive scheduling on identical machines). The batch's (request, head)
// chains of n_r chunks are laid end to end and cut into `grid` ranges of T
// chunk units, T >= the longest chain, one range per SM. A chain crossing the
// boundary between ranges m and m + 1 becomes two pieces: its first chunks
// run at the start of range m + 1 and hand the state on; its last chunks run
// at the end of range m, from that state. The head ends by unit time
// x <= T - (n - x), when the tail starts. Each piece has its planned start
// time in its range; CTAs take pieces in that order from a counter (list
// scheduling), so every wait is for a piece taken earlier, whose first piece
// waits for nothing: no deadlock, whatever runs concurrently.
struct WrapPiece {
  int32_t r, h, c0, c1;  // request, head, chunks [c0, c1)
  int32_t mode;          // 0: whole chain, 1: tail (waits for link), 2: head (sets link)
  int32_t link;          // index of the hand-on state and flag
  int32_t pad0, pad1;
};
struct WrapBuf {
  int32_t* ctl = nullptr;          // [0] pieces, [1] next piece to take
  const WrapPiece* piece = nullptr;  // [pieces], in any order
  const int32_t* order = nullptr;  // [pieces] piece indices by planned start time
  uint32_t* flag = nullptr;        // [grid] set once the state of link i is handed on
  float* state = nullptr;          // [grid][128][K] fp32: that state
};

struct ChunkParams {
  lin_state_pool_t pool;
  lin_prefill_args_t a;
  const int32_t* order;  // requests longest first (nullptr: batch order)
  int seg_mode;          // SegMode
  int seg_len;           // tokens per segment (multiple of 64)
  int seg_first;         // segment of blockIdx.x < H (modes 1 - 3)
  int seg_count;         // segments of the request (mode 4: blocks of offset runs first)
  float* seg_state_out;        // offset runs: fp32 state after the segment, [seg][H][V][K]
  float* seg_trans_out;        // transition runs: likewise
  const float* seg_state_in;   // mode 3: fp32 state before segment k >= 1 at index k - 1
  uint32_t* redo;              // KDA: bit r * H + h set when (request r, head h) left the
                               // factored decay range (cleared before the launch)
  // wrap-around schedule of a batch (wrap == nullptr: one CTA per (request, head))
  WrapBuf wrap;
};

// Longest-first order of a varlen batch: the sequential chunk chain of the
// longest request bounds the call, so its CTAs are dispatched first. One CTA
// bitonic-sorts (length, index) keys in shared memory.
constexpr int kOrderMax = 4096;

__global__ void __launch_bounds__(1024) order_kernel(const int32_t* __restrict__ cu, int batch,
                                                     int32_t* __restrict__ order) {
  __shared__ uint64_t key[kOrderMax];
  int n2 = 1;
  while (n2 < batch) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    if (i < batch) {
      const int64_t len = int64_t(cu[i + 1]) - int64_t(cu[i]);
      const uint32_t l = len < 0 ? 0u : (len > 0x7fffffff ? 0x7fffffffu : static_cast<uint32_t>(len));
      key[i] = (static_cast<uint64_t>(0x7fffffffu - l) << 32) | static_cast<uint32_t>(i);
    } else {
      key[i] = ~0ull;
    }
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ix = i ^ jj;
        if (ix > i) {
          const uint64_t a = key[i], b = key[ix];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            key[i] = b;
            key[ix] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < batch; i += blockDim.x) order[i] = static_cast<int32_t>(key[i] & 0xffffffffu);
}

// Exclusive prefix sum of v over a 1024-thread block, and the block's total
// (warp shuffles, then one warp over the 32 warp sums).
__device__ __forceinline__ int64_t block_exclusive_sum(int64_t v, int64_t* sums, int64_t& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int64_t z = sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, z, d);
      if (lane >= d) z += y;
    }
    sums[lane] = z;
  }
  __syncthreads();
  total = sums[31];
  const int64_t r = (w > 0 ? sums[w - 1] : 0) + x - v;
  __syncthreads();
  return r;
}
__device__ __forceinline__ int64_t block_max(int64_t v, int64_t* sums) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const int64_t y = __shfl_xor_sync(0xffffffffu, v, d);
    v = y > v ? y : v;
  }
  if ((threadIdx.x & 31) == 0) sums[threadIdx.x >> 5] = v;
  __syncthreads();
  int64_t m = sums[0];
  for (int i = 1; i < 32; ++i) m = sums[i] > m ? sums[i] : m;
  __syncthreads();
  return m;
}

// The wrap-around plan of a batch (one CTA): the chunk units n_r of every
// request (0 for an empty request and for one the prefill kernel skips or
// rejects: a negative slot, a slot past the pool, bad cu_seqlens or
// prefix_len, the kernel's own checks), T = max(longest chain,
// ceil(H sum n_r / grid)), the pieces with their planned start times, ordered
// by start time (a counting sort over the T start times, or a bitonic sort of
// (start, piece) keys when T is large), and cleared hand-on flags and counter.
constexpr int kWrapMaxPieces = 8192;
constexpr size_t kWrapPlanSmem = kWrapMaxPieces * sizeof(uint64_t) + kOrderMax * (sizeof(int64_t) + sizeof(int32_t));

__global__ void __launch_bounds__(1024) wrap_plan_kernel(const lin_prefill_args_t a, int H, int num_slots, int grid,
                                                         int32_t* ctl, WrapPiece* piece, int32_t* order,
                                                         uint32_t* flag) {
  extern __shared__ uint64_t wkey[];                                    // [kWrapMaxPieces] sort keys, or
  uint32_t* hist = reinterpret_cast<uint32_t*>(wkey);                  //   [kWrapMaxPieces] start counts
  int32_t* pstart = reinterpret_cast<int32_t*>(hist + kWrapMaxPieces);  //   and [kWrapMaxPieces] starts
  int64_t* first = reinterpret_cast<int64_t*>(wkey + kWrapMaxPieces);  // [batch] first unit of r
  int32_t* units = reinterpret_cast<int32_t*>(first + kOrderMax);      // [batch] n_r
  __shared__ int64_t sums[32];
  __shared__ int count;
  const int t = threadIdx.x, B = a.batch;
  const int per = (B + 1023) / 1024;  // requests t * per .. of this thread
  int64_t sum = 0, mx = 0;
  for (int i = 0; i < per; ++i) {
    const int r = t * per + i;
    if (r >= B) break;
    const int32_t sl = a.slot[r];
    const int64_t b = a.cu_seqlens[r], e = a.cu_seqlens[r + 1];
    const int32_t pf = a.prefix_len[r];
    const bool ok = sl >= 0 && sl < num_slots && b >= 0 && e >= b && e <= a.total_tokens && pf >= 0 && !(pf & 63);
    const int32_t n = ok ? static_cast<int32_t>((e - b + CH - 1) / CH) : 0;
    units[r] = n;
    sum += n;
    mx = n > mx ? n : mx;
  }
  if (t == 0) count = 0;
  int64_t all = 0;
  int64_t run = block_exclusive_sum(sum, sums, all);
  const int64_t maxn = block_max(mx, sums);
  for (int i = 0; i < per; ++i) {
    const int r = t * per + i;
    if (r >= B) break;
    first[r] = run * H;
    run += units[r];
  }
  const int64_t total = all * H;
  int64_t T = (total + grid - 1) / grid;
  if (T < maxn) T = maxn;
  if (T < 1) T = 1;
  const bool counting = T <= kWrapMaxPieces;
  if (counting)
    for (int i = t; i < T; i += 1024) hist[i] = 0u;
  __syncthreads();
  auto emit = [&](int r, int h, int c0, int c1, int mode, int link, int64_t start) {
    const int k = atomicAdd(&count, 1);
    piece[k] = WrapPiece{r, h, c0, c1, mode, link, 0, 0};
    if (counting) {
      pstart[k] = static_cast<int32_t>(start);
      atomicAdd(hist + start, 1u);
    } else {
      const uint64_t st = start < 0x7fffffff ? static_cast<uint64_t>(start) : 0x7fffffffull;
      wkey[k] = (st << 32) | static_cast<uint32_t>(k);
    }
  };
  for (int c = t; c < B * H; c += 1024) {
    const int r = c / H, h = c % H;
    const int64_t n = units[r];
    if (n == 0) {  // nothing to run: checks, and a cold empty request's zero state
      emit(r, h, 0, 0, 0, 0, 0);
      continue;
    }
    const int64_t cs = first[r] + h * n, ce = cs + n;
    const int64_t ms = cs / T, me = (ce - 1) / T;
    if (ms == me) {
      emit(r, h, 0, static_cast<int>(n), 0, 0, cs - ms * T);
    } else {  // crosses the start of range me: head there first, tail at the end of range ms
      const int x = static_cast<int>(ce - me * T);
      emit(r, h, 0, x, 2, static_cast<int>(me), 0);
      emit(r, h, x, static_cast<int>(n), 1, static_cast<int>(me), cs - ms * T);
    }
  }
  __syncthreads();
  const int N = count;
  if (counting) {
    // bucket offsets: thread t sums the counts of buckets t * bpt .. (bpt each)
    const int bpt = static_cast<int>((T + 1023) / 1024);
    uint32_t local = 0;
    for (int i = 0; i < bpt; ++i) {
      const int64_t q = int64_t(t) * bpt + i;
      if (q < T) local += hist[q];
    }
    int64_t dummy = 0;
    uint32_t off = static_cast<uint32_t>(block_exclusive_sum(local, sums, dummy));
    for (int i = 0; i < bpt; ++i) {
      const int64_t q = int64_t(t) * bpt + i;
      if (q < T) {
        const uint32_t c = hist[q];
        hist[q] = off;
        off += c;
      }
    }
    __syncthreads();
    for (int k = t; k < N; k += 1024) order[atomicAdd(hist + pstart[k], 1u)] = k;
  } else {
    int n2 = 2;
    while (n2 < N) n2 <<= 1;
    for (int i = N + t; i < n2; i += 1024) wkey[i] = ~0ull;
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        for (int i = t; i < n2; i += 1024) {
          const int ix = i ^ jj;
          if (ix > i) {
            const uint64_t x = wkey[i], y = wkey[ix];
            if ((x > y) == ((i & k) == 0)) {
              wkey[i] = y;
              wkey[ix] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = t; i < N; i += 1024) order[i] = static_cast<int32_t>(wkey[i] & 0xffffffffu);
  }
  for (int i = t; i < grid; i += 1024) flag[i] = 0u;
  if (t == 0) {
    ctl[0] = N;
    ctl[1] = 0;
  }
}

// Global channel of the head's channel cl in [0, 384): q, k and v parts of
// 128 each; a value part of VD < 128 channels takes the first VD (the rest are
// padding: see valid_channel).
template <int VD>
__device__ __forceinline__ int head_channel(int cl, int h, int H) {
  const int part = cl >> 7, c = cl & 127;
  return part < 2 ? part * H * DH + h * DH + c : 2 * H * DH + h * VD + c;
}
template <int VD>
__device__ __forceinline__ bool valid_channel(int cl) {
  return VD == DH || cl < 2 * DH + VD;
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 4 consecutive 16-bit values (cols c..c+3, c % 4 == 0) of row r of a row-panel buffer.
template <bool BF>
__device__ __forceinline__ void put4(uint32_t buf, int R, int r, int c, float a, float b, float cc,
                                     float d) {
  st_shared_v2(buf + umma::rp_offset(r, c, R), umma::pack2<BF>(a, b), umma::pack2<BF>(cc, d));
}
// 32 consecutive values (cols c0..c0+31) of row r.
template <bool BF>
__device__ __forceinline__ void put32(uint32_t buf, int R, int r, int c0, const float (&v)[32],
                                      float scale) {
#pragma unroll
  for (int m = 0; m < 4; ++m)
    st_shared_v4(buf + umma::rp_offset(r, c0 + 8 * m, R),
                 umma::pack2<BF>(scale * v[8 * m + 0], scale * v[8 * m + 1]),
                 umma::pack2<BF>(scale * v[8 * m + 2], scale * v[8 * m + 3]),
                 umma::pack2<BF>(scale * v[8 * m + 4], scale * v[8 * m + 5]),
                 umma::pack2<BF>(scale * v[8 * m + 6], scale * v[8 * m + 7]));
}

// 16 consecutive values (cols c0..c0+15) of row r.
template <bool BF>
__device__ __forceinline__ void put16(uint32_t buf, int R, int r, int c0, const float (&v)[16],
                                      float scale) {
#pragma unroll
  for (int m = 0; m < 2; ++m)
    st_shared_v4(buf + umma::rp_offset(r, c0 + 8 * m, R),
                 umma::pack2<BF>(scale * v[8 * m + 0], scale * v[8 * m + 1]),
                 umma::pack2<BF>(scale * v[8 * m + 2], scale * v[8 * m + 3]),
                 umma::pack2<BF>(scale * v[8 * m + 4], scale * v[8 * m + 5]),
                 umma::pack2<BF>(scale * v[8 * m + 6], scale * v[8 * m + 7]));
}

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane0, uint32_t col) {
  return base + (static_cast<uint32_t>(lane0) << 16) + col;
}

// Prefetch x rows [row0 - 3, row0 + 64) of the head's q | k | v channel blocks
// into L2 (tensor-map prefetch; the conv phase then reads them from L2).
template <int VD>
__device__ __forceinline__ void prefetch_x_tile(const CUtensorMap* tmap, int64_t row0, int h, int H) {
  const int y = static_cast<int>(row0) - 3;
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const int x = part < 2 ? part * H * DH + h * DH : 2 * H * DH + h * VD;
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y)
                 : "memory");
  }
}

// TMA bulk-group stores from shared memory.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* tmap, uint32_t src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tmap, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* tmap, uint32_t dst, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_but_one() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }
// orders this thread's completed bulk (async-proxy) writes before its later
// generic-proxy operations
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Hand-on flags of the wrap-around schedule: set with release semantics after
// the state they guard is written; waited for (one thread) with acquire
// semantics, giving up after about 4 s of device time.
__device__ __forceinline__ void flag_set(uint32_t* f) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(1u) : "memory");
}
__device__ __forceinline__ bool flag_wait(const uint32_t* f) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v) return true;
    if (global_ns() - t0 > 4000000000ull) return false;
    __nanosleep(256);
  }
  return false;
}

// hi / lo fp16 split of four values: hi = fp16(x), lo = fp16(x - hi).
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint32_t (&hi)[2],
                                       uint32_t (&lo)[2]) {
  const __half2 h0 = __floats2half2_rn(a, b), h1 = __floats2half2_rn(c, d);
  const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
  const __half2 l0 = __floats2half2_rn(a - f0.x, b - f0.y), l1 = __floats2half2_rn(c - f1.x, d - f1.y);
  hi[0] = *reinterpret_cast<const uint32_t*>(&h0);
  hi[1] = *reinterpret_cast<const uint32_t*>(&h1);
  lo[0] = *reinterpret_cast<const uint32_t*>(&l0);
  lo[1] = *reinterpret_cast<const uint32_t*>(&l1);
}

// hi / lo bf16 split of four values: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split4_bf(float a, float b, float c, float d, uint32_t (&hi)[2],
                                          uint32_t (&lo)[2]) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a, b), h1 = __floats2bfloat162_rn(c, d);
  const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
  const __nv_bfloat162 l0 = __floats2bfloat162_rn(a - f0.x, b - f0.y);
  const __nv_bfloat162 l1 = __floats2bfloat162_rn(c - f1.x, d - f1.y);
  hi[0] = *reinterpret_cast<const uint32_t*>(&h0);
  hi[1] = *reinterpret_cast<const uint32_t*>(&h1);
  lo[0] = *reinterpret_cast<const uint32_t*>(&l0);
  lo[1] = *reinterpret_cast<const uint32_t*>(&l1);
}

// Gate inputs of one chunk for this thread: KDA log-decay for TPW tokens x 4
// key channels, or the per-head scalar; beta for the TPW tokens.
template <bool KDA>
__device__ __forceinline__ void load_gates(const lin_prefill_args_t& a, int64_t row0, int n, int h,
                                           int H, int warp, int lane, float (&gk)[TPW][4],
                                           float (&bt)[TPW]) {
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = warp * TPW + i;
    const bool ok = t < n;
    const int64_t tok = row0 + t;
    if (KDA) {
      float4 v = ok ? *reinterpret_cast<const float4*>(a.g + (tok * H + h) * DH + lane * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      gk[i][0] = v.x; gk[i][1] = v.y; gk[i][2] = v.z; gk[i][3] = v.w;
    } else {
      gk[i][0] = ok ? a.g[tok * H + h] : 0.f;
      gk[i][1] = gk[i][2] = gk[i][3] = 0.f;
    }
    bt[i] = ok ? a.beta[tok * H + h] : 0.f;
  }
}

template <int ST>
__device__ __forceinline__ void store_row32(char* base, int v, int c0, const float (&x)[32]) {
  if (ST == LIN_BF16) {
    uint16_t* p = reinterpret_cast<uint16_t*>(base) + v * DH + c0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = static_cast<uint32_t>(f32_to_bf16_bits(x[8 * m + 2 * q])) |
               (static_cast<uint32_t>(f32_to_bf16_bits(x[8 * m + 2 * q + 1])) << 16);
      *reinterpret_cast<uint4*>(p + 8 * m) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    float* p = reinterpret_cast<float*>(base) + v * DH + c0;
#pragma unroll
    for (int m = 0; m < 8; ++m)
      *reinterpret_cast<float4*>(p + 4 * m) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
  }
}

// 16 values (cols c0..c0+15) of row r as fp16 high parts into `hi` and low
// parts into `lo`.
__device__ __forceinline__ void put16_split(uint32_t hi_buf, uint32_t lo_buf, int R, int r, int c0,
                                            const float (&v)[16], float scale) {
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    uint32_t h0[2], l0[2], h1[2], l1[2];
    split4(scale * v[8 * m + 0], scale * v[8 * m + 1], scale * v[8 * m + 2], scale * v[8 * m + 3], h0, l0);
    split4(scale * v[8 * m + 4], scale * v[8 * m + 5], scale * v[8 * m + 6], scale * v[8 * m + 7], h1, l1);
    const uint32_t off = umma::rp_offset(r, c0 + 8 * m, R);
    st_shared_v4(hi_buf + off, h0[0], h0[1], h1[0], h1[1]);
    st_shared_v4(lo_buf + off, l0[0], l0[1], l1[0], l1[1]);
  }
}

// SEG: the instantiation for the segmented launches, whose offset (after the
// first segment) and transition runs write no outputs and skip the q (and, in
// transition runs, the v) part of the conv and the output MMAs; the one-piece
// launch uses SEG = false, where every run has outputs.
// VD: value channels of a head, 128 or 64 (the Mamba2-style head of head dim
// 64 with 128 key channels). A 64-channel head runs on the same 128-row tiles
// with its value side padded by zeros: the padded conv channels have zero
// taps and window, so v, V', U, the state rows v >= 64 and their outputs stay
// zero; only the first VD rows are loaded and stored.
template <bool KDA, int ST, bool SEG, int VD>
__global__ void __launch_bounds__(NT, 1)
    chunked_prefill_kernel(const __grid_constant__ CUtensorMap tmap_x,
                           const __grid_constant__ CUtensorMap tmap_xt,
                           const __grid_constant__ CUtensorMap tmap_state,
                           const __grid_constant__ CUtensorMap tmap_out, const ChunkParams p) {
  // fp32 pools and GDN: fp16 operands with high / low splits on the products
  // that set the error, KDA's MMA1 in bf16 (split); KDA with a bf16 pool:
  // bf16 operands, single products (see the header).
  constexpr bool SPLIT = !KDA || ST == LIN_F32;
  constexpr bool BF = KDA && !SPLIT;  // operand type of every product but MMA1
  constexpr bool BF1 = KDA;           // operand type of MMA1 ([K_l; Q_l] K_r^T)
  extern __shared__ uint8_t dsm[];
  __shared__ uint64_t bar_mma;
  __shared__ uint64_t bar_v;  // MMA-V' of the chunk (and MMA4a) completed
  __shared__ uint64_t bar_x;  // x tile of the next chunk landed
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int range_sh;  // KDA: a key channel's decay left the factored range
  __shared__ int piece_sh[6];  // wrap-around schedule: the piece this CTA took

  const lin_state_pool_t& pool = p.pool;
  const lin_prefill_args_t& a = p.a;
  const int H = pool.num_heads;
  int seg_mode = p.seg_mode;
  int seg = 0;
  if (seg_mode == kSegOffsetAndTransition) {
    const int nb1 = (p.seg_count - 1) * H;  // offset runs of segments 0 .. n-2 first
    if (static_cast<int>(blockIdx.x) < nb1) {
      seg_mode = kSegOffset;
      seg = static_cast<int>(blockIdx.x) / H;
    } else {
      seg_mode = kSegTransition;
      seg = 1 + (static_cast<int>(blockIdx.x) - nb1) / H;
    }
  } else if (seg_mode) {
    seg = p.seg_first + static_cast<int>(blockIdx.x) / H;
  }
  int r, h, c0 = 0, c1 = -1, pmode = 0, plink = 0;
  if (p.wrap.ctl) {
    // the next piece of the wrap-around schedule, in planned start order
    if (threadIdx.x == 0) {
      const int k = atomicAdd(p.wrap.ctl + 1, 1);
      piece_sh[0] = -1;
      if (k < __ldcg(p.wrap.ctl)) {
        const WrapPiece e = p.wrap.piece[__ldcg(p.wrap.order + k)];
        piece_sh[0] = e.r;
        piece_sh[1] = e.h;
        piece_sh[2] = e.c0;
        piece_sh[3] = e.c1;
        piece_sh[4] = e.mode;
        piece_sh[5] = e.link;
      }
    }
    __syncthreads();
    r = piece_sh[0];
    if (r < 0) return;
    h = piece_sh[1];
    c0 = piece_sh[2];
    c1 = piece_sh[3];
    pmode = piece_sh[4];
    plink = piece_sh[5];
  } else {
    r = seg_mode ? 0 : (p.order ? p.order[blockIdx.x / H] : blockIdx.x / H);
    h = blockIdx.x % H;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, slice = warp >> 2;  // four warps share each lane quarter
  const int vrow = quarter * 32 + lane;             // TMEM lane owned in the epilogues
  const bool rep = (h == 0 && tid == 0);

  // ---- request checks (uniform over the CTA) ----
  const int slot = a.slot[r];
  if (slot < 0) return;
  if (slot >= pool.num_slots) {
    if (rep) report(a.status, LIN_ST_BAD_SLOT);
    return;
  }
  const int64_t bos_r = a.cu_seqlens[r], eos = a.cu_seqlens[r + 1];
  if (bos_r < 0 || eos < bos_r || eos > a.total_tokens) {
    if (rep && seg == 0) report(a.status, LIN_ST_BAD_SEQLEN);
    return;
  }
  const int P_r = a.prefix_len[r];
  if (P_r < 0 || (P_r & 63)) {
    if (rep && seg == 0) report(a.status, LIN_ST_BAD_PREFIX);
    return;
  }
  // the tokens this CTA runs: the request, one segment of it, or one piece
  // (chunks c0 .. c1 - 1) of it under the wrap-around schedule
  int64_t bos = bos_r, eos_c = eos;
  if (seg_mode) {
    bos = bos_r + int64_t(seg) * p.seg_len;
    if (bos >= eos) return;
    eos_c = (eos - bos) < p.seg_len ? eos : bos + p.seg_len;
  } else if (c1 >= 0) {
    bos = bos_r + int64_t(c0) * CH;
    const int64_t e1 = bos_r + int64_t(c1) * CH;
    eos_c = e1 < eos ? e1 : eos;
  }
  const int P = P_r + static_cast<int>(bos - bos_r);  // tokens before bos in absolute positions
  const bool seg_last = (eos_c == eos);               // this CTA ends the request
  const bool outputs_on =
      !SEG || seg_mode == kSegOff || seg_mode == kSegFinal || (seg_mode == kSegOffset && seg == 0);
  // the fp32 state after the last chunk also goes to a workspace: a segment's
  // offset or transition run, a wrap-around head piece
  const bool state_to_ws = seg_mode == kSegOffset || seg_mode == kSegTransition || pmode == 2;
  int t0 = 0, ntr = 0;
  if (outputs_on && a.track_stride > 0 && a.cu_track) {
    t0 = a.cu_track[r];
    ntr = a.cu_track[r + 1] - t0;
    for (int i = 0; i < ntr; ++i) {
      const int t = a.track_slots[t0 + i];
      if (t >= pool.num_slots) {
        if (rep && seg == 0) report(a.status, LIN_ST_BAD_SLOT);
        return;
      }
      if (t == slot) {
        if (rep && seg == 0) report(a.status, LIN_ST_TRACK_ALIAS);
        return;
      }
    }
  }
  // initial state: 0 zeros, 1 the slot, 2 identity, 3 an fp32 workspace state
  // (the segment's, or the one a wrap-around head piece handed on)
  if (KDA && seg_mode == kSegFinal && p.redo) {
    // an offset or transition run of this (request, head) left the factored
    // decay range: the token-by-token rerun redoes it from the slot
    const int idx = r * H + h;
    if ((p.redo[idx >> 5] >> (idx & 31)) & 1u) return;
  }
  const bool warm_r = a.has_initial_state[r] != 0;
  int init_kind = warm_r ? 1 : 0;
  if (seg > 0) init_kind = seg_mode == kSegOffset ? 0 : (seg_mode == kSegTransition ? 2 : 3);
  if (pmode == 1) init_kind = 3;
  const bool warm = init_kind == 1;
  const bool zero_v = SEG && seg_mode == kSegTransition;  // transition runs take no value input
  const int L = static_cast<int>(eos_c - bos);
  const int nch = (L + CH - 1) / CH;
  constexpr int ES = ST == LIN_BF16 ? 2 : 4;
  const int64_t head_bytes = int64_t(VD) * DH * ES;
  char* slot_t = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride +
                 slot * pool.temporal_slot_stride + h * head_bytes;
  char* slot_c = static_cast<char*>(pool.conv) + a.layer * pool.conv_layer_stride +
                 slot * pool.conv_slot_stride;
  const uint32_t raw = umma::smem_u32(dsm);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sm = dsm + (sb - raw);
  float* WC = reinterpret_cast<float*>(sm + OFF_WC);
  float* HALO = reinterpret_cast<float*>(sm + OFF_HALO);
  float* WTOT = reinterpret_cast<float*>(sm + OFF_WTOT);
  float* SBETA = reinterpret_cast<float*>(sm + OFF_SBETA);
  float* SB = reinterpret_cast<float*>(sm + OFF_SB);
  float* GLAST = reinterpret_cast<float*>(sm + OFF_GLAST);
  float* CF = reinterpret_cast<float*>(sm + OFF_CF);
  float* WIN = reinterpret_cast<float*>(sm + OFF_WIN);
  float* AX = reinterpret_cast<float*>(sm + OFF_AX);
  float* XD = reinterpret_cast<float*>(sm + OFF_XD);
  float* YB = reinterpret_cast<float*>(sm + OFF_YB);
  float* ZB = reinterpret_cast<float*>(sm + OFF_ZB);

  if (tid == 0) prefetch_x_tile<VD>(&tmap_x, bos, h, H);
  for (int i = tid; i < 384 * 4; i += NT)
    WC[(i & 3) * 384 + (i >> 2)] =
        valid_channel<VD>(i >> 2)
            ? load_elem(a.conv_w, int64_t(head_channel<VD>(i >> 2, h, H)) * 4 + (i & 3), a.io_dtype)
            : 0.f;
  for (int i = tid; i < 3 * 384; i += NT) {
    const int rr = i / 384, cl = i % 384;
    if (!valid_channel<VD>(cl))
      HALO[i] = 0.f;
    else if (bos > bos_r)  // the 3 inputs before the segment or piece
      HALO[i] = load_elem(a.x, (bos - 3 + rr) * int64_t(pool.conv_channels) + head_channel<VD>(cl, h, H), LIN_BF16);
    else
      HALO[i] = warm ? load_elem(slot_c, int64_t(head_channel<VD>(cl, h, H)) * 3 + rr, pool.conv_dtype) : 0.f;
  }

  if (nch == 0) {
    // No tokens: the slot keeps its state; a cold start leaves zeros in it.
    if (!warm) {
      for (int i = tid; i < VD * DH; i += NT) store_elem(slot_t, i, ST, 0.f);
      for (int i = tid; i < 3 * 384; i += NT)
        if (valid_channel<VD>(i / 3))
          store_elem(slot_c, int64_t(head_channel<VD>(i / 3, h, H)) * 3 + (i % 3), pool.conv_dtype, 0.f);
    }
    return;
  }

  if (tid == 0) {
    umma::mbar_init(&bar_mma, 1);
    umma::mbar_init(&bar_v, 1);
    umma::mbar_init(&bar_x, 1);
    umma::mbar_fence_init();
    abort_sh = 0;
    range_sh = 0;
  }
  if (warp == 0) umma::tmem_alloc(&tmem_base_sh, TMEM_COLS);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = tmem_base_sh;
  // Shared-memory descriptors of sb + off differ from those of sb only in the
  // start-address field, (addr >> 4) in the low 14 bits (addresses stay below
  // 2^18), so the issuing thread adds a constant instead of rebuilding them.
  const uint64_t dk0 = umma::smem_desc(sb, 16, 1024);
  const uint64_t dm64 = umma::smem_desc(sb, 64 * 128, 1024);
  const uint64_t dm128 = umma::smem_desc(sb, 128 * 128, 1024);
  // K-major operand at sb + off with `rows` rows: K-step k0 (as umma::desc_kmajor)
  auto kdesc = [&](uint32_t off, int rows, int k0) -> uint64_t {
    return dk0 + ((off + static_cast<uint32_t>(k0 >> 6) * rows * 128 + static_cast<uint32_t>(k0 & 63) * 2) >> 4);
  };
  // MN-major operand at sb + off with `krows` K rows (as umma::desc_mnmajor)
  auto mdesc = [&](uint32_t off, int krows, int k0) -> uint64_t {
    return (krows == 64 ? dm64 : dm128) + ((off + static_cast<uint32_t>(k0) * 128) >> 4);
  };

  // a wrap-around tail piece starts from the state its head piece hands on;
  // it runs nothing when that wait gives up or when the head piece left the
  // KDA factored range (the token-by-token rerun redoes the pair)
  int nrun = nch;
  if (pmode == 1) {
    if (tid == 0 && !flag_wait(p.wrap.flag + plink)) {
      abort_sh = 1;
      report(a.status, LIN_ST_TIMEOUT);
    }
    __syncthreads();
    if (abort_sh) nrun = 0;
    if (KDA && p.redo) {
      const int idx = r * H + h;
      if ((__ldcg(p.redo + (idx >> 5)) >> (idx & 31)) & 1u) nrun = 0;
    }
  }

  // ---- initial state: fp32 into TMEM, 16-bit operand copy into shared memory
  {
    float s[32];
    const int cc = slice * 32;
    if (warm && vrow >= VD) {
#pragma unroll
      for (int m = 0; m < 32; ++m) s[m] = 0.f;  // padding rows of a 64-channel value side
    } else if (warm) {
      if (ST == LIN_BF16) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(slot_t) + vrow * DH + cc;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4 u = *reinterpret_cast<const uint4*>(src + 8 * m);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            s[8 * m + 2 * q] = __uint_as_float(w[q] << 16);
            s[8 * m + 2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
          }
        }
      } else {
        const float* src = reinterpret_cast<const float*>(slot_t) + vrow * DH + cc;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          float4 u = *reinterpret_cast<const float4*>(src + 4 * m);
          s[4 * m] = u.x; s[4 * m + 1] = u.y; s[4 * m + 2] = u.z; s[4 * m + 3] = u.w;
        }
      }
    } else if (init_kind == 3) {
      const float* src = (pmode == 1 ? p.wrap.state + int64_t(plink) * DH * DH
                                     : p.seg_state_in + (int64_t(seg - 1) * H + h) * DH * DH) +
                         int64_t(vrow) * DH + cc;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float4 u = __ldcg(reinterpret_cast<const float4*>(src + 4 * m));
        s[4 * m] = u.x; s[4 * m + 1] = u.y; s[4 * m + 2] = u.z; s[4 * m + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int m = 0; m < 32; ++m) s[m] = (init_kind == 2 && cc + m == vrow) ? 1.f : 0.f;
    }
    umma::tmem_st32(tmem_addr(tm, quarter * 32, COL_S + cc), s);
    put32<BF>(sb + OFF_SOP, 128, vrow, cc, s, 1.f);
  }
  umma::fence_smem_to_async();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();

  float gk[TPW][4], bt[TPW];
  load_gates<KDA>(a, bos, L < CH ? L : CH, h, H, warp, lane, gk, bt);

  uint32_t ph_mma = 0;
  // boundaries snapshotted before bos by earlier segments or pieces of this request
  int snap = (ntr > 0 && bos > bos_r) ? static_cast<int>(P / a.track_stride - P_r / a.track_stride) : 0;
  // Segments run in parallel, so two of them may map boundaries onto the same
  // entry of a cycled track list: there only the snapshots that survive in
  // token order (the request's last ntr) are written.
  const int64_t snap_total =
      ntr > 0 ? (int64_t(P_r) + (eos - bos_r)) / a.track_stride - int64_t(P_r) / a.track_stride : 0;
  const bool silu_on = a.flags & LIN_CONV_SILU;
  const bool l2_on = a.flags & LIN_QK_L2NORM;
  const bool additive = a.flags & LIN_UPDATE_ADDITIVE;  // uniform over the CTA

  // Waits for the MMAs committed so far (thread 0 polls, everyone syncs).
  auto wait_mma = [&]() -> bool {
    if (tid == 0) {
      if (!umma::mbar_wait(&bar_mma, ph_mma, kWaitTries)) {
        abort_sh = 1;
        report(a.status, LIN_ST_TIMEOUT);
      }
    }
    ph_mma ^= 1;
    __syncthreads();
    umma::fence_after_sync();
    return abort_sh == 0;
  };

  uint32_t ph_v = 0;
  // The x tile of the chunk starting at token r0 (thread 0): one TMA load per
  // q | k | v part, completing on bar_x.
  int x_issued = 0;
  auto issue_x_tile = [&](int64_t r0) {
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar_x));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(3 * CH * DH * 2)
                 : "memory");
#pragma unroll
    for (int part = 0; part < 3; ++part)
      tma_load_2d(&tmap_xt, sb + OFF_XT + part * (CH * DH * 2),
                  part < 2 ? part * H * DH + h * DH : 2 * H * DH + h * VD, static_cast<int>(r0), b);
    ++x_issued;
  };
  if (tid == 0 && nrun > 0) issue_x_tile(bos);

  const int tfirst = warp * TPW;
  for (int j = 0; j < nrun; ++j) {
    const int n = (L - j * CH) < CH ? (L - j * CH) : CH;
    const int64_t row0 = bos + int64_t(j) * CH;

    // this chunk's x tile must have landed
    if (tid == 0) {
      if (!umma::mbar_wait(&bar_x, static_cast<uint32_t>(j & 1), kWaitTries)) {
        abort_sh = 1;
        report(a.status, LIN_ST_TIMEOUT);
      }
    }
    __syncthreads();
    if (abort_sh) break;

    // ---- x rows of this warp's tokens from the tile (8 bytes = 4 channels per
    // lane and part); rows before the chunk come from the previous window, rows
    // past its end are zero
    uint2 xr[TPW + 3][3];
#pragma unroll
    for (int m = 0; m < TPW + 3; ++m) {
      const int rel = tfirst - 3 + m;  // row relative to the chunk start
#pragma unroll
      for (int part = 0; part < 3; ++part)
        xr[m][part] = (rel >= 0 && rel < n)
                          ? *reinterpret_cast<const uint2*>(sm + OFF_XT + part * (CH * DH * 2) + rel * (DH * 2) + lane * 8)
                          : make_uint2(0u, 0u);
    }
    // the window before this chunk (its last 3 inputs): the initial conv state
    // for the first chunk, else the previous chunk's window
    const float* wprev = j == 0 ? HALO : WIN + ((j - 1) & 1) * 1152;

    // the chunk's last 3 inputs, for the next chunk and for a conv-state
    // snapshot or the final write-back: each row is written by the warp that
    // holds it (rows before the chunk by warp 0)
    {
      float* wcur = WIN + (j & 1) * 1152;
#pragma unroll
      for (int m = 0; m < TPW + 3; ++m) {
        const int rel = tfirst - 3 + m;
        if (rel >= n - 3 && rel < n && (rel >= tfirst || (warp == 0 && rel < 0))) {
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            float4 wv;
            if (rel < 0) {
              wv = *reinterpret_cast<const float4*>(wprev + (rel + 3) * 384 + part * 128 + lane * 4);
            } else {
              const uint2 u2 = xr[m][part];
              wv = make_float4(__uint_as_float(u2.x << 16), __uint_as_float(u2.x & 0xffff0000u),
                               __uint_as_float(u2.y << 16), __uint_as_float(u2.y & 0xffff0000u));
            }
            *reinterpret_cast<float4*>(wcur + (rel - n + 3) * 384 + part * 128 + lane * 4) = wv;
          }
        }
      }
    }


    // ---- gates: in-chunk inclusive sums b_t (rows past n carry log-decay 0)
    float cs[TPW][4];
    {
      float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          run[e] += gk[i][e];
          cs[i][e] = run[e];
        }
      if (KDA) {
        *reinterpret_cast<float4*>(WTOT + warp * DH + lane * 4) = make_float4(run[0], run[1], run[2], run[3]);
      } else if (lane == 0) {
        WTOT[warp] = run[0];
      }
    }
    __syncthreads();
    float bref[4], blast[4];
    {
      float pre[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bref[e] = 0.f;
        blast[e] = 0.f;
      }
#pragma unroll
      for (int w = 0; w < NW; ++w) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float tw = KDA ? WTOT[w * DH + lane * 4 + e] : WTOT[w];
          if (w < warp) pre[e] += tw;
          if (w < NW / 2) bref[e] += tw;
          blast[e] += tw;
        }
      }
#pragma unroll
      for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) cs[i][e] += pre[e];
      if (warp == 0) {
        if (KDA) {
#pragma unroll
          for (int e = 0; e < 4; ++e) GLAST[lane * 4 + e] = __expf(blast[e]);
        } else if (lane == 0) {
          GLAST[0] = __expf(blast[0]);
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          SBETA[warp * TPW + i] = bt[i];
          SB[warp * TPW + i] = cs[i][0];
        }
      }
    }

    // ---- conv, activation, q/k normalisation, operand rows
    {
      // xr[m]: window row m (chunk row tfirst - 3 + m) of the tile, channels
      // lane*4 .. lane*4+3 per part; rows before the chunk (warp 0, m < 3) hold
      // zeros there and their terms are added from the previous window below
      // part-major: the taps of one part are loaded once and applied to all
      // of this warp's tokens; q and k get their per-token norms
      float yq[TPW][4], yk[TPW][4], yv[TPW][4], rq[TPW], rk[TPW];
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        // runs without outputs need no q; transition runs take no values
        if ((part == 0 && !outputs_on) || (part == 2 && zero_v)) {
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (part == 0) yq[i][e] = 0.f;
              else yv[i][e] = 0.f;
            }
            if (part == 0) rq[i] = 0.f;
          }
          continue;
        }
        float4 w4[4];
#pragma unroll
        for (int tap = 0; tap < 4; ++tap)
          w4[tap] = *reinterpret_cast<const float4*>(WC + tap * 384 + part * 128 + lane * 4);
        // the taps on channel pairs (lane*4 + 0, 1) and (lane*4 + 2, 3), two
        // lanes of fp32 arithmetic per instruction; the x tile's bf16 pairs
        // unpack straight into such pairs
        float ypre[TPW][4];
        {
          uint64_t wp[4][2];
#pragma unroll
          for (int tap = 0; tap < 4; ++tap) {
            wp[tap][0] = f2pack(w4[tap].x, w4[tap].y);
            wp[tap][1] = f2pack(w4[tap].z, w4[tap].w);
          }
          auto xp = [&](int m, int hp) -> uint64_t {
            const uint32_t w = hp ? xr[m][part].y : xr[m][part].x;
            return f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
          };
#pragma unroll
          for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              uint64_t y = fmul2(wp[0][hp], xp(i, hp));
              y = ffma2(wp[1][hp], xp(i + 1, hp), y);
              y = ffma2(wp[2][hp], xp(i + 2, hp), y);
              y = ffma2(wp[3][hp], xp(i + 3, hp), y);
              float lo, hi;
              asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(y));
              ypre[i][2 * hp] = lo;
              ypre[i][2 * hp + 1] = hi;
            }
        }
        if (warp == 0) {
          // tokens 0..2: the taps on the 3 rows before the chunk
          const float* hp = wprev + part * 128 + lane * 4;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float w0 = e == 0 ? w4[0].x : e == 1 ? w4[0].y : e == 2 ? w4[0].z : w4[0].w;
            const float w1 = e == 0 ? w4[1].x : e == 1 ? w4[1].y : e == 2 ? w4[1].z : w4[1].w;
            const float w2 = e == 0 ? w4[2].x : e == 1 ? w4[2].y : e == 2 ? w4[2].z : w4[2].w;
            const float h0 = hp[e], h1 = hp[384 + e], h2 = hp[768 + e];
            ypre[0][e] += w0 * h0 + w1 * h1 + w2 * h2;
            ypre[1][e] += w0 * h1 + w1 * h2;
            ypre[2][e] += w0 * h2;
          }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float yy = ypre[i][e];
            // SiLU from one tanh.approx (relative error 2^-11, below what the
            // fp16 operand splits leave in the results)
            yy = silu_on ? silu_tanh(yy) : yy;
            ss += yy * yy;
            if (part == 0) yq[i][e] = yy;
            else if (part == 1) yk[i][e] = yy;
            else yv[i][e] = yy;
          }
          if (part < 2) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float rr = l2_on ? rsqrtf(ss + 1e-6f) : 1.f;
            if (part == 0) rq[i] = rr * a.q_scale;
            else rk[i] = rr;
          }
        }
      }
      // the previous chunk's TMA stores must have read their staging tiles
      // before the operand rows go over them; those reads ran behind the conv
      if (tid == kStoreTid) bulk_wait_read();
      __syncthreads();
      bool range_bad = false;
      // KDA: exp(b_last - b) = exp(b_last - b_ref) exp(b_ref - b), the first
      // factor per channel for the chunk; both stay inside e^+-80 (the range
      // check below), so the product is the exponential up to one rounding
      float ecl[4], ebr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ecl[e] = KDA ? __expf(blast[e] - bref[e]) : 1.f;
        ebr[e] = (KDA && !SEG) ? __expf(bref[e]) : 1.f;
      }
      // KDA: exp(b) = exp(b - b_ref) exp(b_ref), one exponential fewer per
      // element, unless exp(b_ref) underflows for some lane of the warp (not in
      // the segmented instance, where the extra registers spill)
      const bool eh_prod = KDA && !SEG &&
                           __all_sync(0xffffffffu, ebr[0] > 0.f && ebr[1] > 0.f && ebr[2] > 0.f && ebr[3] > 0.f);
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        const int t = tfirst + i;
        const bool ok = t < n;
        float kn[4], qn[4], vv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kn[e] = ok ? yk[i][e] * rk[i] : 0.f;
          qn[e] = ok ? yq[i][e] * rq[i] : 0.f;
          vv[e] = (ok && !zero_v) ? yv[i][e] : 0.f;
        }
        float eL[4], eR[4], eH[4], eT[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ee = KDA ? e : 0;
          const float b = cs[i][ee];
          eL[e] = KDA ? __expf(b - bref[ee]) : 1.f;
          if (eh_prod)
            eH[e] = eL[e] * ebr[e];
          else
            eH[e] = __expf(b);
          eR[e] = KDA ? __expf(bref[ee] - b) : 1.f;
          eT[e] = KDA ? ecl[e] * eR[e] : __expf(blast[ee] - b);
          // the factored decay must stay inside fp32 range (else the pair is rerun)
          if (KDA && ok && fabsf(b - bref[ee]) > 80.f) range_bad = true;
        }
        const int c = lane * 4;
        if (SPLIT && KDA) {
          // MMA1 operands in bf16 (hi / lo): K_l, Q_l and K_r
          uint32_t hi[2], lo[2];
          split4_bf(kn[0] * eL[0], kn[1] * eL[1], kn[2] * eL[2], kn[3] * eL[3], hi, lo);
          st_shared_v2(sb + OFF_KQ + umma::rp_offset(t, c, 128), hi[0], hi[1]);
          st_shared_v2(sb + OFF_KQL + umma::rp_offset(t, c, 128), lo[0], lo[1]);
          split4_bf(qn[0] * eL[0], qn[1] * eL[1], qn[2] * eL[2], qn[3] * eL[3], hi, lo);
          st_shared_v2(sb + OFF_KQ + umma::rp_offset(CH + t, c, 128), hi[0], hi[1]);
          st_shared_v2(sb + OFF_KQL + umma::rp_offset(CH + t, c, 128), lo[0], lo[1]);
          split4_bf(kn[0] * eR[0], kn[1] * eR[1], kn[2] * eR[2], kn[3] * eR[3], hi, lo);
          st_shared_v2(sb + OFF_KR + umma::rp_offset(t, c, 64), hi[0], hi[1]);
          st_shared_v2(sb + OFF_KRL + umma::rp_offset(t, c, 64), lo[0], lo[1]);
        } else {
          put4<BF1>(sb + OFF_KQ, 128, t, c, kn[0] * eL[0], kn[1] * eL[1], kn[2] * eL[2], kn[3] * eL[3]);
          put4<BF1>(sb + OFF_KQ, 128, CH + t, c, qn[0] * eL[0], qn[1] * eL[1], qn[2] * eL[2], qn[3] * eL[3]);
          if (KDA)
            put4<BF1>(sb + OFF_KR, 64, t, c, kn[0] * eR[0], kn[1] * eR[1], kn[2] * eR[2], kn[3] * eR[3]);
        }
        put4<BF>(sb + OFF_KQH, 128, t, c, -kn[0] * eH[0], -kn[1] * eH[1], -kn[2] * eH[2], -kn[3] * eH[3]);
        put4<BF>(sb + OFF_KQH, 128, CH + t, c, qn[0] * eH[0], qn[1] * eH[1], qn[2] * eH[2], qn[3] * eH[3]);
        put4<BF>(sb + OFF_VV, 64, t, c, vv[0], vv[1], vv[2], vv[3]);
        put4<BF>(sb + OFF_KT, 64, t, c, kn[0] * eT[0], kn[1] * eT[1], kn[2] * eT[2], kn[3] * eT[3]);
      }
      if (KDA && __any_sync(0xffffffffu, range_bad) && lane == 0) range_sh = 1;
    }
    umma::fence_smem_to_async();
    __syncthreads();
    if (KDA && range_sh) {
      // The factored decay of this chunk leaves fp32 range: stop before any
      // of its results (or the final state) is stored, and flag the pair for
      // the token-by-token rerun queued behind this launch. Every MMA and x
      // tile issued so far has completed; the teardown drains the stores.
      if (tid == 0 && p.redo) {
        const int idx = r * H + h;
        atomicOr(p.redo + (idx >> 5), 1u << (idx & 31));
      }
      break;
    }

    // ---- MMA1: [A'; P'] = [K_l; Q_l] K_r^T; prefetch the next chunk's x rows
    if (tid == 0) {
      if (j + 1 < nch) prefetch_x_tile<VD>(&tmap_x, row0 + CH, h, H);
      umma::fence_after_sync();
      constexpr uint32_t id1 = umma::idesc_f16(128, 64, BF1, false, false);
#pragma unroll
      for (int k0 = 0; k0 < DH; k0 += 16) {
        const uint64_t ah = kdesc(OFF_KQ, 128, k0);
        if (SPLIT && KDA) {
          const uint64_t al = kdesc(OFF_KQL, 128, k0);
          const uint64_t bh = kdesc(OFF_KR, 64, k0);
          umma::mma_f16(tm + COL_R1, ah, bh, id1, k0 > 0);
          umma::mma_f16(tm + COL_R1, ah, kdesc(OFF_KRL, 64, k0), id1, 1);
          umma::mma_f16(tm + COL_R1, al, bh, id1, 1);
        } else if (KDA) {
          umma::mma_f16(tm + COL_R1, ah, kdesc(OFF_KR, 64, k0), id1, k0 > 0);
        } else {
          umma::mma_f16(tm + COL_R1, ah, ah, id1, k0 > 0);  // B: rows 0..63 (K) of the same panels
        }
      }
      umma::mma_commit(&bar_mma);
      // the additive form has no MMAV: MMA4a alone, O^T = S0 Qhat^T (RO), B
      // the Qhat rows of the [-Khat; Qhat] panels; it completes before MMA2's
      // commit fires
      if (outputs_on && additive) {
        constexpr uint32_t id4 = umma::idesc_f16(128, 64, BF, false, false);
#pragma unroll
        for (int k0 = 0; k0 < DH; k0 += 16)
          umma::mma_f16(tm + COL_RO, kdesc(OFF_SOP, 128, k0),
                        kdesc(OFF_KQH + CH * 128, 128, k0), id4, k0 > 0);
      }
    }
    if (!KDA && tid >= 32 && tid < 96) {
      // GDN: the in-chunk decay exp(b_t - b_i) factors as exp(b_t - b_s) exp(b_s - b_i),
      // s the first column of i's 16-wide slice; the second factor per column here
      // (-1 where it would leave fp32 range: those columns take the direct exponential)
      const int i = tid - 32;
      const float d = SB[i & ~15] - SB[i];
      CF[i] = d <= 80.f ? __expf(d) : -1.f;
    }
    if (!additive) {
      // V^T (lanes v, columns t) into tensor memory: the accumulator MMAV
      // starts from; zeros where MMA4a accumulates (the two run as one product)
      float v16[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint16_t u = *reinterpret_cast<const uint16_t*>(sm + OFF_VV + umma::rp_offset(slice * 16 + k, vrow, 64));
        v16[k] = BF ? __uint_as_float(static_cast<uint32_t>(u) << 16) : __half2float(__ushort_as_half(u));
      }
      umma::tmem_st16(tmem_addr(tm, quarter * 32, COL_R2 + slice * 16), v16);
      if (outputs_on) {
#pragma unroll
        for (int k = 0; k < 16; ++k) v16[k] = 0.f;
        umma::tmem_st16(tmem_addr(tm, quarter * 32, COL_RO + slice * 16), v16);
      }
      umma::fence_before_sync();
    }
    if (!additive) {
      __syncthreads();  // V^T is in tensor memory
      if (tid == 0) {
        // MMAV and MMA4a as one product S0 [-Khat; Qhat]^T into the adjacent
        // columns R2 | RO: V'^T = V^T - S0 Khat^T (U = T V' below makes the
        // delta-rule correction U = U' - W S0^T without forming W) and
        // O^T = S0 Qhat^T; without outputs, MMAV alone
        umma::fence_after_sync();
        constexpr uint32_t idvo = umma::idesc_f16(128, 128, BF, false, false);
        constexpr uint32_t idv = umma::idesc_f16(128, 64, BF, false, false);
#pragma unroll
        for (int k0 = 0; k0 < DH; k0 += 16)
          umma::mma_f16(tm + COL_R2, kdesc(OFF_SOP, 128, k0),
                        kdesc(OFF_KQH, 128, k0), outputs_on ? idvo : idv, 1);
        umma::mma_commit(&bar_v);
      }
    }
    if (!wait_mma()) break;

    // ---- A (fp32, for the solve) and P (operand) from [A'; P']
    {
      float v[16];
      umma::tmem_ld16(tmem_addr(tm, quarter * 32, COL_R1 + slice * 16), v);
      const int s0 = slice * 16;
      if (quarter < 2) {
        const int t = vrow;
        const float bet = SBETA[t];
        const float bt_ = SB[t];
        const float rfac = (KDA || s0 > t) ? 1.f : __expf(bt_ - SB[s0]);
        // GDN: every lane of the warp reads the same 16 column factors, so the
        // rare fallback to the direct exponential is a uniform branch
        float cfv[16];
        bool fast = true;
        if (!KDA) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 c4 = *reinterpret_cast<const float4*>(CF + s0 + 4 * k4);
            cfv[4 * k4] = c4.x; cfv[4 * k4 + 1] = c4.y; cfv[4 * k4 + 2] = c4.z; cfv[4 * k4 + 3] = c4.w;
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) fast = fast && cfv[k] >= 0.f;
        }
        if (KDA || fast) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = s0 + k;
            const float dec = KDA ? 1.f : rfac * cfv[k];
            AX[t * AXS + i] = (i < t) ? bet * v[k] * dec : 0.f;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = s0 + k;
            const float dec = cfv[k] >= 0.f ? rfac * cfv[k] : __expf(bt_ - SB[i < t ? i : t]);
            AX[t * AXS + i] = (i < t) ? bet * v[k] * dec : 0.f;
          }
        }
      } else {
        const int t = vrow - 64;
        const float bt_ = SB[t];
        const float rfac = (KDA || s0 > t) ? 1.f : __expf(bt_ - SB[s0]);
        float pv[16];
        float cfv[16];
        bool fast = true;
        if (!KDA) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 c4 = *reinterpret_cast<const float4*>(CF + s0 + 4 * k4);
            cfv[4 * k4] = c4.x; cfv[4 * k4 + 1] = c4.y; cfv[4 * k4 + 2] = c4.z; cfv[4 * k4 + 3] = c4.w;
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) fast = fast && cfv[k] >= 0.f;
        }
        if (KDA || fast) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = s0 + k;
            const float dec = KDA ? 1.f : rfac * cfv[k];
            pv[k] = (i <= t) ? v[k] * dec : 0.f;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = s0 + k;
            const float dec = cfv[k] >= 0.f ? rfac * cfv[k] : __expf(bt_ - SB[i <= t ? i : t]);
            pv[k] = (i <= t) ? v[k] * dec : 0.f;
          }
        }
        if (SPLIT)
          put16_split(sb + OFF_PP, sb + OFF_PPL, 64, t, slice * 16, pv, 1.f);
        else
          put16<BF>(sb + OFF_PP, 64, t, slice * 16, pv, 1.f);
      }
    }
    // ---- T = (I + A)^-1 Diag(beta). X = (I + A)^-1 (unit lower triangular) is
    // built in three levels: its four 16 x 16 diagonal blocks X_aa by forward
    // substitution (one thread per column); the two 32 x 32 diagonal blocks,
    // X_10 = -X_11 (A_10 X_00) and X_32 = -X_33 (A_32 X_22); then the lower-left
    // 32 x 32 quarter X_BA = -X_B (A_BA X_A), A and B the two halves. Each
    // off-diagonal X block overwrites its A block in AX once that is used;
    // above the diagonal AX holds zeros throughout.
    // Level 1 runs on warps 0 and 1 while warps 4 .. 15 move V'^T into shared
    // memory (rows v: the A operand of MMA2, high / low parts for the split
    // products) and rescale S0 <- S0 Diag(gamma_last) in tensor memory (MMA5
    // accumulates onto it; this chunk's MMAs read S0 from its shared copy):
    // three warps per TMEM lane quarter, 64 columns each.
    static_assert(NT == 512, "solve thread mapping");
    __syncthreads();  // A (and P) are complete
    if (warp >= 4) {
      if (!additive && warp == 4 && lane == 0) {
        if (!umma::mbar_wait(&bar_v, ph_v, kWaitTries)) {
          abort_sh = 1;
          report(a.status, LIN_ST_TIMEOUT);
        }
      }
      asm volatile("bar.sync 1, 384;" ::: "memory");  // warps 4 .. 15
      umma::fence_after_sync();
      if (!abort_sh) {
        const int part = (warp - 4) >> 2;
        if (part == 0) {
          if (!additive) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              float v16[16];
              umma::tmem_ld16(tmem_addr(tm, quarter * 32, COL_R2 + 16 * m), v16);
              if (SPLIT)
                put16_split(sb + OFF_VPT, sb + OFF_VPTL, 128, vrow, 16 * m, v16, 1.f);
              else
                put16<BF>(sb + OFF_VPT, 128, vrow, 16 * m, v16, 1.f);
            }
          }
        } else {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            float v[32];
            const int cc = (part - 1) * 64 + 32 * m;
            umma::tmem_ld32(tmem_addr(tm, quarter * 32, COL_S + cc), v);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= GLAST[KDA ? cc + k : 0];
            umma::tmem_st32(tmem_addr(tm, quarter * 32, COL_S + cc), v);
          }
        }
      }
      umma::fence_smem_to_async();
      umma::fence_before_sync();
    } else if (!additive) {
      if (tid < 64) {
        const int blk = tid >> 4, jj = tid & 15, base = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float av[16];
          const float4* ar4 = reinterpret_cast<const float4*>(AX + (base + r) * AXS + base);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            if (4 * q4 < r) {
              const float4 f = ar4[q4];
              av[4 * q4] = f.x;
              av[4 * q4 + 1] = f.y;
              av[4 * q4 + 2] = f.z;
              av[4 * q4 + 3] = f.w;
            }
          }
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int i = 0; i < r; ++i) {
            if (i & 1)
              s1 = fmaf(av[i], x[i], s1);
            else
              s0 = fmaf(av[i], x[i], s0);
          }
          // x[i] = 0 for i < jj, so the sum is 0 at and above the diagonal
          x[r] = (r == jj) ? 1.f : -(s0 + s1);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) XD[blk * XBS + r * XDS + jj] = x[r];
      }
    }
    if (!additive) ph_v ^= 1;
    __syncthreads();
    if (abort_sh) break;
    if (!additive) {
    {
      // Y_s = A_{2s+1,2s} X_{2s,2s}
      const int s2 = tid >> 8, r = (tid >> 4) & 15, c = tid & 15;
      const float* arow = AX + (32 * s2 + 16 + r) * AXS + 32 * s2;
      const float* xd = XD + (2 * s2) * XBS + c;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; m += 2) {
        acc0 = fmaf(arow[m], xd[m * XDS], acc0);
        acc1 = fmaf(arow[m + 1], xd[(m + 1) * XDS], acc1);
      }
      YB[s2 * XBS + r * XDS + c] = acc0 + acc1;
    }
    __syncthreads();
    {
      // X_{2s+1,2s} = -X_{2s+1,2s+1} Y_s, over A_{2s+1,2s}
      const int s2 = tid >> 8, r = (tid >> 4) & 15, c = tid & 15;
      const float* xr = XD + (2 * s2 + 1) * XBS + r * XDS;
      const float* yb = YB + s2 * XBS + c;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; m += 2) {
        acc0 = fmaf(xr[m], yb[m * XDS], acc0);
        acc1 = fmaf(xr[m + 1], yb[(m + 1) * XDS], acc1);
      }
      AX[(32 * s2 + 16 + r) * AXS + 32 * s2 + c] = -(acc0 + acc1);
    }
    __syncthreads();
    {
      // Z = A_BA X_A (rows 32.., cols 0..31); a warp keeps to one column half
      const int chalf = tid >> 8, r = (tid >> 3) & 31, c = chalf * 16 + 2 * (tid & 7);
      const float* arow = AX + (32 + r) * AXS;
      float z0 = 0.f, z1 = 0.f;
      if (chalf == 0) {
#pragma unroll
        for (int m = 0; m < 16; ++m) {  // X_00
          const float2 xv = *reinterpret_cast<const float2*>(XD + m * XDS + c);
          z0 = fmaf(arow[m], xv.x, z0);
          z1 = fmaf(arow[m], xv.y, z1);
        }
#pragma unroll
        for (int m = 16; m < 32; ++m) {  // X_10
          const float2 xv = *reinterpret_cast<const float2*>(AX + m * AXS + c);
          z0 = fmaf(arow[m], xv.x, z0);
          z1 = fmaf(arow[m], xv.y, z1);
        }
      } else {
#pragma unroll
        for (int m = 16; m < 32; ++m) {  // X_11
          const float2 xv = *reinterpret_cast<const float2*>(XD + XBS + (m - 16) * XDS + (c - 16));
          z0 = fmaf(arow[m], xv.x, z0);
          z1 = fmaf(arow[m], xv.y, z1);
        }
      }
      *reinterpret_cast<float2*>(ZB + r * ZS + c) = make_float2(z0, z1);
    }
    __syncthreads();
    {
      // X_BA = -X_B Z, over A_BA; a warp keeps to one row half of X_B
      const int rhalf = tid >> 8, rl = (tid >> 4) & 15, c = 2 * (tid & 15);
      float o0 = 0.f, o1 = 0.f;
      if (rhalf == 0) {
        const float* xr = XD + 2 * XBS + rl * XDS;  // X_22 row rl
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 zv = *reinterpret_cast<const float2*>(ZB + m * ZS + c);
          o0 = fmaf(xr[m], zv.x, o0);
          o1 = fmaf(xr[m], zv.y, o1);
        }
      } else {
        const float* xr1 = AX + (48 + rl) * AXS + 32;  // X_32 row rl
        const float* xr2 = XD + 3 * XBS + rl * XDS;    // X_33 row rl
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 zv = *reinterpret_cast<const float2*>(ZB + m * ZS + c);
          o0 = fmaf(xr1[m], zv.x, o0);
          o1 = fmaf(xr1[m], zv.y, o1);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 zv = *reinterpret_cast<const float2*>(ZB + (16 + m) * ZS + c);
          o0 = fmaf(xr2[m], zv.x, o0);
          o1 = fmaf(xr2[m], zv.y, o1);
        }
      }
      *reinterpret_cast<float2*>(AX + (32 + rhalf * 16 + rl) * AXS + c) = make_float2(-o0, -o1);
    }
    __syncthreads();
    }  // !additive
    {
      const int t = tid >> 3, c0 = (tid & 7) * 8;
      // the thread's 8 columns lie in one 16-wide block: a diagonal block of
      // X (XD) or an off-diagonal one (AX, zero above the diagonal)
      float xrow[8];
      if (additive) {
#pragma unroll
        for (int m = 0; m < 8; ++m) xrow[m] = (c0 + m == t) ? 1.f : 0.f;  // X = I
      } else {
        const float* src = ((c0 >> 4) == (t >> 4)) ? XD + (t >> 4) * XBS + (t & 15) * XDS + (c0 & 15)
                                                   : AX + t * AXS + c0;
        const float4 x0 = reinterpret_cast<const float4*>(src)[0], x1 = reinterpret_cast<const float4*>(src)[1];
        xrow[0] = x0.x; xrow[1] = x0.y; xrow[2] = x0.z; xrow[3] = x0.w;
        xrow[4] = x1.x; xrow[5] = x1.y; xrow[6] = x1.z; xrow[7] = x1.w;
      }
      const float4 b0 = *reinterpret_cast<const float4*>(SBETA + c0);
      const float4 b1 = *reinterpret_cast<const float4*>(SBETA + c0 + 4);
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      float tv[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) tv[m] = xrow[m] * bv[m];
      const uint32_t off = umma::rp_offset(t, c0, 64);
      if (SPLIT) {
        uint32_t h0[2], l0[2], h1[2], l1[2];
        split4(tv[0], tv[1], tv[2], tv[3], h0, l0);
        split4(tv[4], tv[5], tv[6], tv[7], h1, l1);
        st_shared_v4(sb + OFF_TT + off, h0[0], h0[1], h1[0], h1[1]);
        st_shared_v4(sb + OFF_TTL + off, l0[0], l0[1], l1[0], l1[1]);
      } else {
        st_shared_v4(sb + OFF_TT + off, umma::pack2<BF>(tv[0], tv[1]), umma::pack2<BF>(tv[2], tv[3]),
                     umma::pack2<BF>(tv[4], tv[5]), umma::pack2<BF>(tv[6], tv[7]));
      }
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    // ---- MMA2: U^T = V'^T T^T (R1); the additive form: U^T = V^T T^T
    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t id2k = umma::idesc_f16(128, 64, BF, false, false);  // A: V'^T, rows v
      constexpr uint32_t id2m = umma::idesc_f16(128, 64, BF, true, false);   // A: V, rows t
      const uint32_t id2 = additive ? id2m : id2k;
#pragma unroll
      for (int k0 = 0; k0 < CH; k0 += 16) {
        const uint64_t av = additive ? mdesc(OFF_VV, 64, k0)
                                     : kdesc(OFF_VPT, 128, k0);
        const uint64_t bt = kdesc(OFF_TT, 64, k0);
        umma::mma_f16(tm + COL_R1, av, bt, id2, k0 > 0);
        if (SPLIT) {
          umma::mma_f16(tm + COL_R1, av, kdesc(OFF_TTL, 64, k0), id2, 1);
          if (!additive) umma::mma_f16(tm + COL_R1, kdesc(OFF_VPTL, 128, k0), bt, id2, 1);
        }
      }
      umma::mma_commit(&bar_mma);
    }
    if (!wait_mma()) break;

    // ---- U^T into shared memory (rows v)
    {
      float v[16];
      umma::tmem_ld16(tmem_addr(tm, quarter * 32, COL_R1 + slice * 16), v);
      if (SPLIT)
        put16_split(sb + OFF_UT, sb + OFF_UTL, 128, vrow, slice * 16, v, 1.f);
      else
        put16<BF>(sb + OFF_UT, 128, vrow, slice * 16, v, 1.f);
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();

    // ---- MMA4b: O^T += U^T P^T (RO);  MMA5: S += U^T Ktil (S)
    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t id4 = umma::idesc_f16(128, 64, BF, false, false);
      constexpr uint32_t id5 = umma::idesc_f16(128, 128, BF, false, true);
#pragma unroll
      for (int k0 = 0; k0 < CH; k0 += 16) {
        const uint64_t ad = kdesc(OFF_UT, 128, k0);
        const uint64_t bp = kdesc(OFF_PP, 64, k0);
        const uint64_t bk = mdesc(OFF_KT, 64, k0);
        if (outputs_on) umma::mma_f16(tm + COL_RO, ad, bp, id4, 1);
        umma::mma_f16(tm + COL_S, ad, bk, id5, 1);
        if (SPLIT) {
          const uint64_t al = kdesc(OFF_UTL, 128, k0);
          if (outputs_on) {
            umma::mma_f16(tm + COL_RO, ad, kdesc(OFF_PPL, 64, k0), id4, 1);
            umma::mma_f16(tm + COL_RO, al, bp, id4, 1);
          }
          umma::mma_f16(tm + COL_S, al, bk, id5, 1);
        }
      }
      umma::mma_commit(&bar_mma);
    }
    // the next chunk's gates and betas, in flight while the last products run
    // and the epilogue stores (their registers are not live across this
    // chunk's heavier phases)
    if (j + 1 < nch) {
      const int n2 = (L - (j + 1) * CH) < CH ? (L - (j + 1) * CH) : CH;
      load_gates<KDA>(a, row0 + CH, n2, h, H, warp, lane, gk, bt);
    }
    // the snapshot this chunk ends at (if any), whether the final state goes
    // to the slot, and the stores of the conv window after the chunk (its last
    // 3 inputs, known since the conv phase). The GDN and SSD instances do both
    // while the last products run; the KDA instances, short of registers
    // there, do them in the epilogue.
    const bool full = (n == CH);
    const bool last = (j == nch - 1);
    int snap_dst = -1;
    bool last_to_slot = false, store_state = false;
    auto decide_snapshot = [&]() {
      const int64_t end_pos = int64_t(P) + int64_t(j) * CH + n;
      if (ntr > 0 && full && (end_pos % a.track_stride) == 0) {
        if (seg_mode == kSegOff || snap >= snap_total - ntr) snap_dst = a.track_slots[t0 + (snap % ntr)];
        ++snap;
      }
      // the final state goes to the slot when this CTA ends the request (and
      // runs with outputs); segment state runs write it to the workspace
      last_to_slot = last && outputs_on && seg_last;
      store_state = snap_dst >= 0 || last_to_slot;
    };
    auto store_window = [&]() {
      if (!store_state) return;
      char* snap_c = snap_dst >= 0 ? static_cast<char*>(pool.conv) +
                                         a.layer * pool.conv_layer_stride +
                                         snap_dst * pool.conv_slot_stride
                                   : nullptr;
      if constexpr (!KDA) {
        // one thread per channel, its three entries (the KDA instances keep
        // one thread per entry: there the other form costs registers)
        for (int cl = tid; cl < 384; cl += NT) {
          if (!valid_channel<VD>(cl)) continue;
          const int64_t off = int64_t(head_channel<VD>(cl, h, H)) * 3;
#pragma unroll
          for (int m = 0; m < 3; ++m) {
            const float wv = WIN[(j & 1) * 1152 + m * 384 + cl];
            if (snap_c) store_elem(snap_c, off + m, pool.conv_dtype, wv);
            if (last_to_slot) store_elem(slot_c, off + m, pool.conv_dtype, wv);
          }
        }
      } else {
        for (int idx = tid; idx < 3 * 384; idx += NT) {
          const int cl = idx / 3, m = idx % 3;
          if (!valid_channel<VD>(cl)) continue;
          const int ch = head_channel<VD>(cl, h, H);
          const float wv = WIN[(j & 1) * 1152 + m * 384 + cl];
          const int64_t off = int64_t(ch) * 3 + m;
          if (snap_c) store_elem(snap_c, off, pool.conv_dtype, wv);
          if (last_to_slot) store_elem(slot_c, off, pool.conv_dtype, wv);
        }
      }
    };
    if constexpr (!KDA) {
      decide_snapshot();
      store_window();
    }
    if (!wait_mma()) break;
    // every MMA of this chunk is done: the next chunk's x tile may land now
    if (tid == 0 && j + 1 < nch) issue_x_tile(row0 + CH);

    // ---- outputs, state operand for the next chunk, snapshots, final state.
    // Full-chunk outputs and every stored state go through swizzled staging
    // tiles and TMA stores, so the copy engine drains them while the next
    // chunk's conv phase runs.
    {
      if constexpr (KDA) decide_snapshot();
      const int oes = a.out_dtype == LIN_BF16 ? 2 : 4;
      if (outputs_on) {
        float o16[16];
        umma::tmem_ld16(tmem_addr(tm, quarter * 32, COL_RO + slice * 16), o16);
        if (vrow >= VD) {
          // padding rows of a 64-channel value side: nothing to store
        } else if (full) {
          uint8_t* ost = sm + OFF_OSTG;
          if (oes == 2) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
              reinterpret_cast<uint16_t*>(ost)[(slice * 16 + k) * VD + vrow] = f32_to_bf16_bits(o16[k]);
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) reinterpret_cast<float*>(ost)[(slice * 16 + k) * VD + vrow] = o16[k];
          }
        } else {
          const int64_t ob = (row0 * H + h) * VD + vrow;
          const int64_t ostep = int64_t(H) * VD;
          if (oes == 2) {
            uint16_t* op = static_cast<uint16_t*>(a.out) + ob;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int t = slice * 16 + k;
              if (t < n) op[t * ostep] = f32_to_bf16_bits(o16[k]);
            }
          } else {
            float* op = static_cast<float*>(a.out) + ob;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int t = slice * 16 + k;
              if (t < n) op[t * ostep] = o16[k];
            }
          }
        }
      }
      {
        float v[32];
        const int cc = slice * 32;
        umma::tmem_ld32(tmem_addr(tm, quarter * 32, COL_S + cc), v);
        if (!last) put32<BF>(sb + OFF_SOP, 128, vrow, cc, v, 1.f);
        if (last && state_to_ws) {
          float* dst = (pmode == 2 ? p.wrap.state + int64_t(plink) * DH * DH
                                   : (seg_mode == kSegTransition ? p.seg_trans_out : p.seg_state_out) +
                                         (int64_t(seg) * H + h) * DH * DH) +
                       int64_t(vrow) * DH + cc;
#pragma unroll
          for (int m = 0; m < 8; ++m)
            *reinterpret_cast<float4*>(dst + 4 * m) = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
        }
        if (store_state) {
          // state tiles of 128 rows x 128 bytes (one per 128-byte column block,
          // rows v in order), 128-byte swizzle (chunk m of row r at m ^ (r % 8))
          if (ST == LIN_BF16) {
            const uint32_t tile = sb + OFF_STG + ((slice >> 1) * 4 + quarter) * 4096 + lane * 128;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int chunk = ((slice & 1) * 4 + m) ^ (lane & 7);
              st_shared_v4(tile + chunk * 16,
                           static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m])) | (static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 1])) << 16),
                           static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 2])) | (static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 3])) << 16),
                           static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 4])) | (static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 5])) << 16),
                           static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 6])) | (static_cast<uint32_t>(f32_to_bf16_bits(v[8 * m + 7])) << 16));
            }
          } else {
            const uint32_t tile = sb + OFF_STG + (slice * 4 + quarter) * 4096 + lane * 128;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int chunk = m ^ (lane & 7);
              st_shared_v4(tile + chunk * 16, __float_as_uint(v[4 * m]), __float_as_uint(v[4 * m + 1]),
                           __float_as_uint(v[4 * m + 2]), __float_as_uint(v[4 * m + 3]));
            }
          }
        }
      }
      if constexpr (KDA) store_window();
      umma::fence_smem_to_async();
      umma::fence_before_sync();
      __syncthreads();
      if (tid == kStoreTid) {
        // bulk stores carry no order among themselves: an earlier snapshot
        // into the same track slot must have landed before this one starts.
        // Each chunk commits one group and a slot recurs every ntr snapshots,
        // so all but the latest group must be complete (all of them for ntr 1).
        if (snap_dst >= 0) {
          if (ntr == 1) bulk_wait_all();
          else bulk_wait_but_one();
        }
        if (full && outputs_on) tma_store_3d(&tmap_out, sb + OFF_OSTG, 0, h, static_cast<int>(row0));
        if (store_state) {
          constexpr int KB = ST == LIN_BF16 ? 64 : 32;  // key channels per tile
#pragma unroll
          for (int kb = 0; kb < DH / KB; ++kb) {
            const uint32_t src = sb + OFF_STG + kb * 16384;
            if (snap_dst >= 0) tma_store_4d(&tmap_state, src, kb * KB, 0, h, snap_dst);
            if (last_to_slot) tma_store_4d(&tmap_state, src, kb * KB, 0, h, slot);
          }
        }
        bulk_commit();
      }
    }
  }

  // ---- teardown: every TMA store issued here has completed, and no x tile is
  // still landing, before exit
  if (tid == kStoreTid) {
    bulk_wait_all();
    if (pmode == 2) fence_async_global();
  }
  // after an early exit the last x tile issued may not have been waited for
  // (each chunk j waited for x tile j, phase j & 1)
  if (tid == 0 && abort_sh && x_issued > 0)
    umma::mbar_wait(&bar_x, static_cast<uint32_t>((x_issued - 1) & 1), kWaitTries);
  __syncthreads();
  umma::fence_after_sync();
  // a wrap-around head piece: the state it handed on and its snapshot stores
  // (the tail's next snapshot may go to the same track slot) have landed
  if (pmode == 2 && tid == 0 && !abort_sh) {
    __threadfence();
    flag_set(p.wrap.flag + plink);
  }
  if (warp == 0) umma::tmem_dealloc(tm, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Carries the true state across the segments of a long request:
// S_{k+1} = S_k M_k + B_k for k = 1 .. nseg - 2, where buf[k] holds B_k on entry
// (buf[0] holds S_1, the offset run of segment 0 from the request's own initial
// state) and S_{k+1} on exit, and mbuf[k] holds M_k. Rows of S evolve
// independently, so CTA (head, 16-row block) runs the whole scan for its rows:
// each warp owns 4 rows and each lane 4 columns (16 fp32 sums), so every M_k
// value read from shared memory feeds 4 rows and every S_k value (the same for
// the whole warp) 4 columns. M_{k+1} lands by a bulk copy into the other of
// two buffers while step k computes. Each sum adds the terms in key order, as
// a plain row-by-matrix product does.
constexpr int kScanRows = 16;
constexpr int kScanThreads = 128;  // 4 warps x 4 rows
constexpr size_t kScanSmem = (2 * size_t(DH) * DH + size_t(kScanRows) * DH) * sizeof(float);

__global__ void __launch_bounds__(kScanThreads)
    seg_scan_kernel(float* buf, const float* mbuf, int nseg, int H, int32_t* status) {
  extern __shared__ __align__(16) float ssm[];
  __shared__ uint64_t mbar[2];
  __shared__ int ok_sh;
  float* Ssh = ssm + 2 * DH * DH;  // this CTA's rows of S_k, 16 x 128
  const int h = blockIdx.x / (DH / kScanRows), rb = blockIdx.x % (DH / kScanRows);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = warp * 4, c0 = lane * 4;  // this thread's rows (of the CTA's 16) and columns
  const int64_t head_elems = int64_t(DH) * DH;
  auto at = [&](const float* base, int k) { return base + (int64_t(k) * H + h) * head_elems; };
  auto atw = [&](float* base, int k) { return base + (int64_t(k) * H + h) * head_elems; };
  if (tid == 0) {
    ok_sh = 1;
    umma::mbar_init(&mbar[0], 1);
    umma::mbar_init(&mbar[1], 1);
    umma::mbar_fence_init();
  }
  for (int i = tid; i < kScanRows * DH / 4; i += kScanThreads)
    reinterpret_cast<float4*>(Ssh)[i] = reinterpret_cast<const float4*>(at(buf, 0) + int64_t(rb) * kScanRows * DH)[i];
  __syncthreads();
  constexpr uint32_t kMBytes = DH * DH * sizeof(float);
  auto issue = [&](int k) {  // thread 0: M_k into buffer k & 1
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[k & 1]));
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(ssm + (k & 1) * DH * DH));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kMBytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(at(mbuf, k)), "r"(kMBytes), "r"(bar)
                 : "memory");
  };
  // thread 0's bookkeeping: each buffer's next phase, and whether a copy into
  // it is in flight
  uint32_t phase[2] = {0u, 0u};
  bool pend[2] = {false, false};
  if (tid == 0 && nseg > 2) {
    issue(1);
    pend[1] = true;
  }
  for (int k = 1; k + 1 < nseg; ++k) {
    const int bi = k & 1;
    // the other buffer's last reader was step k - 1, which every thread finished
    if (tid == 0 && k + 2 < nseg) {
      issue(k + 1);
      pend[bi ^ 1] = true;
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 bv = *reinterpret_cast<const float4*>(atw(buf, k) + int64_t(rb * kScanRows + r0 + i) * DH + c0);
      acc[i][0] = bv.x;
      acc[i][1] = bv.y;
      acc[i][2] = bv.z;
      acc[i][3] = bv.w;
    }
    if (tid == 0) {
      if (umma::mbar_wait(&mbar[bi], phase[bi], kWaitTries)) {
        phase[bi] ^= 1u;
        pend[bi] = false;
      } else {
        ok_sh = 0;
        if (status) atomicOr(status, LIN_ST_TIMEOUT);
      }
    }
    __syncthreads();
    if (!ok_sh) break;
    const float* Msh = ssm + bi * DH * DH;
#pragma unroll 2
    for (int m = 0; m < DH; m += 4) {
      float4 sv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sv[i] = *reinterpret_cast<const float4*>(Ssh + (r0 + i) * DH + m);
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const float4 mv = *reinterpret_cast<const float4*>(Msh + (m + mm) * DH + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float s = mm == 0 ? sv[i].x : mm == 1 ? sv[i].y : mm == 2 ? sv[i].z : sv[i].w;
          acc[i][0] = fmaf(s, mv.x, acc[i][0]);
          acc[i][1] = fmaf(s, mv.y, acc[i][1]);
          acc[i][2] = fmaf(s, mv.z, acc[i][2]);
          acc[i][3] = fmaf(s, mv.w, acc[i][3]);
        }
      }
    }
    __syncthreads();  // every read of S_k and M_k is done
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 o = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(Ssh + (r0 + i) * DH + c0) = o;
      *reinterpret_cast<float4*>(atw(buf, k) + int64_t(rb * kScanRows + r0 + i) * DH + c0) = o;
    }
    __syncthreads();
  }
  if (!ok_sh && tid == 0) {
    // copies may still be landing: wait for them (bounded) before exit
    for (int b = 0; b < 2; ++b)
      if (pend[b]) umma::mbar_wait(&mbar[b], phase[b], kWaitTries);
  }
}

// Segments for one long request: enough (segment, head) CTAs to fill every SM
// about six times, each segment a whole number of chunks (at least 4).
struct SegPlan {
  int nseg = 0, seg_len = 0;
};

SegPlan segment_plan(const lin_state_pool_t& pool, const lin_prefill_args_t& a) {
  SegPlan sp;
  if (a.batch != 1 || (a.flags & LIN_PREFILL_RECURRENT)) return sp;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return sp;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return sp;
  const int64_t nch = (a.total_tokens + CH - 1) / CH;
  const bool forced = (a.flags & LIN_PREFILL_SEGMENTED) != 0;
  const bool want = forced ? nch >= 8 : (int64_t(pool.num_heads) * 4 <= sms && nch >= 64);
  if (!want) return sp;
  const int64_t target = int64_t(6) * sms;
  int64_t seg_ch = (nch * pool.num_heads + target - 1) / target;
  if (seg_ch < 4) seg_ch = 4;
  const int64_t nseg = (nch + seg_ch - 1) / seg_ch;
  if (nseg < 2 || nseg * pool.num_heads >= (int64_t(1) << 31) || seg_ch * CH >= (int64_t(1) << 30))
    return sp;
  sp.nseg = static_cast<int>(nseg);
  sp.seg_len = static_cast<int>(seg_ch * CH);
  return sp;
}

size_t segment_workspace(const lin_state_pool_t& pool, const SegPlan& sp) {
  if (sp.nseg < 2) return 0;
  return 2 * size_t(sp.nseg) * pool.num_heads * DH * DH * sizeof(float);
}

// Wrap-around schedule: for a batch with more (request, head) chains than
// SMs (one chain per SM is already as good as it gets), in one piece per
// chain unless LIN_PREFILL_ONE_PIECE; ranges = SMs.
struct WrapPlan {
  int grid = 0, max_pieces = 0;
};

WrapPlan wrap_plan(const lin_state_pool_t& pool, const lin_prefill_args_t& a, const SegPlan& sp) {
  WrapPlan wp;
  if (sp.nseg >= 2 || (a.flags & (LIN_PREFILL_RECURRENT | LIN_PREFILL_ONE_PIECE))) return wp;
  if (a.batch < 1 || a.batch > kOrderMax) return wp;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return wp;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return wp;
  const int64_t chains = int64_t(a.batch) * pool.num_heads;
  if (chains <= sms || chains + sms > kWrapMaxPieces) return wp;
  wp.grid = sms;
  wp.max_pieces = static_cast<int>(chains + sms);
  return wp;
}

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t wrap_workspace(const WrapPlan& wp) {
  if (wp.grid == 0) return 0;
  return align256(2 * sizeof(int32_t)) + align256(size_t(wp.max_pieces) * sizeof(WrapPiece)) +
         align256(size_t(wp.max_pieces) * sizeof(int32_t)) + align256(size_t(wp.grid) * sizeof(uint32_t)) +
         size_t(wp.grid) * DH * DH * sizeof(float);
}

// The wrap-around buffers carved from a workspace of wrap_workspace(wp) bytes.
struct WrapBufs {
  int grid = 0;
  int32_t* ctl = nullptr;
  WrapPiece* piece = nullptr;
  int32_t* order = nullptr;
  uint32_t* flag = nullptr;
  float* state = nullptr;
};

WrapBufs carve_wrap(const WrapPlan& wp, char* ws) {
  WrapBufs b;
  if (wp.grid == 0 || !ws) return b;
  b.grid = wp.grid;
  b.ctl = reinterpret_cast<int32_t*>(ws);
  ws += align256(2 * sizeof(int32_t));
  b.piece = reinterpret_cast<WrapPiece*>(ws);
  ws += align256(size_t(wp.max_pieces) * sizeof(WrapPiece));
  b.order = reinterpret_cast<int32_t*>(ws);
  ws += align256(size_t(wp.max_pieces) * sizeof(int32_t));
  b.flag = reinterpret_cast<uint32_t*>(ws);
  ws += align256(size_t(wp.grid) * sizeof(uint32_t));
  b.state = reinterpret_cast<float*>(ws);
  return b;
}

template <bool KDA, int ST, int VD>
cudaError_t launch_t(const lin_state_pool_t& pool, const lin_prefill_args_t& a, int32_t* order,
                     const SegPlan& sp, float* seg_buf, uint32_t* redo, const WrapBufs& wb, cudaStream_t s) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(pool.conv_channels),
                              static_cast<cuuint64_t>(a.total_tokens)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pool.conv_channels) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(DH), static_cast<cuuint32_t>(XR)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // x tiles loaded into shared memory: 64 rows x 128 channels, row-major
  CUtensorMap tmap_xt;
  {
    const cuuint32_t bxt[2] = {static_cast<cuuint32_t>(DH), static_cast<cuuint32_t>(CH)};
    cr = enc(&tmap_xt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides, bxt,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // state tiles: [slot][H][V][K] of this layer, box 128 rows x 128 bytes
  CUtensorMap tmap_state;
  {
    const int es = ST == LIN_BF16 ? 2 : 4;
    char* base = static_cast<char*>(pool.temporal) + a.layer * pool.temporal_layer_stride;
    const cuuint64_t d[4] = {DH, VD, static_cast<cuuint64_t>(pool.num_heads),
                             static_cast<cuuint64_t>(pool.num_slots)};
    const cuuint64_t st[3] = {static_cast<cuuint64_t>(DH) * es, static_cast<cuuint64_t>(VD) * DH * es,
                              static_cast<cuuint64_t>(pool.temporal_slot_stride)};
    const cuuint32_t bx[4] = {static_cast<cuuint32_t>(128 / es), VD, 1, 1};
    const cuuint32_t es4[4] = {1, 1, 1, 1};
    cr = enc(&tmap_state, ST == LIN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             4, base, d, st, bx, es4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // output tiles: [T][H][V], box 64 tokens x 1 head x 128
  CUtensorMap tmap_out;
  {
    const int es = a.out_dtype == LIN_BF16 ? 2 : 4;
    const cuuint64_t d[3] = {VD, static_cast<cuuint64_t>(pool.num_heads),
                             static_cast<cuuint64_t>(a.total_tokens)};
    const cuuint64_t st[2] = {static_cast<cuuint64_t>(VD) * es,
                              static_cast<cuuint64_t>(VD) * pool.num_heads * es};
    const cuuint32_t bx[3] = {VD, 1, CH};
    const cuuint32_t es3[3] = {1, 1, 1};
    cr = enc(&tmap_out, a.out_dtype == LIN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             3, a.out, d, st, bx, es3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const bool segmented = sp.nseg >= 2 && seg_buf;
  auto kern = segmented ? chunked_prefill_kernel<KDA, ST, true, VD> : chunked_prefill_kernel<KDA, ST, false, VD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const unsigned H = static_cast<unsigned>(pool.num_heads);
  if (wb.grid > 0 && !segmented) {
    // the wrap-around plan, then one CTA per piece (at most chains + ranges)
    if ((e = cudaFuncSetAttribute(wrap_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kWrapPlanSmem))) != cudaSuccess)
      return e;
    wrap_plan_kernel<<<1, 1024, kWrapPlanSmem, s>>>(a, int(H), pool.num_slots, wb.grid, wb.ctl, wb.piece, wb.order,
                                                    wb.flag);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ChunkParams pw{pool, a, nullptr, kSegOff, 0, 0, 0, nullptr, nullptr, nullptr, redo,
                   WrapBuf{wb.ctl, wb.piece, wb.order, wb.flag, wb.state}};
    const unsigned grid = static_cast<unsigned>(a.batch) * H + static_cast<unsigned>(wb.grid);
    kern<<<grid, NT, SMEM_BYTES, s>>>(tmap, tmap_xt, tmap_state, tmap_out, pw);
    return cudaGetLastError();
  }
  if (order) {
    order_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.batch, order);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
  }
  if (segmented) {
    // one long request in segments: offset runs (segments 0 .. n-2) and
    // transition runs (1 .. n-2), the scan, then the final runs (all)
    float* bbuf = seg_buf;
    float* mbuf = seg_buf + size_t(sp.nseg) * H * DH * DH;
    // offset runs of segments 0 .. n-2 (segment 0 also with its outputs and
    // snapshots) and transition runs of segments 1 .. n-2, one launch
    ChunkParams p1{pool, a, nullptr, kSegOffsetAndTransition, sp.seg_len, 0, sp.nseg, bbuf, mbuf, nullptr, redo};
    kern<<<unsigned(2 * sp.nseg - 3) * H, NT, SMEM_BYTES, s>>>(tmap, tmap_xt, tmap_state, tmap_out, p1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (sp.nseg > 2) {
      if ((e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kScanSmem))) != cudaSuccess)
        return e;
      seg_scan_kernel<<<H * (DH / kScanRows), kScanThreads, kScanSmem, s>>>(bbuf, mbuf, sp.nseg, int(H), a.status);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ChunkParams p3{pool, a, nullptr, kSegFinal, sp.seg_len, 1, sp.nseg, nullptr, nullptr, bbuf, redo};
    kern<<<unsigned(sp.nseg - 1) * H, NT, SMEM_BYTES, s>>>(tmap, tmap_xt, tmap_state, tmap_out, p3);
    return cudaGetLastError();
  }
  ChunkParams p{pool, a, order, kSegOff, 0, 0, 0, nullptr, nullptr, nullptr, redo};
  const unsigned grid = static_cast<unsigned>(a.batch) * H;
  kern<<<grid, NT, SMEM_BYTES, s>>>(tmap, tmap_xt, tmap_state, tmap_out, p);
  return cudaGetLastError();
}

}  // namespace

bool chunked_prefill_supported(const lin_state_pool_t& pool, const lin_prefill_args_t& a) {
  return pool.head_k == DH && (pool.head_v == DH || pool.head_v == 64) && a.io_dtype == LIN_BF16 &&
         a.total_tokens > 0 &&
         int64_t(a.batch) * pool.num_heads < (int64_t(1) << 31) &&
         (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.g) & 15) == 0 && encode_fn() != nullptr;
}

namespace {
// The longest-first order of the batch (int32 per request) when the batch has
// more than one request and fits the sorting kernel.
size_t order_workspace(const lin_prefill_args_t& a) {
  if (a.batch <= 1 || a.batch > kOrderMax) return 0;
  return (static_cast<size_t>(a.batch) * sizeof(int32_t) + 255) & ~size_t(255);
}

// KDA: one bit per (request, head), set for a pair whose decay left the
// chunk's factored range (the token-by-token rerun redoes those pairs).
size_t redo_workspace(const lin_state_pool_t& pool, const lin_prefill_args_t& a) {
  if (a.gate_mode != LIN_GATE_PER_KEY) return 0;
  const size_t words = (static_cast<size_t>(a.batch) * pool.num_heads + 31) / 32;
  return (words * sizeof(uint32_t) + 255) & ~size_t(255);
}

// Order (when given), the chunked launch(es), and for KDA the rerun of the
// pairs the chunked kernel flagged: the flags are cleared first, and the
// token-by-token launch behind the chunked one runs only the flagged pairs
// (the others return at once), so no host synchronisation is needed.
cudaError_t launch_chunked(const lin_state_pool_t& pool, const lin_prefill_args_t& a, int32_t* order,
                           const SegPlan& sp, float* seg_buf, uint32_t* redo, const WrapBufs& wb,
                           cudaStream_t stream) {
  const bool kda = a.gate_mode == LIN_GATE_PER_KEY;
  const bool bf = pool.state_dtype == LIN_BF16;
  const bool v64 = pool.head_v == 64;
  cudaError_t e;
  if (kda) {
    if (!redo) return cudaErrorInvalidValue;
    if ((e = cudaMemsetAsync(redo, 0, redo_workspace(pool, a), stream)) != cudaSuccess) return e;
    if (v64)
      e = bf ? launch_t<true, LIN_BF16, 64>(pool, a, order, sp, seg_buf, redo, wb, stream)
             : launch_t<true, LIN_F32, 64>(pool, a, order, sp, seg_buf, redo, wb, stream);
    else
      e = bf ? launch_t<true, LIN_BF16, DH>(pool, a, order, sp, seg_buf, redo, wb, stream)
             : launch_t<true, LIN_F32, DH>(pool, a, order, sp, seg_buf, redo, wb, stream);
    if (e != cudaSuccess) return e;
    return launch_prefill_recurrent(pool, a, stream, redo);
  }
  if (v64)
    return bf ? launch_t<false, LIN_BF16, 64>(pool, a, order, sp, seg_buf, nullptr, wb, stream)
              : launch_t<false, LIN_F32, 64>(pool, a, order, sp, seg_buf, nullptr, wb, stream);
  return bf ? launch_t<false, LIN_BF16, DH>(pool, a, order, sp, seg_buf, nullptr, wb, stream)
            : launch_t<false, LIN_F32, DH>(pool, a, order, sp, seg_buf, nullptr, wb, stream);
}
}  // namespace

// Workspace: the batch order (varlen batches), the per-segment states of a
// long single request run in segments, and the KDA rerun flags.
size_t chunked_prefill_workspace(const lin_state_pool_t& pool, const lin_prefill_args_t& a) {
  const SegPlan sp = segment_plan(pool, a);
  return order_workspace(a) + segment_workspace(pool, sp) + redo_workspace(pool, a) +
         wrap_workspace(wrap_plan(pool, a, sp));
}

cudaError_t launch_prefill_chunked(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const size_t ow = order_workspace(a), rw = redo_workspace(pool, a);
  SegPlan sp = segment_plan(pool, a);
  const size_t sw = segment_workspace(pool, sp);
  const WrapPlan wp = wrap_plan(pool, a, sp);
  const size_t ww = wrap_workspace(wp);
  if (ow + sw + rw + ww > 0 && (!workspace || workspace_bytes < ow + sw + rw + ww)) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(workspace);
  int32_t* order = ow > 0 ? reinterpret_cast<int32_t*>(ws) : nullptr;
  float* seg_buf = sw > 0 ? reinterpret_cast<float*>(ws + ow) : nullptr;
  uint32_t* redo = rw > 0 ? reinterpret_cast<uint32_t*>(ws + ow + sw) : nullptr;
  const WrapBufs wb = carve_wrap(wp, ww > 0 ? ws + ow + sw + rw : nullptr);
  if (!seg_buf) sp = SegPlan{};
  return launch_chunked(pool, a, order, sp, seg_buf, redo, wb, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free prefill: its scratch (the batch order, the KDA rerun flags)
// lives in fixed device arrays of this file instead of a caller workspace.
// Every GPU that loads the library holds them until exit. All calls share
// them, so calls that overlap on the GPU race on them. Each call rewrites the
// order entries it reads and clears the flags it uses before its launch.
// ---------------------------------------------------------------------------
constexpr int kNoAllocMaxBatch = kOrderMax;        // requests of a sorted batch: 16 KB
constexpr int64_t kNoAllocMaxPairs = int64_t(1) << 18;  // (request, head) pairs of a KDA call: 32 KB
static __device__ __align__(256) int32_t g_noalloc_order[kNoAllocMaxBatch];
static __device__ __align__(256) uint32_t g_noalloc_redo[kNoAllocMaxPairs / 32];

namespace {
// In host code the arrays' names are stand-ins, not device addresses: the
// addresses are looked up with the device current, once per device and
// context (a new context of the device, e.g. after cudaDeviceReset, may load
// the module elsewhere), and cached.
struct NoAllocAddrs {
  unsigned long long ctx = 0;  // id of the context the addresses belong to (0: none yet)
  int32_t* order = nullptr;
  uint32_t* redo = nullptr;
};
std::mutex g_noalloc_mu;
NoAllocAddrs g_noalloc_addrs[kMaxDevices];

// Id of the calling thread's current context, 0 when it cannot be read (the
// addresses are then looked up on every call).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t noalloc_addresses(int32_t** order, uint32_t** redo) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocAddrs& c = g_noalloc_addrs[dev];
  if (ctx == 0 || c.ctx != ctx) {
    NoAllocAddrs n;
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&n.order), g_noalloc_order)) != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&n.redo), g_noalloc_redo)) != cudaSuccess) return e;
    n.ctx = ctx;
    c = n;
  }
  *order = c.order;
  *redo = c.redo;
  return cudaSuccess;
}
}  // namespace

int noalloc_max_batch() { return kNoAllocMaxBatch; }
int64_t noalloc_max_pairs() { return kNoAllocMaxPairs; }

cudaError_t launch_prefill_noalloc(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                                   cudaStream_t stream) {
  if (!chunked_prefill_supported(pool, a) || (a.flags & LIN_PREFILL_RECURRENT))
    return launch_prefill_recurrent(pool, a, stream);  // needs no scratch
  const bool sorted = order_workspace(a) > 0;
  const bool kda = a.gate_mode == LIN_GATE_PER_KEY;
  if (sorted && a.batch > kNoAllocMaxBatch) return cudaErrorInvalidValue;
  if (kda && int64_t(a.batch) * pool.num_heads > kNoAllocMaxPairs) return cudaErrorInvalidValue;
  int32_t* order = nullptr;
  uint32_t* redo = nullptr;
  if (sorted || kda) {
    cudaError_t e = noalloc_addresses(&order, &redo);
    if (e != cudaSuccess) return e;
  }
  // a single long request runs in one piece: the segmented mode needs
  // per-segment state scratch that grows with the request
  return launch_chunked(pool, a, sorted ? order : nullptr, SegPlan{}, nullptr, kda ? redo : nullptr, WrapBufs{},
                        stream);
}

}  // namespace lin
