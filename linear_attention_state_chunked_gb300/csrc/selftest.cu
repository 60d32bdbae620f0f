// Self-test of the tensor-core operand layouts the chunked prefill relies on:
// one CTA stages A [128][K] and B [N][K] into shared memory as K-major or
// MN-major row panels, runs D = A B^T with tcgen05.mma (fp16 or bf16 operands,
// fp32 accumulator in tensor memory) over K/16 steps, and writes D [128][N].

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace lin {
namespace {

constexpr uint32_t kWaitTries = 1u << 24;

__global__ void __launch_bounds__(128) mma_selftest_kernel(const float* __restrict__ A,
                                                           const float* __restrict__ B,
                                                           float* __restrict__ D, int N, int K,
                                                           int flags, int32_t* status) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const bool a_mn = flags & 1, b_mn = flags & 2, bf = flags & 4;
  const uint32_t base = (umma::smem_u32(dyn_smem) + 1023u) & ~1023u;
  uint8_t* sp = dyn_smem + (base - umma::smem_u32(dyn_smem));
  const uint32_t a_off = 0;
  const uint32_t b_off = a_mn ? umma::rp_bytes(K, 128) : umma::rp_bytes(128, K);
  const int tid = threadIdx.x;
  for (int i = tid; i < 128 * K; i += 128) {
    const int m = i / K, k = i % K;
    const float v = A[i];
    const uint32_t o = a_mn ? umma::rp_offset(k, m, K) : umma::rp_offset(m, k, 128);
    uint16_t h;
    if (bf) { __nv_bfloat16 t = __float2bfloat16_rn(v); h = *reinterpret_cast<uint16_t*>(&t); }
    else { __half t = __float2half_rn(v); h = *reinterpret_cast<uint16_t*>(&t); }
    *reinterpret_cast<uint16_t*>(sp + a_off + o) = h;
  }
  for (int i = tid; i < N * K; i += 128) {
    const int n = i / K, k = i % K;
    const float v = B[i];
    const uint32_t o = b_mn ? umma::rp_offset(k, n, K) : umma::rp_offset(n, k, N);
    uint16_t h;
    if (bf) { __nv_bfloat16 t = __float2bfloat16_rn(v); h = *reinterpret_cast<uint16_t*>(&t); }
    else { __half t = __float2half_rn(v); h = *reinterpret_cast<uint16_t*>(&t); }
    *reinterpret_cast<uint16_t*>(sp + b_off + o) = h;
  }
  umma::fence_smem_to_async();
  if (tid == 0) {
    umma::mbar_init(&bar, 1);
    umma::mbar_fence_init();
    abort_flag = 0;
  }
  if (tid < 32) umma::tmem_alloc(&tmem_base, 128);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tm = tmem_base;
  if (tid == 0) {
    const uint32_t idesc = umma::idesc_f16(128, N, bf, a_mn, b_mn);
    for (int k0 = 0; k0 < K; k0 += 16) {
      const uint64_t ad = a_mn ? umma::desc_mnmajor(base + a_off, K, k0)
                               : umma::desc_kmajor(base + a_off, 128, k0);
      const uint64_t bd = b_mn ? umma::desc_mnmajor(base + b_off, K, k0)
                               : umma::desc_kmajor(base + b_off, N, k0);
      umma::mma_f16(tm, ad, bd, idesc, k0 > 0);
    }
    umma::mma_commit(&bar);
    if (!umma::mbar_wait(&bar, 0, kWaitTries)) {
      abort_flag = 1;
      report(status, LIN_ST_TIMEOUT);
    }
  }
  __syncthreads();
  umma::fence_after_sync();
  if (!abort_flag) {
    const int w = tid >> 5, lane = tid & 31;
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      umma::tmem_ld32(tm + ((static_cast<uint32_t>(w * 32)) << 16) + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) D[(w * 32 + lane) * N + c0 + i] = v[i];
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tm, 128);
}

}  // namespace

cudaError_t launch_mma_selftest(const float* A, const float* B, float* D, int N, int K, int flags,
                                int32_t* status, cudaStream_t stream) {
  const size_t a_bytes = (flags & 1) ? umma::rp_bytes(K, 128) : umma::rp_bytes(128, K);
  const size_t b_bytes = (flags & 2) ? umma::rp_bytes(K, N) : umma::rp_bytes(N, K);
  const size_t smem = a_bytes + b_bytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(mma_selftest_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  mma_selftest_kernel<<<1, 128, smem, stream>>>(A, B, D, N, K, flags, status);
  return cudaGetLastError();
}

}  // namespace lin
