// Internal launchers shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lin_state.h"

namespace lin {

__host__ __device__ inline int dtype_size(int dt) { return dt == LIN_BF16 ? 2 : 4; }

// Devices a process may address through the per-device caches below.
constexpr int kMaxDevices = 64;
// Streaming multiprocessors of device `dev` (queried once per device; 0 when
// the query fails or dev is out of range).
int device_sm_count(int dev);

// Slot copy family (copy_kernels.cu).
cudaError_t launch_copy_slots(const lin_state_pool_t& pool, const int32_t* src,
                              const int32_t* dst, int32_t n, int32_t layer_begin,
                              int32_t layer_end, uint32_t flags, int32_t* status,
                              cudaStream_t stream);
cudaError_t launch_restore(const lin_state_pool_t& pool, const lin_cache_op_t* ops,
                           int32_t n, int64_t* has_initial_state, int32_t* status,
                           cudaStream_t stream);
cudaError_t launch_spec_commit(const lin_state_pool_t& pool, const lin_commit_args_t& a,
                               cudaStream_t stream);

// Token-by-token kernels (token_kernels.cu).
// Bytes one decode item stages in shared memory (state block, conv window,
// taps, n_draft x rows and per-key g rows, 128-aligned); the kernel holds two.
int decode_stage_bytes(const lin_state_pool_t& pool, const lin_decode_args_t& a);
constexpr int kDecodeMaxStage = 110 * 1024;
// accept: NULL for decode / verify; per-request accepted token counts for a
// replay commit (in place, no outputs).
cudaError_t launch_decode(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                          const int32_t* accept, cudaStream_t stream);
// redo: when given, one bit per (request, head) (bit r * H + h); only the
// pairs whose bit is set run (the rerun behind a KDA chunked launch).
cudaError_t launch_prefill_recurrent(const lin_state_pool_t& pool,
                                     const lin_prefill_args_t& a, cudaStream_t stream,
                                     const uint32_t* redo = nullptr);

// Outputs-only verify as one chunk of drafts (verify_chunk.cu): the drafts'
// outputs from the slot state with the state carried in fp32 across them.
constexpr int kVerifyChunkMaxDraft = 32;
int verify_chunk_smem(const lin_state_pool_t& pool, const lin_decode_args_t& a);
cudaError_t launch_verify_chunk(const lin_state_pool_t& pool, const lin_decode_args_t& a,
                                cudaStream_t stream);

// Chunked tensor-core prefill (chunked_prefill.cu).
bool chunked_prefill_supported(const lin_state_pool_t& pool, const lin_prefill_args_t& a);
size_t chunked_prefill_workspace(const lin_state_pool_t& pool, const lin_prefill_args_t& a);
cudaError_t launch_prefill_chunked(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                                   void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

// Prefill whose scratch is fixed device arrays (chunked_prefill.cu): at most
// noalloc_max_batch() requests when the chunked kernel sorts the batch (more
// than one request), at most noalloc_max_pairs() (request, head) pairs for
// per-key (KDA) gates on the chunked kernel.
int noalloc_max_batch();
int64_t noalloc_max_pairs();
cudaError_t launch_prefill_noalloc(const lin_state_pool_t& pool, const lin_prefill_args_t& a,
                                   cudaStream_t stream);

// Tensor-core layout self-test (selftest.cu).
cudaError_t launch_mma_selftest(const float* A, const float* B, float* D, int N, int K, int flags,
                                int32_t* status, cudaStream_t stream);

}  // namespace lin
