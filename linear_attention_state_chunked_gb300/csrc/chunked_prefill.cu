// Chunked tensor-core prefill (tcgen05 / TMEM / TMA, sm_103a).
#include "common.cuh"
#include "internal.h"

namespace lin {

bool chunked_prefill_supported(const lin_state_pool_t&, const lin_prefill_args_t&) { return false; }
size_t chunked_prefill_workspace(const lin_state_pool_t&, const lin_prefill_args_t&) { return 0; }
cudaError_t launch_prefill_chunked(const lin_state_pool_t&, const lin_prefill_args_t&, void*, size_t,
                                   cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace lin
