// C-ABI entry points: host-side validation, then one or two launches on the
// caller's stream. Nothing here allocates device memory or synchronises,
// except lin_state_read_status.

#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_last_error[0] = '\0';
  return LIN_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(LIN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_dtype(int d) { return d == LIN_F32 || d == LIN_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_pool(const lin_state_pool_t* p) {
  if (!p) return fail(LIN_EINVAL, "pool is NULL");
  if (p->num_layers <= 0 || p->num_slots <= 0 || p->num_heads <= 0)
    return fail(LIN_EINVAL, "pool: num_layers, num_slots, num_heads must be positive");
  if (!valid_dtype(p->state_dtype) || !valid_dtype(p->conv_dtype))
    return fail(LIN_EINVAL, "pool: state_dtype / conv_dtype must be LIN_F32 or LIN_BF16");
  if (p->conv_width != 4) return fail(LIN_EUNSUPPORTED, "pool: conv_width must be 4");
  const bool square = p->head_k == p->head_v &&
                      (p->head_k == 16 || p->head_k == 32 || p->head_k == 64 || p->head_k == 128);
  if (!square && !(p->head_k == 128 && p->head_v == 64))
    return fail(LIN_EUNSUPPORTED,
                "pool: (head_k, head_v) must be (16,16), (32,32), (64,64), (128,128) or (128,64) (got (%d,%d))",
                p->head_k, p->head_v);
  const int64_t C = 2LL * p->num_heads * p->head_k + int64_t(p->num_heads) * p->head_v;
  if (p->conv_channels != C)
    return fail(LIN_EINVAL, "pool: conv_channels must be 2*H*K + H*V = %lld (got %d)",
                static_cast<long long>(C), p->conv_channels);
  if (!p->temporal || !p->conv) return fail(LIN_EINVAL, "pool: temporal / conv is NULL");
  if (!aligned16(p->temporal) || !aligned16(p->conv))
    return fail(LIN_EINVAL, "pool: temporal / conv must be 16-byte aligned");
  const int64_t tb = int64_t(p->num_heads) * p->head_v * p->head_k * lin::dtype_size(p->state_dtype);
  const int64_t cb = C * (p->conv_width - 1) * lin::dtype_size(p->conv_dtype);
  const int64_t strides[4] = {p->temporal_layer_stride, p->temporal_slot_stride,
                              p->conv_layer_stride, p->conv_slot_stride};
  for (int i = 0; i < 4; ++i)
    if (strides[i] < 0 || (strides[i] & 15))
      return fail(LIN_EINVAL, "pool: strides must be non-negative multiples of 16 bytes");
  if (p->temporal_slot_stride < tb || (p->num_layers > 1 && p->temporal_layer_stride < tb))
    return fail(LIN_EINVAL, "pool: temporal strides smaller than one [H][V][K] block");
  if (p->conv_slot_stride < cb || (p->num_layers > 1 && p->conv_layer_stride < cb))
    return fail(LIN_EINVAL, "pool: conv strides smaller than one [C][3] block");
  auto no_overlap = [&](int64_t ls, int64_t ss) {
    return p->num_layers == 1 || ls >= int64_t(p->num_slots) * ss ||
           ss >= int64_t(p->num_layers) * ls;
  };
  if (!no_overlap(p->temporal_layer_stride, p->temporal_slot_stride) ||
      !no_overlap(p->conv_layer_stride, p->conv_slot_stride))
    return fail(LIN_EINVAL, "pool: layer and slot strides make blocks overlap");
  return LIN_OK;
}

int check_spec(const lin_state_pool_t* p, const lin_spec_buf_t& s, int batch, int n_draft,
               int layer_end) {
  if (!s.temporal || !s.conv) return fail(LIN_EINVAL, "spec buffer is NULL");
  if (layer_end > s.num_layers)
    return fail(LIN_EINVAL, "spec buffer holds %d layers, layer %d requested", s.num_layers,
                layer_end - 1);
  if (!aligned16(s.temporal) || !aligned16(s.conv))
    return fail(LIN_EINVAL, "spec buffer must be 16-byte aligned");
  if (s.max_batch < batch || s.max_draft < n_draft)
    return fail(LIN_EINVAL, "spec buffer too small: max_batch %d < %d or max_draft %d < %d",
                s.max_batch, batch, s.max_draft, n_draft);
  const int64_t st[6] = {s.temporal_layer_stride, s.temporal_req_stride, s.temporal_step_stride,
                         s.conv_layer_stride, s.conv_req_stride, s.conv_step_stride};
  for (int i = 0; i < 6; ++i)
    if (st[i] < 0 || (st[i] & 15))
      return fail(LIN_EINVAL, "spec buffer strides must be non-negative multiples of 16 bytes");
  const int64_t tb = int64_t(p->num_heads) * p->head_v * p->head_k * lin::dtype_size(p->state_dtype);
  if (n_draft > 1 && s.temporal_step_stride < tb)
    return fail(LIN_EINVAL, "spec buffer step stride smaller than one state block");
  return LIN_OK;
}

}  // namespace

extern "C" {

int lin_state_version(void) { return (1 << 16) | 1; }

int lin_state_selftest_mma(const float* A, const float* B, float* D, int32_t n, int32_t k,
                           int32_t flags, int32_t* status, void* stream) {
  if (!A || !B || !D) return fail(LIN_EINVAL, "selftest: NULL matrix");
  if ((n != 32 && n != 64 && n != 128) || k < 16 || k > 128 || (k % 16))
    return fail(LIN_EINVAL, "selftest: n in {32,64,128}, k a multiple of 16 up to 128");
  cudaError_t e = lin::launch_mma_selftest(A, B, D, n, k, flags & 7, status,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_selftest_mma launch");
  return ok();
}

const char* lin_state_strerror(int code) {
  switch (code) {
    case LIN_OK: return "ok";
    case LIN_EINVAL: return "invalid argument";
    case LIN_EUNSUPPORTED: return "unsupported configuration";
    case LIN_ECUDA: return "CUDA runtime error";
    case LIN_EWORKSPACE: return "workspace too small";
    default: return "unknown error";
  }
}

const char* lin_state_last_error(void) { return g_last_error; }

int64_t lin_state_slot_bytes(const lin_state_pool_t* pool) {
  int rc = check_pool(pool);
  if (rc) return rc;
  const int64_t tb = int64_t(pool->num_heads) * pool->head_v * pool->head_k *
                     lin::dtype_size(pool->state_dtype);
  const int64_t cb = int64_t(pool->conv_channels) * (pool->conv_width - 1) *
                     lin::dtype_size(pool->conv_dtype);
  return int64_t(pool->num_layers) * (tb + cb);
}

int lin_state_read_status(int32_t* status, int32_t* value, void* stream) {
  if (!status || !value) return fail(LIN_EINVAL, "status / value is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(value, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_read_status");
  return ok();
}

static int check_prefill(const lin_state_pool_t* pool, const lin_prefill_args_t* a) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (!a) return fail(LIN_EINVAL, "prefill args is NULL");
  if (a->layer < 0 || a->layer >= pool->num_layers)
    return fail(LIN_EINVAL, "prefill: layer %d outside [0, %d)", a->layer, pool->num_layers);
  if (a->batch < 0 || a->total_tokens < 0) return fail(LIN_EINVAL, "prefill: negative batch / total_tokens");
  if (!valid_dtype(a->io_dtype) || !valid_dtype(a->out_dtype))
    return fail(LIN_EINVAL, "prefill: io_dtype / out_dtype");
  if (a->gate_mode != LIN_GATE_PER_HEAD && a->gate_mode != LIN_GATE_PER_KEY)
    return fail(LIN_EINVAL, "prefill: gate_mode");
  if (a->track_stride < 0 || (a->track_stride % 64) != 0)
    return fail(LIN_EINVAL, "prefill: track_stride must be 0 or a positive multiple of 64 (got %d)",
                a->track_stride);
  if (a->batch > 0 && (!a->cu_seqlens || !a->prefix_len || !a->slot || !a->has_initial_state))
    return fail(LIN_EINVAL, "prefill: cu_seqlens / prefix_len / slot / has_initial_state is NULL");
  if (a->total_tokens > 0 && (!a->x || !a->conv_w || !a->g || !a->beta || !a->out))
    return fail(LIN_EINVAL, "prefill: x / conv_w / g / beta / out is NULL");
  if (a->track_stride > 0 && a->batch > 0 && (!a->track_slots || !a->cu_track))
    return fail(LIN_EINVAL, "prefill: track_stride > 0 needs track_slots and cu_track");
  if (a->batch > 65535 && (a->flags & LIN_PREFILL_RECURRENT))
    return fail(LIN_EINVAL, "prefill: batch above 65535");
  return LIN_OK;
}

int lin_state_prefill_kernel(const lin_state_pool_t* pool, const lin_prefill_args_t* a) {
  int rc = check_prefill(pool, a);
  if (rc) return rc;
  if (!(a->flags & LIN_PREFILL_RECURRENT) && lin::chunked_prefill_supported(*pool, *a))
    return LIN_KERNEL_CHUNKED;
  return LIN_KERNEL_RECURRENT;
}

size_t lin_state_prefill_workspace(const lin_state_pool_t* pool, const lin_prefill_args_t* a) {
  if (check_prefill(pool, a)) return 0;
  if ((a->flags & LIN_PREFILL_RECURRENT) || !lin::chunked_prefill_supported(*pool, *a)) return 0;
  return lin::chunked_prefill_workspace(*pool, *a);
}

int lin_state_prefill(const lin_state_pool_t* pool, const lin_prefill_args_t* a, void* workspace,
                      size_t workspace_bytes, void* stream) {
  int rc = check_prefill(pool, a);
  if (rc) return rc;
  if (a->batch == 0) return ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (!(a->flags & LIN_PREFILL_RECURRENT) && lin::chunked_prefill_supported(*pool, *a)) {
    const size_t need = lin::chunked_prefill_workspace(*pool, *a);
    if (workspace_bytes < need || (need > 0 && !workspace))
      return fail(LIN_EWORKSPACE, "prefill: workspace of %zu bytes needed, %zu given", need,
                  workspace_bytes);
    e = lin::launch_prefill_chunked(*pool, *a, workspace, workspace_bytes, s);
  } else {
    if (a->batch > 65535) return fail(LIN_EINVAL, "prefill: batch above 65535");
    e = lin::launch_prefill_recurrent(*pool, *a, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_prefill launch");
  return ok();
}

int lin_state_prefill_noalloc(const lin_state_pool_t* pool, const lin_prefill_args_t* a,
                              void* stream) {
  int rc = check_prefill(pool, a);
  if (rc) return rc;
  if (a->batch == 0) return ok();
  // the fixed scratch bounds only the chunked kernel: its batch order (more
  // than one request) and its per-key rerun flags; the token-by-token kernel
  // takes what lin_state_prefill takes
  const bool chunked = !(a->flags & LIN_PREFILL_RECURRENT) && lin::chunked_prefill_supported(*pool, *a);
  if (chunked && a->batch > 1 && a->batch > lin::noalloc_max_batch())
    return fail(LIN_EINVAL, "prefill_noalloc: batch %d above the fixed scratch of %d requests",
                a->batch, lin::noalloc_max_batch());
  if (chunked && a->gate_mode == LIN_GATE_PER_KEY &&
      int64_t(a->batch) * pool->num_heads > lin::noalloc_max_pairs())
    return fail(LIN_EINVAL,
                "prefill_noalloc: %lld (request, head) pairs above the fixed scratch of %lld",
                static_cast<long long>(int64_t(a->batch) * pool->num_heads),
                static_cast<long long>(lin::noalloc_max_pairs()));
  if (!chunked && a->batch > 65535) return fail(LIN_EINVAL, "prefill: batch above 65535");
  cudaError_t e = lin::launch_prefill_noalloc(*pool, *a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_prefill_noalloc launch");
  return ok();
}

int lin_state_decode(const lin_state_pool_t* pool, const lin_decode_args_t* a, void* stream) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (!a) return fail(LIN_EINVAL, "decode args is NULL");
  if (a->layer < 0 || a->layer >= pool->num_layers)
    return fail(LIN_EINVAL, "decode: layer %d outside [0, %d)", a->layer, pool->num_layers);
  if (a->batch < 0 || a->batch > 65535) return fail(LIN_EINVAL, "decode: batch outside [0, 65535]");
  if (a->n_draft < 1) return fail(LIN_EINVAL, "decode: n_draft must be >= 1");
  if (!valid_dtype(a->io_dtype) || !valid_dtype(a->out_dtype))
    return fail(LIN_EINVAL, "decode: io_dtype / out_dtype");
  if (a->gate_mode != LIN_GATE_PER_HEAD && a->gate_mode != LIN_GATE_PER_KEY)
    return fail(LIN_EINVAL, "decode: gate_mode");
  if (a->track_interval < 0) return fail(LIN_EINVAL, "decode: negative track_interval");
  if (a->batch == 0) return ok();
  if (!a->x || !a->conv_w || !a->g || !a->beta || !a->out || !a->slot || !a->pos)
    return fail(LIN_EINVAL, "decode: x / conv_w / g / beta / out / slot / pos is NULL");
  if (!aligned16(a->x) || !aligned16(a->conv_w) || !aligned16(a->g) || !aligned16(a->out))
    return fail(LIN_EINVAL, "decode: x, conv_w, g and out must be 16-byte aligned");
  // n_draft > 1 with no spec buffer at all: a verify that writes outputs only
  const bool spec_less = a->spec.temporal == nullptr && a->spec.conv == nullptr;
  if (a->n_draft > 1 && !spec_less) {
    rc = check_spec(pool, a->spec, a->batch, a->n_draft, a->layer + 1);
    if (rc) return rc;
  }
  if (a->parent) {
    if (a->n_draft <= 1 || spec_less)
      return fail(LIN_EINVAL, "decode: a draft tree needs n_draft > 1 and a spec buffer");
    if (a->n_draft > 32)
      return fail(LIN_EUNSUPPORTED, "decode: a draft tree holds at most 32 drafts, not %d", a->n_draft);
  }
  if (lin::decode_stage_bytes(*pool, *a) > lin::kDecodeMaxStage)
    return fail(LIN_EUNSUPPORTED, "decode: n_draft %d stages %d bytes per (request, head), over %d",
                a->n_draft, lin::decode_stage_bytes(*pool, *a), lin::kDecodeMaxStage);
  cudaError_t e;
  if (a->n_draft > 1 && spec_less) {
    // outputs only: the drafts as one chunk from the slot state
    if (a->n_draft > lin::kVerifyChunkMaxDraft)
      return fail(LIN_EUNSUPPORTED, "decode: a verify without a spec buffer takes at most %d drafts, not %d",
                  lin::kVerifyChunkMaxDraft, a->n_draft);
    if (lin::verify_chunk_smem(*pool, *a) > 220 * 1024)
      return fail(LIN_EUNSUPPORTED, "decode: n_draft %d needs %d bytes of shared memory per (request, head)",
                  a->n_draft, lin::verify_chunk_smem(*pool, *a));
    e = lin::launch_verify_chunk(*pool, *a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "lin_state_decode launch");
    return ok();
  }
  e = lin::launch_decode(*pool, *a, nullptr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_decode launch");
  return ok();
}

int lin_state_replay_commit(const lin_state_pool_t* pool, const lin_replay_args_t* a, void* stream) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (!a) return fail(LIN_EINVAL, "replay commit args is NULL");
  if (a->layer < 0 || a->layer >= pool->num_layers)
    return fail(LIN_EINVAL, "replay commit: layer %d outside [0, %d)", a->layer, pool->num_layers);
  if (a->batch < 0 || a->batch > 65535) return fail(LIN_EINVAL, "replay commit: batch outside [0, 65535]");
  if (a->n_draft < 1) return fail(LIN_EINVAL, "replay commit: n_draft must be >= 1");
  if (!valid_dtype(a->io_dtype)) return fail(LIN_EINVAL, "replay commit: io_dtype");
  if (a->gate_mode != LIN_GATE_PER_HEAD && a->gate_mode != LIN_GATE_PER_KEY)
    return fail(LIN_EINVAL, "replay commit: gate_mode");
  if (a->track_interval < 0) return fail(LIN_EINVAL, "replay commit: negative track_interval");
  if (a->batch == 0) return ok();
  if (!a->x || !a->conv_w || !a->g || !a->beta || !a->slot || !a->pos || !a->accept_len)
    return fail(LIN_EINVAL, "replay commit: x / conv_w / g / beta / slot / pos / accept_len is NULL");
  if (!aligned16(a->x) || !aligned16(a->conv_w) || !aligned16(a->g))
    return fail(LIN_EINVAL, "replay commit: x, conv_w and g must be 16-byte aligned");
  lin_decode_args_t d;
  memset(&d, 0, sizeof(d));
  d.layer = a->layer;
  d.batch = a->batch;
  d.n_draft = a->n_draft;
  d.io_dtype = a->io_dtype;
  d.out_dtype = LIN_F32;  // no outputs are written
  d.gate_mode = a->gate_mode;
  d.flags = a->flags;
  d.q_scale = a->q_scale;
  d.track_interval = a->track_interval;
  d.x = a->x;
  d.conv_w = a->conv_w;
  d.g = a->g;
  d.beta = a->beta;
  d.out = nullptr;
  d.slot = a->slot;
  d.pos = a->pos;
  d.track_slot = a->track_slot;
  d.status = a->status;
  if (lin::decode_stage_bytes(*pool, d) > lin::kDecodeMaxStage)
    return fail(LIN_EUNSUPPORTED, "replay commit: n_draft %d stages %d bytes per (request, head), over %d",
                d.n_draft, lin::decode_stage_bytes(*pool, d), lin::kDecodeMaxStage);
  cudaError_t e = lin::launch_decode(*pool, d, a->accept_len, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_replay_commit launch");
  return ok();
}

int lin_state_spec_commit(const lin_state_pool_t* pool, const lin_commit_args_t* a, void* stream) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (!a) return fail(LIN_EINVAL, "commit args is NULL");
  if (a->layer_begin < 0 || a->layer_end > pool->num_layers || a->layer_begin > a->layer_end)
    return fail(LIN_EINVAL, "commit: bad layer range [%d, %d)", a->layer_begin, a->layer_end);
  if (a->batch < 0 || a->n_draft < 1 || a->track_interval < 0)
    return fail(LIN_EINVAL, "commit: batch / n_draft / track_interval");
  if (a->batch == 0 || a->layer_begin == a->layer_end) return ok();
  if (!a->slot || !a->pos || (a->parent ? !a->accept_node : !a->accept_len))
    return fail(LIN_EINVAL, "commit: slot / pos / accept_len (accept_node with a tree) is NULL");
  rc = check_spec(pool, a->spec, a->batch, a->n_draft, a->layer_end);
  if (rc) return rc;
  cudaError_t e = lin::launch_spec_commit(*pool, *a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_spec_commit launch");
  return ok();
}

int lin_state_copy_slots(const lin_state_pool_t* pool, const int32_t* src, const int32_t* dst,
                         int32_t n, int32_t layer_begin, int32_t layer_end, uint32_t flags,
                         int32_t* status, void* stream) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (n < 0) return fail(LIN_EINVAL, "copy_slots: negative n");
  if (layer_begin < 0 || layer_end > pool->num_layers || layer_begin > layer_end)
    return fail(LIN_EINVAL, "copy_slots: bad layer range [%d, %d)", layer_begin, layer_end);
  if (n == 0 || layer_begin == layer_end) return ok();
  if (!src || !dst) return fail(LIN_EINVAL, "copy_slots: src / dst is NULL");
  cudaError_t e = lin::launch_copy_slots(*pool, src, dst, n, layer_begin, layer_end, flags, status,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_copy_slots launch");
  return ok();
}

int lin_state_restore(const lin_state_pool_t* pool, const lin_cache_op_t* ops, int32_t n,
                      int64_t* has_initial_state, int32_t* status, void* stream) {
  int rc = check_pool(pool);
  if (rc) return rc;
  if (n < 0) return fail(LIN_EINVAL, "restore: negative n");
  if (n == 0) return ok();
  if (!ops || !has_initial_state) return fail(LIN_EINVAL, "restore: ops / has_initial_state is NULL");
  cudaError_t e = lin::launch_restore(*pool, ops, n, has_initial_state, status,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lin_state_restore launch");
  return ok();
}

}  // extern "C"
