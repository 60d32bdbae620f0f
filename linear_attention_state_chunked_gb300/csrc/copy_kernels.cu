// Slot copies: fork / COW copy_from, restore, and speculative commit.
//
// MambaRadixCache page, 3.2: copy_from moves conv[:, src] and temporal[:, src]
// into dst for every linear layer. Qwen3.5 Linear-State Prefix Cache, 6.4:
// restore copies a checkpoint into the live slot across all layers and sets
// has_initial_state. MambaRadixCache page, 8.4 / 8.6: commit is
// main_state[slot] = buffer[accepted step], plus the ping-pong track slot when
// the accepted tokens cross the interval.
//
// All three are pure byte movers and HBM-bound. One CTA moves one 16 KB
// segment of one (item, layer) state block with 128-bit loads, four in flight
// per thread, and the grid covers items x layers x segments; there is no
// inter-CTA communication.

#include "common.cuh"
#include "internal.h"

namespace lin {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int64_t kSegBytes = int64_t(kCopyThreads) * kVecPerThread * 16;  // 16 KB

enum CopyMode { kModeCopy = 0, kModeRestore = 1, kModeCommit = 2 };

struct CopyParams {
  lin_state_pool_t pool;
  int mode;
  int32_t n_items;
  int32_t layer_begin, n_layers;
  int64_t t_bytes, c_bytes;  // bytes of one temporal / conv block
  int32_t segs_t, segs_c;
  uint32_t flags;
  int32_t* status;
  // copy
  const int32_t* src;
  const int32_t* dst;
  // restore
  const lin_cache_op_t* ops;
  int64_t* has_initial_state;
  // commit
  lin_commit_args_t commit;
};

// Moves `bytes` bytes (both pointers 16-byte aligned) starting at byte `off`.
__device__ __forceinline__ void move_segment(const char* __restrict__ s, char* __restrict__ d,
                                             int64_t off, int64_t bytes) {
  int64_t end = off + kSegBytes < bytes ? off + kSegBytes : bytes;
  int64_t nvec = (end - off) >> 4;
  const uint4* sv = reinterpret_cast<const uint4*>(s + off);
  uint4* dv = reinterpret_cast<uint4*>(d + off);
  uint4 r[kVecPerThread];
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    int64_t v = threadIdx.x + int64_t(i) * kCopyThreads;
    if (v < nvec) r[i] = __ldcs(sv + v);
  }
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    int64_t v = threadIdx.x + int64_t(i) * kCopyThreads;
    if (v < nvec) __stcs(dv + v, r[i]);
  }
  // A block whose size is not a multiple of 16 bytes: the tail byte by byte.
  int64_t tail0 = off + (nvec << 4);
  for (int64_t b = tail0 + threadIdx.x; b < end; b += kCopyThreads) d[b] = s[b];
}

__global__ void __launch_bounds__(kCopyThreads) slot_copy_kernel(CopyParams p) {
  const int segs = p.segs_t + p.segs_c;
  const int64_t bid = blockIdx.x;
  const int seg = static_cast<int>(bid % segs);
  const int64_t il = bid / segs;
  const int layer_rel = static_cast<int>(il % p.n_layers);
  const int item = static_cast<int>(il / p.n_layers);
  const int layer = p.layer_begin + layer_rel;
  const bool reporter = (seg == 0 && layer_rel == 0 && threadIdx.x == 0);
  const int ns = p.pool.num_slots;

  const char* src_t;
  const char* src_c;
  int dst_slot;
  const char* src2_t = nullptr;  // commit: the track slot's source and slot
  const char* src2_c = nullptr;
  int dst2_slot = -1;
  const char* pool_t = static_cast<const char*>(p.pool.temporal);
  const char* pool_c = static_cast<const char*>(p.pool.conv);

  if (p.mode == kModeCopy) {
    int s = p.src[item], d = p.dst[item];
    if (s < 0 || d < 0) return;
    if (s >= ns || d >= ns) {
      if (reporter) report(p.status, LIN_ST_BAD_SLOT);
      return;
    }
    if (s == d) return;
    if (p.flags & LIN_VALIDATE) {
      for (int j = 0; j < p.n_items; ++j) {
        if (j == item) continue;
        if (p.dst[j] == d || p.src[j] == d) {
          if (reporter) report(p.status, LIN_ST_COPY_ALIAS);
          return;
        }
      }
    }
    src_t = pool_t + layer * p.pool.temporal_layer_stride + s * p.pool.temporal_slot_stride;
    src_c = pool_c + layer * p.pool.conv_layer_stride + s * p.pool.conv_slot_stride;
    dst_slot = d;
  } else if (p.mode == kModeRestore) {
    lin_cache_op_t op = p.ops[item];
    if (op.linear_state_id < 0) return;
    if (op.linear_state_id >= ns) {
      if (reporter) {
        report(p.status, LIN_ST_BAD_SLOT);
        if (op.restore_requested) p.has_initial_state[item] = 0;
      }
      return;
    }
    if (!op.restore_requested) return;
    const int s = op.restore_src_slot_id;
    if (s < 0 || s >= ns) {
      if (reporter) p.has_initial_state[item] = 0;  // COLD_START
      return;
    }
    if (reporter) p.has_initial_state[item] = 1;  // RESTORED
    if (s == op.linear_state_id) return;
    src_t = pool_t + layer * p.pool.temporal_layer_stride + s * p.pool.temporal_slot_stride;
    src_c = pool_c + layer * p.pool.conv_layer_stride + s * p.pool.conv_slot_stride;
    dst_slot = op.linear_state_id;
  } else {  // kModeCommit: the live slot, and the track slot when a boundary is crossed
    const lin_commit_args_t& c = p.commit;
    const int32_t* par = c.parent ? c.parent + int64_t(item) * c.n_draft : nullptr;
    // the request's values, loaded together (no load waits on another)
    const int s = c.slot[item];
    const int a_in = par ? 0 : c.accept_len[item];
    const int node_in = par ? c.accept_node[item] : -1;
    const int ts = c.track_slot ? c.track_slot[item] : -1;
    const int pos = c.pos ? c.pos[item] : 0;
    if (s < 0) return;
    if (s >= ns) {
      if (reporter) report(p.status, LIN_ST_BAD_SLOT);
      return;
    }
    // the accepted path: drafts 0 .. a-1 of a chain, or a tree node and its
    // ancestors (each parent strictly earlier, so the walk ends in <= n_draft steps)
    int a, last;
    if (par) {
      last = node_in;
      if (last < -1 || last >= c.n_draft) {
        if (reporter) report(p.status, LIN_ST_BAD_TREE);
        return;
      }
      a = 0;
      for (int nd = last; nd >= 0; ++a) {
        const int up = par[nd];
        if (up < -1 || up >= nd) {
          if (reporter) report(p.status, LIN_ST_BAD_TREE);
          return;
        }
        nd = up;
      }
    } else {
      a = a_in;
      if (a < 0 || a > c.n_draft) {
        if (reporter) report(p.status, LIN_ST_BAD_ACCEPT);
        return;
      }
      last = a - 1;
    }
    if (a == 0) return;
    if (ts >= ns) {
      if (reporter) report(p.status, LIN_ST_BAD_SLOT);
      return;
    }
    if (ts == s) {
      if (reporter) report(p.status, LIN_ST_TRACK_ALIAS);
      return;
    }
    auto spec_t = [&](int step) {
      return static_cast<const char*>(c.spec.temporal) + layer * c.spec.temporal_layer_stride +
             item * c.spec.temporal_req_stride + step * c.spec.temporal_step_stride;
    };
    auto spec_c = [&](int step) {
      return static_cast<const char*>(c.spec.conv) + layer * c.spec.conv_layer_stride +
             item * c.spec.conv_req_stride + step * c.spec.conv_step_stride;
    };
    src_t = spec_t(last);
    src_c = spec_c(last);
    dst_slot = s;
    if (ts >= 0 && c.track_interval > 0) {
      const int nb = ((pos + a) / c.track_interval) * c.track_interval;
      if (nb > pos) {
        // the path's node at depth nb - pos: nb - pos - 1 in a chain, or the
        // accepted node's ancestor a - (nb - pos) levels up
        int step = nb - pos - 1;
        if (par) {
          step = last;
          for (int up = a - (nb - pos); up > 0; --up) step = par[step];
        }
        src2_t = spec_t(step);
        src2_c = spec_c(step);
        dst2_slot = ts;
      }
    }
  }

  char* dst_t = static_cast<char*>(p.pool.temporal) + layer * p.pool.temporal_layer_stride +
                dst_slot * p.pool.temporal_slot_stride;
  char* dst_c = static_cast<char*>(p.pool.conv) + layer * p.pool.conv_layer_stride +
                dst_slot * p.pool.conv_slot_stride;
  if (seg < p.segs_t)
    move_segment(src_t, dst_t, seg * kSegBytes, p.t_bytes);
  else
    move_segment(src_c, dst_c, (seg - p.segs_t) * kSegBytes, p.c_bytes);
  if (dst2_slot >= 0) {
    char* d2_t = static_cast<char*>(p.pool.temporal) + layer * p.pool.temporal_layer_stride +
                 dst2_slot * p.pool.temporal_slot_stride;
    char* d2_c = static_cast<char*>(p.pool.conv) + layer * p.pool.conv_layer_stride +
                 dst2_slot * p.pool.conv_slot_stride;
    if (seg < p.segs_t)
      move_segment(src2_t, d2_t, seg * kSegBytes, p.t_bytes);
    else
      move_segment(src2_c, d2_c, (seg - p.segs_t) * kSegBytes, p.c_bytes);
  }
}

CopyParams base_params(const lin_state_pool_t& pool, int mode, int32_t n, int32_t lb,
                       int32_t le) {
  CopyParams p{};
  p.pool = pool;
  p.mode = mode;
  p.n_items = n;
  p.layer_begin = lb;
  p.n_layers = le - lb;
  p.t_bytes = int64_t(pool.num_heads) * pool.head_v * pool.head_k * dtype_size(pool.state_dtype);
  p.c_bytes = int64_t(pool.conv_channels) * (pool.conv_width - 1) * dtype_size(pool.conv_dtype);
  p.segs_t = static_cast<int32_t>((p.t_bytes + kSegBytes - 1) / kSegBytes);
  p.segs_c = static_cast<int32_t>((p.c_bytes + kSegBytes - 1) / kSegBytes);
  return p;
}

cudaError_t launch(const CopyParams& p, cudaStream_t stream) {
  if (p.n_items <= 0 || p.n_layers <= 0) return cudaSuccess;
  int64_t blocks = int64_t(p.n_items) * p.n_layers * (p.segs_t + p.segs_c);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  slot_copy_kernel<<<static_cast<unsigned>(blocks), kCopyThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_copy_slots(const lin_state_pool_t& pool, const int32_t* src,
                              const int32_t* dst, int32_t n, int32_t layer_begin,
                              int32_t layer_end, uint32_t flags, int32_t* status,
                              cudaStream_t stream) {
  CopyParams p = base_params(pool, kModeCopy, n, layer_begin, layer_end);
  p.src = src;
  p.dst = dst;
  p.flags = flags;
  p.status = status;
  return launch(p, stream);
}

cudaError_t launch_restore(const lin_state_pool_t& pool, const lin_cache_op_t* ops,
                           int32_t n, int64_t* has_initial_state, int32_t* status,
                           cudaStream_t stream) {
  CopyParams p = base_params(pool, kModeRestore, n, 0, pool.num_layers);
  p.ops = ops;
  p.has_initial_state = has_initial_state;
  p.status = status;
  return launch(p, stream);
}

cudaError_t launch_spec_commit(const lin_state_pool_t& pool, const lin_commit_args_t& a,
                               cudaStream_t stream) {
  CopyParams p = base_params(pool, kModeCommit, a.batch, a.layer_begin, a.layer_end);
  p.commit = a;
  p.status = a.status;
  return launch(p, stream);
}

}  // namespace lin
