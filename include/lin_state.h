/*
 * lin_state.h -- C ABI of the GB300 (sm_103a) state path of hybrid
 * linear-attention layers: gated delta-rule (GDN / KDA) prefill over a
 * slot-indexed state pool, decode with speculative verify and commit, and
 * batched slot copies / restore.
 *
 * Sources (web pages, cited by title and section):
 *   [K3]  "企业官网建设流程全解析" (Kimi-K3 / SGLang mamba-ish notes):
 *         "状态通常包含什么" (conv state, temporal [HV, V, K]),
 *         "Linear的kv cache大小具体计算逻辑" (shapes, sizes),
 *         "Speculative decoding" (the KDA update), "--mamba-track-interval".
 *   [MRC] "SGLang之MambaRadixCache机制": 1.3 (pool), 3.2 (copy_from),
 *         3.4 (ping-pong track), 5.1 (decode), 8.3-8.6 (verify / commit).
 *   [PP]  "SGLang Mamba Radix Cache 深度解析：extra_buffer 模式的 Ping-Pong
 *         缓冲机制": parameters (chunk 64), chunk-boundary tracking, flows.
 *   [XL]  "Qwen3.5 Linear-State Prefix Cache": 2.2, 2.3, 5.1, 6.1, 6.4, 7.1.
 *
 * The update, per head, with S in R^{V x K}:
 *     S_t = S_{t-1} Diag(alpha_t) + d_t k_t^T,
 *     d_t = beta_t (v_t - S_{t-1} Diag(alpha_t) k_t),      o_t = S_t q_t
 * alpha_t = exp(g_t): one value per head (GDN) or per key channel (KDA).
 * q|k|v come out of a width-4 causal depthwise conv over the projection
 * inputs; the conv state is the last 3 inputs ([K3] "Conv state").
 *
 * Conventions for every call
 *   - Memory: every buffer belongs to the caller. Pointers marked "device"
 *     must be device memory of the current device; the library allocates
 *     nothing. Byte strides must be multiples of 16.
 *   - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).
 *     All calls only enqueue work on it; none synchronises, except
 *     lin_state_read_status. Index arrays live on the device and are never
 *     copied to the host.
 *   - Errors: a call returns LIN_OK (0) or a negative LIN_E* code when a host
 *     check fails; on failure nothing is enqueued and lin_state_last_error()
 *     gives the reason (thread-local). Errors only a kernel can see (a slot id
 *     out of range, a misaligned prefix, ...) set LIN_ST_* bits in the
 *     optional device word `status` (atomic OR; NULL = not reported) and the
 *     offending item is skipped; the rest of the batch completes.
 *   - Slot ids: valid ids are [0, num_slots). A negative slot id marks a
 *     padding entry and is a no-op ([XL] 6.1: ids default to -1).
 */
#ifndef LIN_STATE_H_
#define LIN_STATE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LIN_API __attribute__((visibility("default")))
#else
#define LIN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define LIN_OK 0
#define LIN_EINVAL (-1)        /* bad argument: NULL, bad dtype, stride, size */
#define LIN_EUNSUPPORTED (-2)  /* valid but not implemented: head dims, ...   */
#define LIN_ECUDA (-3)         /* a CUDA runtime call failed                  */
#define LIN_EWORKSPACE (-4)    /* workspace smaller than the query asked for  */

/* ---- device status bits (OR-ed into *status) --------------------------- */
#define LIN_ST_BAD_SLOT 1      /* slot / track slot id >= num_slots            */
#define LIN_ST_BAD_PREFIX 2    /* prefill prefix_len < 0 or not a multiple of 64 */
#define LIN_ST_TRACK_ALIAS 4   /* a track slot equals the request's live slot  */
#define LIN_ST_BAD_SEQLEN 8    /* cu_seqlens not monotone or past total_tokens */
#define LIN_ST_COPY_ALIAS 16   /* LIN_VALIDATE: a copy dst is another pair's dst or src */
#define LIN_ST_TIMEOUT 32      /* a bounded device wait gave up               */
#define LIN_ST_BAD_ACCEPT 64   /* commit accept_len outside [0, n_draft]      */
#define LIN_ST_BAD_TREE 256    /* a draft's parent outside [-1, j), or an
                                  accepted node outside [-1, n_draft)         */

/* ---- enums ------------------------------------------------------------- */
typedef enum { LIN_F32 = 0, LIN_BF16 = 1 } lin_dtype_t;
/* GDN: alpha is one scalar per head; KDA: one value per key channel
   ([K3] "g": GDN g has shape [..,H], KDA g has 128 values per head). */
typedef enum { LIN_GATE_PER_HEAD = 0, LIN_GATE_PER_KEY = 1 } lin_gate_t;

enum {
  LIN_QK_L2NORM = 1u,        /* L2-normalise q and k per head, eps 1e-6 inside the sqrt */
  LIN_CONV_SILU = 2u,        /* SiLU on the conv output                        */
  LIN_VALIDATE = 4u,         /* extra device checks (copy aliasing)            */
  LIN_PREFILL_RECURRENT = 8u, /* prefill: force the token-by-token kernel      */
  LIN_PREFILL_SEGMENTED = 16u, /* prefill: run a batch of one request in segments
                                 even when it is short (see lin_state_prefill) */
  LIN_UPDATE_ADDITIVE = 32u,  /* prefill, decode, verify, replay: the additive
                                 (Mamba2 SSD) update S' = S Diag(alpha) + beta v k^T
                                 with no delta correction ([MRC] 9.3: S_new =
                                 A S_old + B x; alpha = exp(dt A), beta = dt,
                                 k = B, v = x, q = C); the pool, tracking,
                                 verify and commit work unchanged */
  LIN_PREFILL_ONE_PIECE = 64u  /* prefill, chunked kernel: every (request, head)
                                 in one piece on one SM, no wrap-around
                                 schedule (see lin_state_prefill); same results */
};

/* ---- the state pool ([MRC] 1.3; [K3] shapes) ----------------------------
 * temporal: base of [num_layers][num_slots][H][V][K] in state_dtype; the
 *   inner [H][V][K] block of one (layer, slot) is contiguous, row v holds the
 *   K key channels of S. Layer and slot strides are given in bytes.
 * conv: base of [num_layers][num_slots][C][conv_width-1] in conv_dtype; the
 *   inner [C][3] block is contiguous, [c][0] is the oldest input.
 * C = conv_channels = 2*H*K + H*V, ordered q | k | v, head-major inside each.
 * Requirements: conv_width == 4; (head_k, head_v) one of (16,16), (32,32),
 * (64,64), (128,128), or (128,64) (128 key channels with 64 value channels:
 * the SSD head, state size 128 and head dim 64). Anything else is
 * LIN_EUNSUPPORTED. */
typedef struct {
  int32_t num_layers, num_slots, num_heads, head_k, head_v;
  int32_t conv_channels, conv_width;
  int32_t state_dtype, conv_dtype; /* lin_dtype_t */
  void* temporal;                  /* device */
  int64_t temporal_layer_stride, temporal_slot_stride;
  void* conv;                      /* device */
  int64_t conv_layer_stride, conv_slot_stride;
} lin_state_pool_t;

/* ---- prefill ------------------------------------------------------------
 * For each request r of a varlen batch: start from slot[r] if
 * has_initial_state[r] != 0, else from zero state and zero conv window
 * ([XL] 5.1 step 5, 6.4); run its tokens x[cu_seqlens[r] .. cu_seqlens[r+1]);
 * at every absolute position b = prefix_len[r] + i + 1 with
 * b % track_stride == 0, copy (state, conv window) into
 * track_slots[cu_track[r] + (j mod n_r)], j = 0, 1, ... counted within this
 * call, n_r = cu_track[r+1] - cu_track[r] ([PP] chunk-boundary tracking;
 * a two-entry list is the ping-pong pair of [MRC] 3.4; the caller rotates it
 * between calls); finally write the state and conv window back into slot[r].
 * The state is carried in fp32 inside the call and rounded (RNE) to the
 * pool dtype where it is stored. Chunks align to absolute multiples of 64,
 * so prefix_len[r] must be a multiple of 64 ([PP]: FLA 64-token alignment);
 * otherwise the request is skipped with LIN_ST_BAD_PREFIX.
 * Inputs (device): x [T][C] io_dtype (q|k|v projection inputs before the
 * conv), conv_w [C][4] io_dtype (conv_w[c][3] multiplies the current token,
 * no bias), g fp32 log(alpha) [T][H] (GDN) or [T][H][K] (KDA), beta fp32
 * [T][H] (already through the sigmoid); out [T][H][V] out_dtype.
 * cu_seqlens [batch+1], prefix_len [batch], slot [batch], cu_track
 * [batch+1] int32; has_initial_state [batch] int64 (the array
 * lin_state_restore writes); track_slots int32 (NULL if track_stride == 0).
 * track_stride: 0 = no snapshots, else a positive multiple of 64.
 * A negative entry in a track list skips that snapshot. Requests must use
 * distinct live slots; a track slot equal to the live slot is rejected
 * (LIN_ST_TRACK_ALIAS). Workspace: lin_state_prefill_workspace() bytes of
 * device memory (may be 0 -> workspace may be NULL).
 * Per-key (KDA) gates on the chunked kernel: the chunk factors each key
 * channel's decay around the chunk's middle row, which holds while no channel
 * decays by more than e^80 across half a chunk (a mean log-decay above about
 * -2.5 per token). A (request, head) beyond that stops before it stores its
 * state and is rerun token by token by a launch the call queues behind the
 * chunked one (it runs only such pairs and needs no host synchronisation),
 * so every valid g gives a valid result.
 * Precision: the chunked kernel carries the state in fp32; its tensor-core
 * operands are fp16 with high / low splits where the pool is fp32 (and for
 * per-head gates), so outputs and states of an fp32 pool stay within a few
 * 1e-4 (relative L2 per request and head) of an exact computation; a bf16
 * pool with per-key gates takes bf16 operands. The conv's SiLU is computed as
 * (y/2)(1 + tanh(y/2)) with a hardware tanh (relative error about 2^-11). The
 * token-by-token kernel computes in fp32 throughout.
 * Long single requests: with the chunked kernel, a batch of one request
 * whose heads alone cannot fill the GPU (heads x 4 <= SMs, >= 4096 tokens
 * by total_tokens; any request of >= 8 chunks with LIN_PREFILL_SEGMENTED)
 * runs in segments: the state after a segment is affine in the state before
 * it (S M + B), so every segment's offset B (from a zero state) and
 * transition M (from the identity, with zero values) are computed in
 * parallel, a scan carries the true state across segments (fp32), and every
 * segment then runs in parallel from its true initial state; with a cycled
 * track list only the snapshots that remain at the end in token order (the
 * request's last n_r) are written, so the slots end up as in one piece. The workspace
 * then holds 2 fp32 states per (segment, head).
 * Batches with more (request, head) pairs than SMs (up to 4096 requests and
 * 8192 pairs plus SMs): with the chunked kernel, the pairs' chunk chains are
 * laid end to end and cut into one range of equal chunk units per SM
 * (McNaughton's wrap-around rule), so the SMs finish together instead of in
 * rounds of whole requests. A chain crossing a range boundary runs as two
 * pieces: the first hands its fp32 state (through the workspace) to the
 * second, which waits for it (bounded: LIN_ST_TIMEOUT after about 4 s). A
 * one-CTA plan kernel orders the pieces by planned start and the CTAs take
 * them from a counter, so a wait is always for a piece already running; no
 * co-residency is assumed. The results equal the one-piece schedule's bit for
 * bit; LIN_PREFILL_ONE_PIECE selects that schedule. The workspace then holds
 * the plan and one fp32 state per SM (about 10 MB on 152 SMs). Less workspace than the
 * query reports is an error (LIN_EWORKSPACE); lin_state_prefill_noalloc runs
 * the request in one piece. The workspace also holds the longest-first order
 * of a varlen batch and, for per-key gates, one rerun bit per (request, head). */
typedef struct {
  int32_t layer;
  int32_t batch;
  int64_t total_tokens;
  int32_t io_dtype;   /* lin_dtype_t of x and conv_w */
  int32_t out_dtype;  /* lin_dtype_t of out */
  int32_t gate_mode;  /* lin_gate_t */
  uint32_t flags;
  float q_scale;      /* multiplies q after the L2 norm; 1.0 = none */
  int32_t track_stride;
  const void* x;
  const void* conv_w;
  const float* g;
  const float* beta;
  void* out;
  const int32_t* cu_seqlens;
  const int32_t* prefix_len;
  const int32_t* slot;
  const int64_t* has_initial_state;
  const int32_t* track_slots;
  const int32_t* cu_track;
  int32_t* status;
} lin_prefill_args_t;

/* Which kernel lin_state_prefill would run for these arguments:
 * LIN_KERNEL_CHUNKED (the tensor-core chunked kernel: head_k == 128 and
 * head_v 128 or 64, bf16 x)
 * or LIN_KERNEL_RECURRENT (token by token; any supported head dim, or when
 * LIN_PREFILL_RECURRENT is set). A negative LIN_E* code for invalid args. */
#define LIN_KERNEL_RECURRENT 0
#define LIN_KERNEL_CHUNKED 1
LIN_API int lin_state_prefill_kernel(const lin_state_pool_t* pool, const lin_prefill_args_t* args);

LIN_API size_t lin_state_prefill_workspace(const lin_state_pool_t* pool,
                                   const lin_prefill_args_t* args);
LIN_API int lin_state_prefill(const lin_state_pool_t* pool, const lin_prefill_args_t* args,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Prefill that allocates nothing and takes no workspace. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory during a step: serving engines that give all device memory to their
 * own pools at start-up (so an extra allocation fails or fragments it) and
 * loops that must not pay the device-wide synchronisation of cudaMalloc /
 * cudaFree. Same arguments as lin_state_prefill; the results are the same
 * within rounding (a batch equal bit for bit), except that a batch of one long
 * request runs in one piece, not in segments: the same values within the
 * fp32 / bf16 tolerances, but on only `heads` CTAs, so much slower than
 * lin_state_prefill for such a request; likewise every (request, head) runs
 * in one piece, not under the wrap-around schedule. Its scratch (the longest-first order
 * of a batch, the per-key rerun bits) is fixed arrays in the library's device
 * memory (48 KB), held by every GPU that loads the library until the process
 * exits:
 *   - on the chunked kernel, batches of more than one request above 4096
 *     requests, and per-key gates with more than 262,144 (request, head)
 *     pairs, are rejected with LIN_EINVAL; the token-by-token kernel has
 *     lin_state_prefill's limits;
 *   - the first call on a device looks up the arrays' device addresses with
 *     the device current (and again in a new context of that device, e.g.
 *     after cudaDeviceReset), so make the first call before any stream capture;
 *   - all calls share the arrays, so calls that overlap on the GPU (different
 *     streams, no ordering between them) race on them; each call clears what
 *     must start at zero. */
LIN_API int lin_state_prefill_noalloc(const lin_state_pool_t* pool,
                                      const lin_prefill_args_t* args, void* stream);

/* ---- speculative per-step buffer ([MRC] 8.4) ----------------------------
 * temporal: [layers][max_batch][max_draft][H][V][K] in the pool's state
 * dtype; conv: [layers][max_batch][max_draft][C][3] in the pool's conv
 * dtype; strides in bytes. Buffer row r belongs to the r-th request of the
 * decode / commit batch. decode needs layer < num_layers, commit needs
 * layer_end <= num_layers. */
typedef struct {
  int32_t num_layers, max_batch, max_draft;
  void* temporal; /* device */
  int64_t temporal_layer_stride, temporal_req_stride, temporal_step_stride;
  void* conv;     /* device */
  int64_t conv_layer_stride, conv_req_stride, conv_step_stride;
} lin_spec_buf_t;

/* ---- decode -------------------------------------------------------------
 * Each request r advances n_draft tokens from the state in slot[r] of
 * `layer`. pos[r] = tokens already folded into that state.
 * n_draft == 1: the state is updated in place ([MRC] 5.1); when the state
 *   then covers n = pos[r] + 1 tokens with n % track_interval == 0 and
 *   track_slot[r] >= 0, it is also copied into track_slot[r] ([K3]
 *   "--mamba-track-interval": prompt 1000, interval 256 -> 1024, 1280, ...).
 * n_draft > 1 (verify, [MRC] 8.3): the tokens run in order from the slot
 *   state; the state after draft step j goes to spec row r, step j; the slot
 *   is not modified and nothing is tracked (commit does that). With no spec
 *   buffer (spec.temporal and spec.conv both NULL) only the outputs are
 *   written: the replay form of speculative decoding, where
 *   lin_state_replay_commit later re-runs the accepted prefix ([K3]
 *   "ReplaySSM"; [MRC] 9).
 * The state is rounded to the pool dtype after every token, so a verify
 *   step equals the same number of single-token decodes bit for bit.
 * Inputs (device): x [batch][n_draft][C] io_dtype, g [batch][n_draft][H]
 * or [..][H][K] fp32, beta [batch][n_draft][H] fp32, out
 * [batch][n_draft][H][V] out_dtype; slot, pos [batch] int32; track_slot
 * [batch] int32 or NULL. Live slots must be distinct within the batch.
 * x, conv_w, g and out move by bulk async copies and must be 16-byte
 * aligned (LIN_EINVAL otherwise).
 * One (request, head) stages its state block, conv window, taps and n_draft
 * x (and per-key g) rows in shared memory; past 110 KB of staging the call
 * returns LIN_EUNSUPPORTED (head 128, fp32 state, conv and io, per-key
 * gates: n_draft <= 17). */
typedef struct {
  int32_t layer;
  int32_t batch;
  int32_t n_draft;
  int32_t io_dtype;  /* x, conv_w */
  int32_t out_dtype; /* out */
  int32_t gate_mode;
  uint32_t flags;
  float q_scale;
  int32_t track_interval; /* 0 = never track */
  const void* x;
  const void* conv_w;
  const float* g;
  const float* beta;
  void* out;
  const int32_t* slot;
  const int32_t* pos;
  const int32_t* track_slot;
  lin_spec_buf_t spec; /* used when n_draft > 1 */
  int32_t* status;
  /* Draft tree ([MRC] 8.3, 9.6 retrieve_parent_token): device [batch][n_draft]
   * int32, or NULL for a linear chain. With a spec buffer and n_draft <= 32,
   * draft j of request r starts from the state and conv window after draft
   * parent[r][j] (-1: the slot's); parent[r][j] must lie in [-1, j), else the
   * request is skipped with LIN_ST_BAD_TREE. */
  const int32_t* parent;
} lin_decode_args_t;

LIN_API int lin_state_decode(const lin_state_pool_t* pool, const lin_decode_args_t* args,
                     void* stream);

/* ---- speculative commit / rollback ([MRC] 8.4, 8.6) ---------------------
 * For every layer in [layer_begin, layer_end) and request r with
 * a = accept_len[r] in 1..n_draft: slot[r] <- spec row r, step a-1
 * (main_state = buffer[accepted step]). When (pos[r], pos[r] + a] holds a
 * multiple of track_interval and track_slot[r] >= 0, the state at the
 * largest such multiple n (spec step n - pos[r] - 1) is also copied into
 * track_slot[r] ([MRC] 8.6: crossing the interval also updates the
 * ping-pong buffer). a == 0 changes nothing (full rollback). */
typedef struct {
  int32_t layer_begin, layer_end;
  int32_t batch;
  int32_t n_draft;
  int32_t track_interval;
  const int32_t* slot;       /* device [batch] */
  const int32_t* pos;        /* device [batch] */
  const int32_t* accept_len; /* device [batch] */
  const int32_t* track_slot; /* device [batch] or NULL */
  lin_spec_buf_t spec;
  int32_t* status;
  /* Draft tree: parent as in lin_decode_args_t (device [batch][n_draft]) and
   * accept_node (device [batch]): the last node of the accepted path (-1:
   * nothing), whose length then plays the part of accept_len (accept_len is
   * not read); the boundary snapshot comes from the path's node at that
   * depth. NULL parent: the linear chain above. */
  const int32_t* parent;
  const int32_t* accept_node;
} lin_commit_args_t;

LIN_API int lin_state_spec_commit(const lin_state_pool_t* pool, const lin_commit_args_t* args,
                          void* stream);

/* ---- replay commit ([K3] "ReplaySSM" exact-fold; [MRC] 9.2 - 9.10) -------
 * The commit of a verify that kept no per-step states: for each request r,
 * the first a = accept_len[r] (0..n_draft) of its n_draft draft tokens run
 * again, in order, from the state in slot[r] of `layer`, with the same inputs
 * the verify call had (x [batch][n_draft][C], g, beta as in lin_decode_args_t;
 * only the accepted rows are read), and the state and conv window after them
 * replace the slot's; no outputs are written. A boundary crossed on the way
 * ((pos[r] + j + 1) % track_interval == 0, track_slot[r] >= 0) snapshots the
 * state and window there into track_slot[r] ([MRC] 9.10), so the track slot
 * ends up as lin_state_spec_commit leaves it. The arithmetic is the decode
 * kernel's, token by token with the state rounded to the pool dtype after
 * each token, so the slot equals what the per-step-state path commits, bit
 * for bit. a == 0 leaves the slot unchanged. x, conv_w, g must be 16-byte
 * aligned; the staging limit of lin_state_decode applies to n_draft. */
typedef struct {
  int32_t layer;
  int32_t batch;
  int32_t n_draft;
  int32_t io_dtype;  /* x, conv_w */
  int32_t gate_mode;
  uint32_t flags;
  float q_scale;
  int32_t track_interval; /* 0 = never track */
  const void* x;
  const void* conv_w;
  const float* g;
  const float* beta;
  const int32_t* slot;       /* device [batch] */
  const int32_t* pos;        /* device [batch]: tokens already in the slot's state */
  const int32_t* accept_len; /* device [batch] */
  const int32_t* track_slot; /* device [batch] or NULL */
  int32_t* status;
} lin_replay_args_t;

LIN_API int lin_state_replay_commit(const lin_state_pool_t* pool, const lin_replay_args_t* args,
                                    void* stream);

/* ---- batched slot copies ([MRC] 3.2 copy_from / COW; [PP] fork_from) ----
 * For i < n and every layer in [layer_begin, layer_end):
 *   conv[l][dst[i]] = conv[l][src[i]]; temporal[l][dst[i]] = temporal[l][src[i]].
 * src, dst: device int32 [n]. A pair with a negative id is skipped;
 * src == dst is a no-op. A dst may appear once and may not also be a src
 * in the same batch (otherwise the result is undefined); srcs may repeat
 * (one checkpoint forked many times). With LIN_VALIDATE in flags such
 * pairs are detected, skipped and reported as LIN_ST_COPY_ALIAS. */
LIN_API int lin_state_copy_slots(const lin_state_pool_t* pool, const int32_t* src,
                         const int32_t* dst, int32_t n, int32_t layer_begin,
                         int32_t layer_end, uint32_t flags, int32_t* status,
                         void* stream);

/* ---- restore ([XL] 6.1 LinearStateCacheOp, 6.4 restore_linear_state_slots)
 * For op i: live = linear_state_id (negative = padding, skipped).
 *   restore_requested and 0 <= restore_src_slot_id < num_slots:
 *       copy the source into the live slot across all layers,
 *       has_initial_state[i] = 1 (RESTORED, warm);
 *   restore_requested and the source does not resolve:
 *       has_initial_state[i] = 0 (COLD_START);
 *   not requested: has_initial_state[i] is left as it was.
 * ops: device array of n records; has_initial_state: device int64 [n].
 * The copy is enqueued on `stream`, so it is ordered before a prefill
 * enqueued after it on the same stream ([XL] 7.1). */
typedef struct {
  int32_t linear_state_id;
  int32_t restore_requested; /* 0 / 1 */
  int32_t restore_src_slot_id;
} lin_cache_op_t;

LIN_API int lin_state_restore(const lin_state_pool_t* pool, const lin_cache_op_t* ops,
                      int32_t n, int64_t* has_initial_state, int32_t* status,
                      void* stream);

/* ---- helpers ------------------------------------------------------------ */
/* Bytes of one slot over all layers: num_layers * (H*V*K*size(state_dtype)
 * + C*(conv_width-1)*size(conv_dtype)); e.g. 29,039,616 for the Kimi-K3 TP8
 * shard over 69 layers in bf16 ([K3]: 25.9 MB SSM + 1.82 MB conv).
 * Returns a negative LIN_E* code for an invalid descriptor. */
LIN_API int64_t lin_state_slot_bytes(const lin_state_pool_t* pool);

/* Synchronises `stream`, copies the device status word into *value and
 * clears the device word. */
LIN_API int lin_state_read_status(int32_t* status, int32_t* value, void* stream);

/* Static text for a LIN_E* code. */
LIN_API const char* lin_state_strerror(int code);
/* Text of the last host-side error on this thread ("" if none). */
LIN_API const char* lin_state_last_error(void);
/* Diagnostic: checks on the current device the tensor-core operand layouts
 * the chunked prefill uses. Computes D[128][n] = A[128][k] * B[n][k]^T in one
 * CTA with tcgen05.mma, operands rounded to fp16 (or bf16 with flags & 4) and
 * staged in shared memory K-major, or MN-major for A (flags & 1) / B
 * (flags & 2); fp32 accumulation. A, B, D: device fp32, row-major.
 * n in {32, 64, 128}, k a multiple of 16 in [16, 128]. */
LIN_API int lin_state_selftest_mma(const float* A, const float* B, float* D, int32_t n, int32_t k,
                                   int32_t flags, int32_t* status, void* stream);

/* ABI version: (major << 16) | minor. */
LIN_API int lin_state_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LIN_STATE_H_ */
