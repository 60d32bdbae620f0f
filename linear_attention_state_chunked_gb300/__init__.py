"""Python binding of liblinstate.so, the GB300 state path of hybrid
linear-attention layers (GDN / KDA prefill, decode, speculative commit, slot
copies and restore).

The binding only marshals arguments: every step runs in the library's CUDA
kernels, and each function has the name of the C entry point it calls. PyTorch
provides device memory (the pool tensors, inputs, outputs) and streams. There
is no fallback: if the compiled library is missing the import fails.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblinstate.so")

# ---- constants (mirror include/lin_state.h) --------------------------------
LIN_OK, LIN_EINVAL, LIN_EUNSUPPORTED, LIN_ECUDA, LIN_EWORKSPACE = 0, -1, -2, -3, -4
LIN_F32, LIN_BF16 = 0, 1
LIN_GATE_PER_HEAD, LIN_GATE_PER_KEY = 0, 1
LIN_QK_L2NORM, LIN_CONV_SILU, LIN_VALIDATE, LIN_PREFILL_RECURRENT = 1, 2, 4, 8
LIN_PREFILL_SEGMENTED = 16
LIN_PREFILL_ONE_PIECE = 64
LIN_UPDATE_ADDITIVE = 32
LIN_ST_BAD_SLOT, LIN_ST_BAD_PREFIX, LIN_ST_TRACK_ALIAS, LIN_ST_BAD_SEQLEN = 1, 2, 4, 8
LIN_ST_COPY_ALIAS, LIN_ST_TIMEOUT, LIN_ST_BAD_ACCEPT = 16, 32, 64
LIN_ST_BAD_TREE = 256

LIN_KERNEL_RECURRENT, LIN_KERNEL_CHUNKED = 0, 1

EXPORTED = (
    "lin_state_prefill_kernel", "lin_state_prefill_workspace", "lin_state_prefill_noalloc", "lin_state_prefill", "lin_state_decode",
    "lin_state_spec_commit", "lin_state_replay_commit", "lin_state_copy_slots", "lin_state_restore",
    "lin_state_slot_bytes", "lin_state_read_status", "lin_state_strerror",
    "lin_state_last_error", "lin_state_version", "lin_state_selftest_mma",
)

_c_i32p = ctypes.c_void_p


class PoolT(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("num_heads", ctypes.c_int32), ("head_k", ctypes.c_int32), ("head_v", ctypes.c_int32),
        ("conv_channels", ctypes.c_int32), ("conv_width", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("conv_dtype", ctypes.c_int32),
        ("temporal", ctypes.c_void_p),
        ("temporal_layer_stride", ctypes.c_int64), ("temporal_slot_stride", ctypes.c_int64),
        ("conv", ctypes.c_void_p),
        ("conv_layer_stride", ctypes.c_int64), ("conv_slot_stride", ctypes.c_int64),
    ]


class PrefillArgsT(ctypes.Structure):
    _fields_ = [
        ("layer", ctypes.c_int32), ("batch", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
        ("io_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
        ("flags", ctypes.c_uint32), ("q_scale", ctypes.c_float), ("track_stride", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("conv_w", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
        ("slot", ctypes.c_void_p), ("has_initial_state", ctypes.c_void_p),
        ("track_slots", ctypes.c_void_p), ("cu_track", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


class SpecBufT(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_draft", ctypes.c_int32),
        ("temporal", ctypes.c_void_p),
        ("temporal_layer_stride", ctypes.c_int64), ("temporal_req_stride", ctypes.c_int64),
        ("temporal_step_stride", ctypes.c_int64),
        ("conv", ctypes.c_void_p),
        ("conv_layer_stride", ctypes.c_int64), ("conv_req_stride", ctypes.c_int64),
        ("conv_step_stride", ctypes.c_int64),
    ]


class DecodeArgsT(ctypes.Structure):
    _fields_ = [
        ("layer", ctypes.c_int32), ("batch", ctypes.c_int32), ("n_draft", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
        ("flags", ctypes.c_uint32), ("q_scale", ctypes.c_float), ("track_interval", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("conv_w", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("slot", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("track_slot", ctypes.c_void_p),
        ("spec", SpecBufT), ("status", ctypes.c_void_p), ("parent", ctypes.c_void_p),
    ]


class ReplayArgsT(ctypes.Structure):
    _fields_ = [
        ("layer", ctypes.c_int32), ("batch", ctypes.c_int32), ("n_draft", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32), ("gate_mode", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("q_scale", ctypes.c_float), ("track_interval", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("conv_w", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("slot", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("accept_len", ctypes.c_void_p), ("track_slot", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


class CommitArgsT(ctypes.Structure):
    _fields_ = [
        ("layer_begin", ctypes.c_int32), ("layer_end", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("n_draft", ctypes.c_int32),
        ("track_interval", ctypes.c_int32),
        ("slot", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("accept_len", ctypes.c_void_p),
        ("track_slot", ctypes.c_void_p), ("spec", SpecBufT), ("status", ctypes.c_void_p),
        ("parent", ctypes.c_void_p), ("accept_node", ctypes.c_void_p),
    ]


class CacheOpT(ctypes.Structure):
    _fields_ = [("linear_state_id", ctypes.c_int32), ("restore_requested", ctypes.c_int32),
                ("restore_src_slot_id", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.lin_state_prefill_kernel.argtypes = [P(PoolT), P(PrefillArgsT)]
    lib.lin_state_prefill_kernel.restype = ctypes.c_int
    lib.lin_state_prefill_workspace.argtypes = [P(PoolT), P(PrefillArgsT)]
    lib.lin_state_prefill_workspace.restype = ctypes.c_size_t
    lib.lin_state_prefill.argtypes = [P(PoolT), P(PrefillArgsT), vp, ctypes.c_size_t, vp]
    lib.lin_state_prefill.restype = ctypes.c_int
    lib.lin_state_prefill_noalloc.argtypes = [P(PoolT), P(PrefillArgsT), vp]
    lib.lin_state_prefill_noalloc.restype = ctypes.c_int
    lib.lin_state_decode.argtypes = [P(PoolT), P(DecodeArgsT), vp]
    lib.lin_state_decode.restype = ctypes.c_int
    lib.lin_state_spec_commit.argtypes = [P(PoolT), P(CommitArgsT), vp]
    lib.lin_state_spec_commit.restype = ctypes.c_int
    lib.lin_state_replay_commit.argtypes = [P(PoolT), P(ReplayArgsT), vp]
    lib.lin_state_replay_commit.restype = ctypes.c_int
    lib.lin_state_copy_slots.argtypes = [P(PoolT), vp, vp, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_uint32, vp, vp]
    lib.lin_state_copy_slots.restype = ctypes.c_int
    lib.lin_state_restore.argtypes = [P(PoolT), vp, ctypes.c_int32, vp, vp, vp]
    lib.lin_state_restore.restype = ctypes.c_int
    lib.lin_state_slot_bytes.argtypes = [P(PoolT)]
    lib.lin_state_slot_bytes.restype = ctypes.c_int64
    lib.lin_state_read_status.argtypes = [vp, P(ctypes.c_int32), vp]
    lib.lin_state_read_status.restype = ctypes.c_int
    lib.lin_state_strerror.argtypes = [ctypes.c_int]
    lib.lin_state_strerror.restype = ctypes.c_char_p
    lib.lin_state_last_error.argtypes = []
    lib.lin_state_last_error.restype = ctypes.c_char_p
    lib.lin_state_version.argtypes = []
    lib.lin_state_version.restype = ctypes.c_int
    lib.lin_state_selftest_mma.argtypes = [vp, vp, vp, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, vp, vp]
    lib.lin_state_selftest_mma.restype = ctypes.c_int
    return lib


lib = _load()


class LinStateError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib.lin_state_last_error().decode() or lib.lin_state_strerror(code).decode()
        super().__init__(f"{where}: {lib.lin_state_strerror(code).decode()} ({code}): {msg}")


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise LinStateError(rc, where)
    return rc


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_TORCH_DT = {LIN_F32: torch.float32, LIN_BF16: torch.bfloat16}


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return LIN_F32
    if dt == torch.bfloat16:
        return LIN_BF16
    raise ValueError(f"unsupported dtype {dt}")


class StatePool:
    """The slot-indexed state pool: temporal [L][S][H][V][K] and conv
    [L][S][C][3] torch tensors (layer-major, the layout of MambaPool in the
    MambaRadixCache page, 1.3), or views with any 16-byte-multiple strides.
    head_dim is K (key channels, the state row length); head_v is V (value
    channels, the state rows), K unless given."""

    def __init__(self, num_layers: int, num_slots: int, num_heads: int, head_dim: int,
                 state_dtype=torch.float32, conv_dtype=torch.bfloat16, device="cuda",
                 temporal: Optional[torch.Tensor] = None, conv: Optional[torch.Tensor] = None,
                 head_v: Optional[int] = None):
        H, D = num_heads, head_dim
        V = D if head_v is None else head_v
        C = 2 * H * D + H * V
        self.num_layers, self.num_slots, self.num_heads, self.head_dim = num_layers, num_slots, H, D
        self.head_k, self.head_v = D, V
        self.conv_channels = C
        if temporal is None:
            temporal = torch.zeros((num_layers, num_slots, H, V, D), dtype=state_dtype, device=device)
        if conv is None:
            conv = torch.zeros((num_layers, num_slots, C, 3), dtype=conv_dtype, device=device)
        self.temporal, self.conv = temporal, conv
        self._desc = None

    def desc(self) -> PoolT:
        t, c = self.temporal, self.conv
        es_t, es_c = t.element_size(), c.element_size()
        d = PoolT()
        d.num_layers, d.num_slots, d.num_heads = self.num_layers, self.num_slots, self.num_heads
        d.head_k, d.head_v = self.head_k, self.head_v
        d.conv_channels, d.conv_width = self.conv_channels, 4
        d.state_dtype, d.conv_dtype = dtype_code(t.dtype), dtype_code(c.dtype)
        d.temporal = t.data_ptr()
        d.temporal_layer_stride, d.temporal_slot_stride = t.stride(0) * es_t, t.stride(1) * es_t
        d.conv = c.data_ptr()
        d.conv_layer_stride, d.conv_slot_stride = c.stride(0) * es_c, c.stride(1) * es_c
        return d


class SpecBuffer:
    """Per-step verify states: temporal [L][B][D][H][V][K], conv [L][B][D][C][3]
    (the intermediate buffer of the MambaRadixCache page, 8.4)."""

    def __init__(self, pool: StatePool, max_batch: int, max_draft: int, num_layers=None):
        L = num_layers or pool.num_layers
        H, K, V, C = pool.num_heads, pool.head_k, pool.head_v, pool.conv_channels
        dev = pool.temporal.device
        self.temporal = torch.zeros((L, max_batch, max_draft, H, V, K), dtype=pool.temporal.dtype, device=dev)
        self.conv = torch.zeros((L, max_batch, max_draft, C, 3), dtype=pool.conv.dtype, device=dev)
        self.num_layers, self.max_batch, self.max_draft = L, max_batch, max_draft

    def desc(self) -> SpecBufT:
        t, c = self.temporal, self.conv
        et, ec = t.element_size(), c.element_size()
        s = SpecBufT()
        s.num_layers, s.max_batch, s.max_draft = self.num_layers, self.max_batch, self.max_draft
        s.temporal = t.data_ptr()
        s.temporal_layer_stride, s.temporal_req_stride, s.temporal_step_stride = (
            t.stride(0) * et, t.stride(1) * et, t.stride(2) * et)
        s.conv = c.data_ptr()
        s.conv_layer_stride, s.conv_req_stride, s.conv_step_stride = (
            c.stride(0) * ec, c.stride(1) * ec, c.stride(2) * ec)
        return s


# ---- entry points ------------------------------------------------------------

def _prefill_args(layer, x, conv_w, g, beta, out, cu_seqlens, prefix_len, slot,
                  has_initial_state, track_slots, cu_track, track_stride, gate_mode,
                  flags, q_scale, status) -> PrefillArgsT:
    a = PrefillArgsT()
    a.layer = layer
    a.batch = cu_seqlens.numel() - 1
    a.total_tokens = x.shape[0]
    a.io_dtype, a.out_dtype = dtype_code(x.dtype), dtype_code(out.dtype)
    a.gate_mode, a.flags, a.q_scale, a.track_stride = gate_mode, flags, q_scale, track_stride
    a.x, a.conv_w, a.g, a.beta, a.out = (t.data_ptr() for t in (x, conv_w, g, beta, out))
    a.cu_seqlens, a.prefix_len, a.slot = cu_seqlens.data_ptr(), prefix_len.data_ptr(), slot.data_ptr()
    a.has_initial_state = has_initial_state.data_ptr()
    a.track_slots = track_slots.data_ptr() if track_slots is not None else None
    a.cu_track = cu_track.data_ptr() if cu_track is not None else None
    a.status = status.data_ptr() if status is not None else None
    return a


def _kw_args(layer=0, *, x, conv_w, g, beta, out, cu_seqlens, prefix_len, slot,
             has_initial_state, track_slots=None, cu_track=None, track_stride=0,
             gate_mode=LIN_GATE_PER_KEY, flags=LIN_QK_L2NORM | LIN_CONV_SILU, q_scale=1.0,
             status=None, **_):
    return _prefill_args(layer, x, conv_w, g, beta, out, cu_seqlens, prefix_len, slot,
                         has_initial_state, track_slots, cu_track, track_stride, gate_mode,
                         flags, q_scale, status)


def lin_state_prefill_workspace(pool: StatePool, **kw) -> int:
    """Bytes of workspace lin_state_prefill needs (same keywords as the call)."""
    return int(lib.lin_state_prefill_workspace(ctypes.byref(pool.desc()),
                                               ctypes.byref(_kw_args(**kw))))


def lin_state_prefill_kernel(pool: StatePool, **kw) -> int:
    """LIN_KERNEL_CHUNKED or LIN_KERNEL_RECURRENT for these arguments."""
    return _check(int(lib.lin_state_prefill_kernel(ctypes.byref(pool.desc()),
                                                   ctypes.byref(_kw_args(**kw)))),
                  "lin_state_prefill_kernel")


def lin_state_prefill(pool: StatePool, *, layer: int, x, conv_w, g, beta, out, cu_seqlens,
                      prefix_len, slot, has_initial_state, track_slots=None, cu_track=None,
                      track_stride: int = 0, gate_mode: int = LIN_GATE_PER_KEY,
                      flags: int = LIN_QK_L2NORM | LIN_CONV_SILU, q_scale: float = 1.0,
                      status=None, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Calls lin_state_prefill. Tensors are device tensors in the layouts of
    include/lin_state.h. `workspace` is a uint8 device tensor of at least
    lin_state_prefill_workspace() bytes (allocated here when omitted)."""
    a = _prefill_args(layer, x, conv_w, g, beta, out, cu_seqlens, prefix_len, slot,
                      has_initial_state, track_slots, cu_track, track_stride, gate_mode,
                      flags, q_scale, status)
    pd = pool.desc()
    need = int(lib.lin_state_prefill_workspace(ctypes.byref(pd), ctypes.byref(a)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.lin_state_prefill(ctypes.byref(pd), ctypes.byref(a), _ptr(workspace), nbytes,
                                 _stream(stream)), "lin_state_prefill")


def lin_state_prefill_noalloc(pool: StatePool, *, layer: int, x, conv_w, g, beta, out,
                              cu_seqlens, prefix_len, slot, has_initial_state, track_slots=None,
                              cu_track=None, track_stride: int = 0,
                              gate_mode: int = LIN_GATE_PER_KEY,
                              flags: int = LIN_QK_L2NORM | LIN_CONV_SILU, q_scale: float = 1.0,
                              status=None, stream=None) -> None:
    """Calls lin_state_prefill_noalloc: the same prefill with no workspace and
    no allocation (its scratch is a fixed array inside the library)."""
    a = _prefill_args(layer, x, conv_w, g, beta, out, cu_seqlens, prefix_len, slot,
                      has_initial_state, track_slots, cu_track, track_stride, gate_mode,
                      flags, q_scale, status)
    _check(lib.lin_state_prefill_noalloc(ctypes.byref(pool.desc()), ctypes.byref(a),
                                         _stream(stream)), "lin_state_prefill_noalloc")


def lin_state_decode(pool: StatePool, *, layer: int, x, conv_w, g, beta, out, slot, pos,
                     track_slot=None, track_interval: int = 0, spec: Optional[SpecBuffer] = None,
                     gate_mode: int = LIN_GATE_PER_KEY, flags: int = LIN_QK_L2NORM | LIN_CONV_SILU,
                     q_scale: float = 1.0, status=None, stream=None, parent=None) -> None:
    """Calls lin_state_decode. x [B][n_draft][C]; with n_draft > 1 the per-step
    states go to `spec`, or, with spec None, only the outputs are written (the
    replay form: lin_state_replay_commit then runs the accepted prefix).
    parent [B][n_draft] int32 (with `spec`): a draft tree, draft j starting
    from the state after draft parent[r][j] (-1: the slot's)."""
    a = DecodeArgsT()
    a.layer, a.batch, a.n_draft = layer, x.shape[0], x.shape[1]
    a.io_dtype, a.out_dtype = dtype_code(x.dtype), dtype_code(out.dtype)
    a.gate_mode, a.flags, a.q_scale, a.track_interval = gate_mode, flags, q_scale, track_interval
    a.x, a.conv_w, a.g, a.beta, a.out = (t.data_ptr() for t in (x, conv_w, g, beta, out))
    a.slot, a.pos = slot.data_ptr(), pos.data_ptr()
    a.track_slot = track_slot.data_ptr() if track_slot is not None else None
    if spec is not None:
        a.spec = spec.desc()
    a.status = status.data_ptr() if status is not None else None
    a.parent = parent.data_ptr() if parent is not None else None
    _check(lib.lin_state_decode(ctypes.byref(pool.desc()), ctypes.byref(a), _stream(stream)),
           "lin_state_decode")


def lin_state_spec_commit(pool: StatePool, *, spec: SpecBuffer, slot, pos, accept_len=None,
                          n_draft: int, track_slot=None, track_interval: int = 0,
                          layer_begin: int = 0, layer_end: Optional[int] = None,
                          status=None, stream=None, parent=None, accept_node=None) -> None:
    """Calls lin_state_spec_commit: accept_len for a chain, or parent +
    accept_node (the last accepted node) for a draft tree."""
    a = CommitArgsT()
    a.layer_begin = layer_begin
    a.layer_end = pool.num_layers if layer_end is None else layer_end
    a.batch, a.n_draft, a.track_interval = slot.numel(), n_draft, track_interval
    a.slot, a.pos = slot.data_ptr(), pos.data_ptr()
    a.accept_len = accept_len.data_ptr() if accept_len is not None else None
    a.track_slot = track_slot.data_ptr() if track_slot is not None else None
    a.parent = parent.data_ptr() if parent is not None else None
    a.accept_node = accept_node.data_ptr() if accept_node is not None else None
    a.spec = spec.desc()
    a.status = status.data_ptr() if status is not None else None
    _check(lib.lin_state_spec_commit(ctypes.byref(pool.desc()), ctypes.byref(a), _stream(stream)),
           "lin_state_spec_commit")


def lin_state_replay_commit(pool: StatePool, *, layer: int, x, conv_w, g, beta, slot, pos,
                            accept_len, track_slot=None, track_interval: int = 0,
                            gate_mode: int = LIN_GATE_PER_KEY,
                            flags: int = LIN_QK_L2NORM | LIN_CONV_SILU, q_scale: float = 1.0,
                            status=None, stream=None) -> None:
    """Calls lin_state_replay_commit: runs the first accept_len[r] of request r's
    n_draft tokens (x [B][n_draft][C], the verify call's inputs) into its slot."""
    a = ReplayArgsT()
    a.layer, a.batch, a.n_draft = layer, x.shape[0], x.shape[1]
    a.io_dtype, a.gate_mode, a.flags = dtype_code(x.dtype), gate_mode, flags
    a.q_scale, a.track_interval = q_scale, track_interval
    a.x, a.conv_w, a.g, a.beta = (t.data_ptr() for t in (x, conv_w, g, beta))
    a.slot, a.pos, a.accept_len = slot.data_ptr(), pos.data_ptr(), accept_len.data_ptr()
    a.track_slot = track_slot.data_ptr() if track_slot is not None else None
    a.status = status.data_ptr() if status is not None else None
    _check(lib.lin_state_replay_commit(ctypes.byref(pool.desc()), ctypes.byref(a), _stream(stream)),
           "lin_state_replay_commit")


def lin_state_copy_slots(pool: StatePool, src, dst, layer_begin: int = 0,
                         layer_end: Optional[int] = None, flags: int = 0, status=None,
                         stream=None) -> None:
    le = pool.num_layers if layer_end is None else layer_end
    _check(lib.lin_state_copy_slots(ctypes.byref(pool.desc()), _ptr(src), _ptr(dst), src.numel(),
                                    layer_begin, le, flags, _ptr(status), _stream(stream)),
           "lin_state_copy_slots")


def lin_state_restore(pool: StatePool, ops, has_initial_state, status=None, stream=None) -> None:
    """ops: int32 device tensor [n][3] of (linear_state_id, restore_requested,
    restore_src_slot_id) records; has_initial_state: int64 device tensor [n]."""
    assert ops.dtype == torch.int32 and ops.shape[-1] == 3 and ops.is_contiguous()
    _check(lib.lin_state_restore(ctypes.byref(pool.desc()), _ptr(ops), ops.shape[0],
                                 _ptr(has_initial_state), _ptr(status), _stream(stream)),
           "lin_state_restore")


def lin_state_slot_bytes(pool: StatePool) -> int:
    return _check(int(lib.lin_state_slot_bytes(ctypes.byref(pool.desc()))), "lin_state_slot_bytes")


def lin_state_read_status(status: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib.lin_state_read_status(_ptr(status), ctypes.byref(v), _stream(stream)),
           "lin_state_read_status")
    return v.value


def lin_state_selftest_mma(A, B, D, a_mn=False, b_mn=False, bf16=False, status=None,
                           stream=None) -> None:
    """D[128][n] = A[128][k] B[n][k]^T on the tensor cores (layout self-test)."""
    flags = (1 if a_mn else 0) | (2 if b_mn else 0) | (4 if bf16 else 0)
    _check(lib.lin_state_selftest_mma(_ptr(A), _ptr(B), _ptr(D), B.shape[0], A.shape[1], flags,
                                      _ptr(status), _stream(stream)), "lin_state_selftest_mma")


def lin_state_version() -> int:
    return int(lib.lin_state_version())
