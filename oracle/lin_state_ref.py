"""ctypes front end of lin_state_ref.c, the plain C restatement of the oracle's
token recurrence, compiled for float64 (checked against the numpy oracle in
lin_state_oracle.py) and float32 (the CPU baseline the benchmark times on all
host cores).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU legs may import this module. The library never imports it and shares no
code with it.

The dict-level functions (prefill, decode) take and update the numpy oracle's
pool dict and return what the numpy oracle returns; the *_arrays functions
work on contiguous arrays of one layer in the working precision and are what
the benchmark times.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lin_state_ref.c")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liblinstate_ref.so")

ROUND = {"f64": 0, "f32": 1, "bf16": 2}
DTYPE = {"f64": np.float64, "f32": np.float32}


def build(force: bool = False) -> str:
    """Compiles the float64 and float32 forms of lin_state_ref.c into one
    shared library (gcc, -O2, POSIX threads)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-fPIC", "-pthread", "-c", SRC]
    o64, o32 = os.path.join(BUILD, "ref_f64.o"), os.path.join(BUILD, "ref_f32.o")
    subprocess.run(base + ["-DREAL=double", "-DSUFFIX=f64", "-o", o64], check=True)
    subprocess.run(base + ["-DREAL=float", "-DREAL_FLOAT", "-DSUFFIX=f32", "-o", o32], check=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.run([cc, "-shared", "-pthread", "-o", tmp, o64, o32, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        for sfx in ("f64", "f32"):
            f = getattr(_lib, f"lin_ref_prefill_{sfx}")
            f.argtypes = [I, I, I, I, I, P, P, I, I, P, P, P, P, I, I64, P, P, P, P, P, P, I, I, I, D,
                          I, P, I]
            f.restype = I
            f = getattr(_lib, f"lin_ref_decode_{sfx}")
            f.argtypes = [I, I, I, I, I, P, P, I, I, P, P, P, P, I, I, P, P, P, I, I, I, D, I, P, P, P,
                          I]
            f.restype = I
            f = getattr(_lib, f"lin_ref_commit_{sfx}")
            f.argtypes = [I, I, I, I, P, P, I, I, P, P, P, P, I, P, P]
            f.restype = None
            f = getattr(_lib, f"lin_ref_copy_slots_{sfx}")
            f.argtypes = [P, I64, I64, I64, I, I, P, P, I]
            f.restype = None
    return _lib


def host_threads() -> int:
    return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name as /proc/cpuinfo gives it (Arm hosts give an
    implementer / part pair instead of a name)."""
    try:
        with open("/proc/cpuinfo") as fh:
            info = fh.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "cpu model"):
        for line in info.splitlines():
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    impl = part = None
    for line in info.splitlines():
        k = line.split(":")[0].strip()
        if k == "CPU implementer" and impl is None:
            impl = line.split(":", 1)[1].strip()
        if k == "CPU part" and part is None:
            part = line.split(":", 1)[1].strip()
    return f"implementer {impl}, part {part}" if impl else "unknown"


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i64(v):
    return None if v is None else np.ascontiguousarray(np.asarray(v, np.int64))


def _arr(a, dt):
    return np.ascontiguousarray(np.asarray(a, dt))


# ----------------------------------------------------------------------------
# array level: one layer of the pool, in the working precision
# ----------------------------------------------------------------------------

def prefill_arrays(prec, temporal, conv, x, conv_w, g, beta, cu_seqlens, prefix_len, slot,
                   has_initial_state, track_slots, cu_track, track_stride, gate_mode, flags,
                   q_scale, out, state_round, conv_round, out_round, nthreads=None):
    """temporal [slots][H][V][K], conv [slots][C][3], out [T][H][V]: contiguous
    arrays of the working precision (updated in place). Returns the status."""
    dt = DTYPE[prec]
    for a in (temporal, conv, x, conv_w, g, beta, out):
        assert a.dtype == dt and a.flags.c_contiguous
    S, H, V, K = temporal.shape
    C = conv.shape[1]
    cu, pre, sl, warm = (_i64(v) for v in (cu_seqlens, prefix_len, slot, has_initial_state))
    tr = _i64(track_slots) if track_stride and track_slots is not None and len(track_slots) else None
    ctr = _i64(cu_track) if tr is not None else None
    f = getattr(lib(), f"lin_ref_prefill_{prec}")
    return f(H, K, V, C, S, _p(temporal), _p(conv), ROUND[state_round], ROUND[conv_round], _p(x),
             _p(conv_w), _p(g), _p(beta), len(sl), x.shape[0], _p(cu), _p(pre), _p(sl), _p(warm),
             _p(tr), _p(ctr), int(track_stride if tr is not None else 0), int(gate_mode), int(flags),
             float(q_scale), ROUND[out_round], _p(out), int(nthreads or host_threads()))


def decode_arrays(prec, temporal, conv, x, conv_w, g, beta, slot, pos, track_slot, track_interval,
                  gate_mode, flags, q_scale, out, state_round, conv_round, out_round,
                  spec_t=None, spec_c=None, nthreads=None):
    """x [B][D][C]; out [B][D][H][V]; spec_t [B][D][H][V][K], spec_c [B][D][C][3]
    or None. Returns the status."""
    dt = DTYPE[prec]
    for a in (temporal, conv, x, conv_w, g, beta, out):
        assert a.dtype == dt and a.flags.c_contiguous
    S, H, V, K = temporal.shape
    C = conv.shape[1]
    B, D = x.shape[0], x.shape[1]
    sl, ps = _i64(slot), _i64(pos)
    ts = _i64(track_slot) if track_slot is not None else None
    f = getattr(lib(), f"lin_ref_decode_{prec}")
    return f(H, K, V, C, S, _p(temporal), _p(conv), ROUND[state_round], ROUND[conv_round], _p(x),
             _p(conv_w), _p(g), _p(beta), B, D, _p(sl), _p(ps), _p(ts), int(track_interval),
             int(gate_mode), int(flags), float(q_scale), ROUND[out_round], _p(out), _p(spec_t),
             _p(spec_c), int(nthreads or host_threads()))


def commit_arrays(prec, temporal, conv, slot, pos, accept_len, track_slot, track_interval,
                  spec_t, spec_c):
    S, H, V, K = temporal.shape
    C = conv.shape[1]
    B, D = spec_t.shape[0], spec_t.shape[1]
    sl, ps, acc = _i64(slot), _i64(pos), _i64(accept_len)
    ts = _i64(track_slot) if track_slot is not None else None
    getattr(lib(), f"lin_ref_commit_{prec}")(H, K, V, C, _p(temporal), _p(conv), B, D, _p(sl),
                                             _p(ps), _p(acc), _p(ts), int(track_interval),
                                             _p(spec_t), _p(spec_c))


def copy_slots_bytes(buf, src, dst, nthreads=None):
    """buf: a contiguous array [layers][slots][...] of any dtype; block
    dst[i] <- block src[i] in every layer (negative ids skip the pair)."""
    assert buf.flags.c_contiguous
    layers, slots = buf.shape[0], buf.shape[1]
    block = buf[0, 0].nbytes
    s, d = _i64(src), _i64(dst)
    lib().lin_ref_copy_slots_f64(_p(buf), buf[0].nbytes, block, block, layers, len(s), _p(s), _p(d),
                                 int(nthreads or host_threads()))


# ----------------------------------------------------------------------------
# dict level: the numpy oracle's pool and call shapes
# ----------------------------------------------------------------------------

def prefill(pool, layer, x, conv_w, g, beta, cu_seqlens, prefix_len, slot, has_initial_state,
            track_slots, cu_track, track_stride, gate_mode, flags, q_scale=1.0, out_dtype="f32",
            precision="f64", nthreads=None):
    """lin_state_oracle.prefill's contract (pool updated in place; returns
    (out [T][H][V] as float64, status)), computed in `precision`."""
    dt = DTYPE[precision]
    temporal = _arr(pool["temporal"][layer], dt)
    conv = _arr(pool["conv"][layer], dt)
    T = x.shape[0]
    H, V = temporal.shape[1], temporal.shape[2]
    out = np.zeros((T, H, V), dt)
    st = prefill_arrays(precision, temporal, conv, _arr(x, dt), _arr(conv_w, dt), _arr(g, dt),
                        _arr(beta, dt), cu_seqlens, prefix_len, slot, has_initial_state,
                        track_slots, cu_track, track_stride, gate_mode, flags, q_scale, out,
                        pool["state_dtype"], pool["conv_dtype"], out_dtype, nthreads)
    pool["temporal"][layer] = temporal
    pool["conv"][layer] = conv
    return out.astype(np.float64), st


def decode(pool, layer, x, conv_w, g, beta, slot, pos, track_slot, track_interval, gate_mode,
           flags, q_scale=1.0, out_dtype="f32", spec=None, precision="f64", nthreads=None):
    """lin_state_oracle.decode's contract for a linear chain (no draft tree)."""
    dt = DTYPE[precision]
    temporal = _arr(pool["temporal"][layer], dt)
    conv = _arr(pool["conv"][layer], dt)
    B, D = x.shape[0], x.shape[1]
    H, V = temporal.shape[1], temporal.shape[2]
    out = np.zeros((B, D, H, V), dt)
    spec_t = spec_c = None
    if spec is not None and D > 1:
        spec_t = _arr(spec["temporal"][layer][:B, :D], dt)
        spec_c = _arr(spec["conv"][layer][:B, :D], dt)
    st = decode_arrays(precision, temporal, conv, _arr(x, dt), _arr(conv_w, dt), _arr(g, dt),
                       _arr(beta, dt), slot, pos, track_slot, track_interval, gate_mode, flags,
                       q_scale, out, pool["state_dtype"], pool["conv_dtype"], out_dtype, spec_t,
                       spec_c, nthreads)
    pool["temporal"][layer] = temporal
    pool["conv"][layer] = conv
    if spec_t is not None:
        spec["temporal"][layer][:B, :D] = spec_t
        spec["conv"][layer][:B, :D] = spec_c
    return out.astype(np.float64), st
