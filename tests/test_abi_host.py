"""Host-side checks of the C ABI: the library loads on a machine without a
GPU, exports every entry point the header declares, computes slot sizes, and
rejects bad arguments before touching the device. CPU only."""

import ctypes
import json
import os
import re

import pytest
import torch

import linear_attention_state_chunked_gb300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_symbols():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        names |= set(re.findall(r"LIN_API\s+[\w\s\*]+?\b(lin_state_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert names, "no declarations found"
    lib = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(L.EXPORTED) <= names


def fake_pool(num_layers=69, num_slots=257, H=12, D=128, st=L.LIN_BF16, ct=L.LIN_BF16):
    p = L.PoolT()
    p.num_layers, p.num_slots, p.num_heads = num_layers, num_slots, H
    p.head_k = p.head_v = D
    p.conv_channels, p.conv_width = 3 * H * D, 4
    p.state_dtype, p.conv_dtype = st, ct
    es_t = 2 if st == L.LIN_BF16 else 4
    es_c = 2 if ct == L.LIN_BF16 else 4
    p.temporal = 0x100000  # never dereferenced by the host-side checks
    p.temporal_slot_stride = H * D * D * es_t
    p.temporal_layer_stride = num_slots * p.temporal_slot_stride
    p.conv = 0x200000
    p.conv_slot_stride = 3 * H * D * 3 * es_c
    p.conv_layer_stride = num_slots * p.conv_slot_stride
    return p


def test_slot_bytes_kimi_k3_shard():
    """Kimi-K3 notes: 25.9 MB SSM + 1.82 MB conv per GPU-slot over 69 layers."""
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "state_sizes.json")))["kimi_k3_tp8"]
    p = fake_pool()
    n = L.lib.lin_state_slot_bytes(ctypes.byref(p))
    assert n == gold["ssm_bytes_per_slot"] + gold["conv_bytes_per_slot"] == 29039616


def test_slot_bytes_qwen3_next_layer_fp32():
    p = fake_pool(num_layers=32, H=32, D=128, st=L.LIN_F32)
    n = L.lib.lin_state_slot_bytes(ctypes.byref(p))
    ssm = 32 * 32 * 128 * 128 * 4
    assert n == ssm + 32 * (3 * 32 * 128 * 3 * 2)
    assert ssm == 64 * 2 ** 20  # about 64 MB per fork over 32 layers


@pytest.mark.parametrize("field,value,code", [
    ("head_k", 96, L.LIN_EUNSUPPORTED),
    ("conv_width", 3, L.LIN_EUNSUPPORTED),
    ("conv_channels", 100, L.LIN_EINVAL),
    ("state_dtype", 7, L.LIN_EINVAL),
    ("temporal_slot_stride", 24, L.LIN_EINVAL),
    ("num_slots", 0, L.LIN_EINVAL),
])
def test_pool_validation(field, value, code):
    p = fake_pool()
    setattr(p, field, value)
    if field == "head_k":
        p.head_v = value
    assert L.lib.lin_state_slot_bytes(ctypes.byref(p)) == code
    assert L.lib.lin_state_last_error().decode()


@pytest.mark.parametrize("hk,hv,ok", [(128, 64, True), (128, 32, False), (64, 32, False),
                                      (64, 128, False)])
def test_pool_value_head_dim(hk, hv, ok):
    """Heads with V != K: (128, 64) is accepted (slot bytes count the [H][V][K]
    state and the 2HK + HV conv channels); other pairs are LIN_EUNSUPPORTED."""
    H, S, NL = 3, 5, 2
    pool = L.StatePool(NL, S, H, hk, state_dtype=torch.bfloat16, conv_dtype=torch.bfloat16,
                       device="cpu", head_v=hv)
    assert tuple(pool.temporal.shape) == (NL, S, H, hv, hk)
    assert pool.conv_channels == 2 * H * hk + H * hv
    n = L.lib.lin_state_slot_bytes(ctypes.byref(pool.desc()))
    if ok:
        assert n == NL * (H * hv * hk * 2 + (2 * H * hk + H * hv) * 3 * 2)
    else:
        assert n == L.LIN_EUNSUPPORTED
        assert "head_v" in L.lib.lin_state_last_error().decode()


def _prefill_args(**kw):
    a = L.PrefillArgsT()
    a.layer, a.batch, a.total_tokens = 0, 1, 64
    a.io_dtype = a.out_dtype = L.LIN_BF16
    a.gate_mode, a.flags, a.q_scale, a.track_stride = L.LIN_GATE_PER_KEY, 3, 1.0, 64
    for f in ("x", "conv_w", "g", "beta", "out", "cu_seqlens", "prefix_len", "slot",
              "has_initial_state", "track_slots", "cu_track"):
        setattr(a, f, 0x300000)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(track_stride=65), L.LIN_EINVAL),
    (dict(track_stride=-64), L.LIN_EINVAL),
    (dict(layer=69), L.LIN_EINVAL),
    (dict(io_dtype=5), L.LIN_EINVAL),
    (dict(gate_mode=3), L.LIN_EINVAL),
    (dict(x=None), L.LIN_EINVAL),
    (dict(track_slots=None), L.LIN_EINVAL),
])
def test_prefill_rejects_bad_args_on_host(kw, code):
    p = fake_pool()
    a = _prefill_args(**kw)
    rc = L.lib.lin_state_prefill(ctypes.byref(p), ctypes.byref(a), None, 0, None)
    assert rc == code, (rc, L.lib.lin_state_last_error())


def test_decode_and_copy_reject_bad_args_on_host():
    p = fake_pool()
    d = L.DecodeArgsT()
    d.layer, d.batch, d.n_draft = 0, 4, 0
    assert L.lib.lin_state_decode(ctypes.byref(p), ctypes.byref(d), None) == L.LIN_EINVAL
    d.n_draft = 4  # a verify with half a spec buffer (no conv part) is rejected
    d.io_dtype = d.out_dtype = L.LIN_BF16
    for f in ("x", "conv_w", "g", "beta", "out", "slot", "pos"):
        setattr(d, f, 0x300000)
    d.spec.temporal = 0x400000
    assert L.lib.lin_state_decode(ctypes.byref(p), ctypes.byref(d), None) == L.LIN_EINVAL
    assert "spec" in L.lib.lin_state_last_error().decode()
    # replay commit: accept_len is required, and inputs must be 16-byte aligned
    r = L.ReplayArgsT()
    r.layer, r.batch, r.n_draft, r.io_dtype = 0, 4, 4, L.LIN_BF16
    r.gate_mode = L.LIN_GATE_PER_KEY
    for f in ("x", "conv_w", "g", "beta", "slot", "pos"):
        setattr(r, f, 0x300000)
    assert L.lib.lin_state_replay_commit(ctypes.byref(p), ctypes.byref(r), None) == L.LIN_EINVAL
    assert "accept_len" in L.lib.lin_state_last_error().decode()
    r.accept_len, r.x = 0x300000, 0x300004
    assert L.lib.lin_state_replay_commit(ctypes.byref(p), ctypes.byref(r), None) == L.LIN_EINVAL
    assert "aligned" in L.lib.lin_state_last_error().decode()
    r.n_draft = 0
    assert L.lib.lin_state_replay_commit(ctypes.byref(p), ctypes.byref(r), None) == L.LIN_EINVAL
    assert L.lib.lin_state_copy_slots(ctypes.byref(p), None, None, 3, 0, 69, 0, None, None) == L.LIN_EINVAL
    assert L.lib.lin_state_copy_slots(ctypes.byref(p), 0x10, 0x10, 3, 5, 2, 0, None, None) == L.LIN_EINVAL
    # empty work is a no-op that never reaches the device
    assert L.lib.lin_state_copy_slots(ctypes.byref(p), None, None, 0, 0, 69, 0, None, None) == 0
    assert L.lib.lin_state_restore(ctypes.byref(p), None, 0, None, None, None) == 0


def test_decode_rejects_drafts_past_the_staging_limit():
    """Head 128 with fp32 state, conv and io and per-key gates stages
    76,288 + 2,048 bytes per draft (state 64 KB, conv window, taps; x and g
    rows per draft) per (request, head): 17 drafts fit in 110 KB, 18 do not,
    and the host says so before any launch."""
    p = fake_pool(num_layers=2, st=L.LIN_F32, ct=L.LIN_F32)
    d = L.DecodeArgsT()
    d.layer, d.batch, d.n_draft = 0, 4, 18
    d.io_dtype = d.out_dtype = L.LIN_F32
    d.gate_mode, d.flags, d.q_scale = L.LIN_GATE_PER_KEY, 3, 1.0
    for f in ("x", "conv_w", "g", "beta", "out", "slot", "pos"):
        setattr(d, f, 0x300000)
    sp = d.spec
    sp.num_layers, sp.max_batch, sp.max_draft = 2, 4, 32
    sp.temporal, sp.conv = 0x400000, 0x500000
    blk = p.temporal_slot_stride
    sp.temporal_step_stride, sp.temporal_req_stride = blk, 32 * blk
    sp.temporal_layer_stride = 4 * 32 * blk
    sp.conv_step_stride = p.conv_slot_stride
    sp.conv_req_stride = 32 * p.conv_slot_stride
    sp.conv_layer_stride = 4 * 32 * p.conv_slot_stride
    d.spec = sp
    assert L.lib.lin_state_decode(ctypes.byref(p), ctypes.byref(d), None) == L.LIN_EUNSUPPORTED
    assert "n_draft 18" in L.lib.lin_state_last_error().decode()


def test_strerror_and_version():
    assert L.lib.lin_state_strerror(L.LIN_EINVAL) == b"invalid argument"
    assert L.lin_state_version() >> 16 == 1


def test_binding_constants_match_header():
    """Every flag, status bit and dtype / gate code the binding exports has the
    header's value (the flags of the enum, the LIN_ST_* and LIN_KERNEL_* defines)."""
    src = "".join(open(h).read() for h in HEADERS)
    values = {n: int(v) for n, v in re.findall(r"\b(LIN_[A-Z0-9_]+)\s*=\s*(\d+)u?\b", src)}
    values.update({n: int(v) for n, v in re.findall(r"#define\s+(LIN_(?:ST|KERNEL)_[A-Z0-9_]+)\s+(\d+)", src)})
    assert "LIN_PREFILL_ONE_PIECE" in values and "LIN_ST_TIMEOUT" in values
    exported = {n: getattr(L, n) for n in values if hasattr(L, n)}
    assert len(exported) >= 15
    assert all(exported[n] == values[n] for n in exported), {n: (exported[n], values[n]) for n in exported
                                                              if exported[n] != values[n]}
