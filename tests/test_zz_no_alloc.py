"""lin_state_prefill_noalloc: the prefill for callers that cannot allocate
device memory during a step (serving engines whose own pools take all device
memory at start-up, loops that must not pay the device-wide synchronisation of
cudaMalloc / cudaFree). Its scratch is fixed arrays inside the library, shared
by every call, instead of a caller workspace.

Checked here, through the C ABI:
  - batches, two calls in a row (the second finds the scratch as the first left
    it): outputs, states, snapshots and windows equal lin_state_prefill's bit
    for bit (the same kernel in the same longest-first order), and the oracle
    within the fp32-state bar;
  - a single long request, which lin_state_prefill runs in segments and this
    call in one piece: both against the oracle;
  - the token-by-token kernel (LIN_PREFILL_RECURRENT) against the oracle;
  - a per-key request whose decay leaves the chunk's factored range, rerun
    through the fixed rerun flags, against the oracle;
  - the size limits of the fixed scratch, which bind only the chunked kernel.

pytest collects this file last (its name sorts after the other test files), so
a run that stops at the first failure has run every other test before it. No
test here depends on another having run: each passes alone in a fresh process.
"""

import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import TOL_F32, compare_outputs, compare_slots, fill_pool, np64, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAGS = L.LIN_QK_L2NORM | L.LIN_CONV_SILU


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def _kwargs(b, out, slots, tracks, cu_track, stride, status, flags=FLAGS):
    return dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV), beta=b.beta.to(DEV),
                out=out, cu_seqlens=b.cu_seqlens.to(DEV), prefix_len=b.prefix_len.to(DEV),
                slot=_i32(slots), has_initial_state=b.has_initial_state.to(DEV),
                track_slots=_i32(tracks) if stride else None,
                cu_track=_i32(cu_track) if stride else None, track_stride=stride,
                gate_mode=b.gate_mode, flags=flags, status=status)


def _oracle(op, b, slots, tracks, cu_track, stride, flags=FLAGS):
    return O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta),
                     b.cu_seqlens.tolist(), b.prefix_len.tolist(), slots,
                     b.has_initial_state.tolist(), tracks, cu_track, stride, b.gate_mode,
                     flags, 1.0, "f32")


@pytest.mark.parametrize("gate", [W.GATE_PER_HEAD, W.GATE_PER_KEY])
def test_noalloc_prefill_equals_prefill_twice(gate):
    dims = W.LayerDims(num_heads=4, head_k=128, head_v=128)
    pools = []
    for _ in range(2):
        p = L.StatePool(1, 32, 4, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                        device=DEV)
        fill_pool(p, 41)
        pools.append(p)
    op = oracle_pool(pools[1])
    for call, lengths in enumerate([[300, 64, 1000, 5], [700, 129, 64, 0, 256]]):
        B = len(lengths)
        prefixes = [64 * (i % 2) for i in range(B)]
        warm = [i % 2 for i in range(B)]
        b = W.make_prefill_batch(dims, lengths, gate, dtype=torch.bfloat16, seed=call,
                                 prefixes=prefixes, warm=warm, tag=f"noalloc{call}")
        slots = list(range(1, B + 1))
        tracks, cu_track = list(range(8, 8 + 2 * B)), list(range(0, 2 * B + 1, 2))
        outs = []
        for k, pool in enumerate(pools):
            out = torch.full((b.total_tokens, 4, 128), -9.0, device=DEV)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            kw = _kwargs(b, out, slots, tracks, cu_track, 64, st)
            if k == 0:
                L.lin_state_prefill(pool, **kw)
            else:
                L.lin_state_prefill_noalloc(pool, **kw)
            assert L.lin_state_read_status(st) == 0
            outs.append(out)
        assert torch.equal(outs[1], outs[0])
        assert torch.equal(pools[1].temporal, pools[0].temporal)
        assert torch.equal(pools[1].conv, pools[0].conv)
        oo, ost = _oracle(op, b, slots, tracks, cu_track, 64)
        assert ost == 0
        compare_outputs(outs[1], oo, b.cu_seqlens.tolist(), TOL_F32)
        compare_slots(pools[1], op, slots + tracks, TOL_F32)


@pytest.mark.parametrize("gate", [W.GATE_PER_HEAD, W.GATE_PER_KEY])
def test_noalloc_long_single_request_in_one_piece(gate):
    """4,200 tokens of one request: lin_state_prefill runs it in segments (the
    request's 2 heads leave most SMs idle), the allocation-free call in one
    piece; both match the oracle."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    n = 4200
    b = W.make_prefill_batch(dims, [n], gate, dtype=torch.bfloat16, seed=11, tag="noalloc.long",
                             gate="softplus" if gate == W.GATE_PER_KEY else "uniform",
                             prefixes=[64], warm=[1])
    n_tr = (64 + n) // 256 - 64 // 256
    tracks = list(range(2, 2 + n_tr))
    for k in range(2):
        pool = L.StatePool(1, 2 + n_tr, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                           device=DEV)
        fill_pool(pool, 12)
        op = oracle_pool(pool)
        out = torch.zeros((n, 2, 128), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        kw = _kwargs(b, out, [1], tracks, [0, n_tr], 256, st)
        if k == 0:
            need = L.lin_state_prefill_workspace(pool, **kw)
            assert need > 16 * 1024  # the segmented mode's per-segment states
            ws = torch.empty(need, dtype=torch.uint8, device=DEV)
            L.lin_state_prefill(pool, workspace=ws, **kw)
        else:
            L.lin_state_prefill_noalloc(pool, **kw)
        assert L.lin_state_read_status(st) == 0
        oo, ost = _oracle(op, b, [1], tracks, [0, n_tr], 256)
        assert ost == 0
        compare_outputs(out, oo, [0, n], TOL_F32)
        compare_slots(pool, op, [1] + tracks, TOL_F32)


def test_noalloc_recurrent_kernel():
    """LIN_PREFILL_RECURRENT through the allocation-free call: the token-by-token
    kernel, which takes no scratch, against the oracle."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, [150, 70, 64], W.GATE_PER_KEY, dtype=torch.bfloat16, seed=13,
                             tag="noalloc.rec", prefixes=[0, 64, 0], warm=[0, 1, 0])
    pool = L.StatePool(1, 10, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 14)
    op = oracle_pool(pool)
    out = torch.zeros((b.total_tokens, 2, 128), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    flags = FLAGS | L.LIN_PREFILL_RECURRENT
    kw = _kwargs(b, out, [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 64, st, flags=flags)
    assert L.lin_state_prefill_kernel(pool, **kw) == L.LIN_KERNEL_RECURRENT
    L.lin_state_prefill_noalloc(pool, **kw)
    assert L.lin_state_read_status(st) == 0
    oo, _ = _oracle(op, b, [1, 2, 3], [4, 5, 6, 7, 8, 9], [0, 2, 4, 6], 64, flags=flags)
    compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
    compare_slots(pool, op, list(range(1, 10)), TOL_F32)


def test_noalloc_kda_decay_beyond_chunk_range():
    """Per-key gates where one (request, head) decays beyond the chunk's
    factored range: the fixed rerun flags route it to the token-by-token
    rerun; two calls in a row, so the second finds the flags the first set
    and must clear them."""
    dims = W.LayerDims(num_heads=2, head_k=128, head_v=128)
    pool = L.StatePool(1, 12, 2, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16, device=DEV)
    fill_pool(pool, 15)
    op = oracle_pool(pool)
    for call in range(2):
        b = W.make_prefill_batch(dims, [200, 333], W.GATE_PER_KEY, dtype=torch.bfloat16,
                                 seed=16 + call, gate="softplus", tag=f"noalloc.dr{call}",
                                 prefixes=[0, 64], warm=[0, 1])
        if call == 0:
            b.g[0:200, 1] *= 30.0
        out = torch.zeros((b.total_tokens, 2, 128), device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        kw = _kwargs(b, out, [1, 2], [4, 5, 6, 7], [0, 2, 4], 64, st)
        L.lin_state_prefill_noalloc(pool, **kw)
        assert L.lin_state_read_status(st) == 0
        oo, _ = _oracle(op, b, [1, 2], [4, 5, 6, 7], [0, 2, 4], 64)
        compare_outputs(out, oo, b.cu_seqlens.tolist(), TOL_F32)
        compare_slots(pool, op, [1, 2, 4, 5, 6, 7], TOL_F32)


def test_noalloc_limits_bind_only_the_chunked_kernel():
    dims = W.LayerDims(num_heads=1, head_k=128, head_v=128)
    B = 4097
    pool = L.StatePool(1, 4, 1, 128, device=DEV)
    x = torch.zeros((B, dims.conv_channels), dtype=torch.bfloat16, device=DEV)
    kw = dict(layer=0, x=x, conv_w=torch.zeros((dims.conv_channels, 4), dtype=torch.bfloat16, device=DEV),
              g=torch.zeros((B, 1, 128), device=DEV), beta=torch.zeros((B, 1), device=DEV),
              out=torch.zeros((B, 1, 128), device=DEV),
              cu_seqlens=torch.arange(B + 1, dtype=torch.int32, device=DEV),
              prefix_len=torch.zeros(B, dtype=torch.int32, device=DEV),
              slot=torch.full((B,), -1, dtype=torch.int32, device=DEV),
              has_initial_state=torch.zeros(B, dtype=torch.int64, device=DEV),
              gate_mode=W.GATE_PER_KEY)
    assert L.lin_state_prefill_kernel(pool, **kw) == L.LIN_KERNEL_CHUNKED
    with pytest.raises(L.LinStateError, match="above the fixed scratch"):
        L.lin_state_prefill_noalloc(pool, **kw)
    # the token-by-token kernel needs no scratch: the same batch runs (every
    # slot is padding, so nothing is written)
    L.lin_state_prefill_noalloc(pool, flags=L.LIN_PREFILL_RECURRENT, **kw)
    torch.cuda.synchronize()
