"""The wrap-around schedule of the chunked prefill (McNaughton's wrap-around
rule). A batch with more (request, head) chains than SMs is laid end to end in
chunk units and cut into one range of equal units per SM; a chain that crosses
a range boundary runs as a head piece, which hands its fp32 state on, and a
tail piece, which starts from it. Each piece runs the same arithmetic as the
chain in one piece, so outputs, states, conv windows and snapshots must equal
LIN_PREFILL_ONE_PIECE's bit for bit; they are also checked against the oracle.

The batches here have 5 requests of 48 heads (240 chains, more than the SMs of
one GB300), ragged lengths of 0-16 chunks, warm and cold starts, a request the
call skips (slot -1) and snapshots at every chunk into ping-pong track pairs, so
the head and the tail of a chain write into the same two track slots.
"""

import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from oracle import lin_state_oracle as O
from tests.helpers import TOL_BF16, TOL_F32, compare_outputs, compare_slots, fill_pool, np64, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAGS = L.LIN_QK_L2NORM | L.LIN_CONV_SILU
H = 48


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def _run(pool, b, slots, tracks, cu_track, flags):
    out = torch.full((b.total_tokens, H, pool.head_v), -7.0, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV), beta=b.beta.to(DEV),
              out=out, cu_seqlens=b.cu_seqlens.to(DEV), prefix_len=b.prefix_len.to(DEV),
              slot=_i32(slots), has_initial_state=b.has_initial_state.to(DEV),
              track_slots=_i32(tracks), cu_track=_i32(cu_track), track_stride=64,
              gate_mode=b.gate_mode, flags=flags, status=st)
    need = L.lin_state_prefill_workspace(pool, **kw)
    L.lin_state_prefill(pool, **kw)
    assert L.lin_state_read_status(st) == 0
    return out, need


CASES = {
    # gate, state dtype, value channels, strong KDA decay on some pairs
    "gdn_f32": (W.GATE_PER_HEAD, torch.float32, 128, False),
    "kda_f32": (W.GATE_PER_KEY, torch.float32, 128, False),
    "kda_bf16_rerun": (W.GATE_PER_KEY, torch.bfloat16, 128, True),
    "ssd_hd64": (W.GATE_PER_HEAD, torch.float32, 64, False),
}


@pytest.mark.parametrize("case", list(CASES))
def test_wrap_pieces_equal_one_piece_and_oracle(case):
    gate_mode, sdt, hv, strong = CASES[case]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lengths = [700, 0, 130, 1000, 333]
    assert len(lengths) * H > sms, "the batch must have more chains than SMs"
    prefixes, warm = [0, 64, 128, 0, 64], [0, 1, 1, 0, 1]
    dims = W.LayerDims(num_heads=H, head_k=128, head_v=hv)
    gate = "ssd" if hv == 64 else ("softplus" if gate_mode == W.GATE_PER_KEY else "uniform")
    b = W.make_prefill_batch(dims, lengths, gate_mode, dtype=torch.bfloat16, seed=21, gate=gate,
                             prefixes=prefixes, warm=warm, tag=f"wrap.{case}")
    cu = b.cu_seqlens.tolist()
    if strong:
        # requests 0 and 4, heads 0-2: a stretch far beyond the chunk's
        # factored decay range, so those pairs are rerun token by token;
        # wherever the stretch falls (head or tail piece), the results agree
        b.g[cu[0] + 300:cu[0] + 400, 0:3] *= 30.0
        b.g[cu[4] + 10:cu[4] + 60, 0:3] *= 30.0
    flags = FLAGS | (L.LIN_UPDATE_ADDITIVE if hv == 64 else 0)
    slots = [1, 2, 3, -1, 4]
    tracks = list(range(5, 15))
    cu_track = [0, 2, 4, 6, 8, 10]
    pools = []
    for _ in range(2):
        p = L.StatePool(1, 16, H, 128, state_dtype=sdt, conv_dtype=torch.bfloat16, device=DEV, head_v=hv)
        fill_pool(p, 22)
        pools.append(p)
    op = oracle_pool(pools[0])
    out1, need1 = _run(pools[0], b, slots, tracks, cu_track, flags | L.LIN_PREFILL_ONE_PIECE)
    out2, need2 = _run(pools[1], b, slots, tracks, cu_track, flags)
    assert need2 > need1, "the default call must take the wrap-around schedule here"
    assert torch.equal(out2, out1)
    assert torch.equal(pools[1].temporal, pools[0].temporal)
    assert torch.equal(pools[1].conv, pools[0].conv)
    oo, ost = O.prefill(op, 0, np64(b.x), np64(b.conv_w), np64(b.g), np64(b.beta), cu,
                        b.prefix_len.tolist(), slots, b.has_initial_state.tolist(), tracks, cu_track, 64,
                        b.gate_mode, flags, 1.0, "f32")
    assert ost == 0
    tol = TOL_BF16 if sdt == torch.bfloat16 else TOL_F32
    compare_outputs(out2, oo, cu, tol, skip=(3,))
    compare_slots(pools[1], op, [1, 2, 3, 4] + tracks, tol)
    # the skipped request's outputs stay as they were
    assert torch.all(out2[cu[3]:cu[4]] == -7.0)


def test_wrap_two_calls_at_once_on_two_streams():
    """Two wrap-around calls in flight together on two streams (separate pools
    and workspaces), so their pieces compete for the SMs. A tail piece only
    ever waits for a head piece that a running CTA has taken, and head pieces
    wait for nothing, so both calls finish, with the one-piece results."""
    lengths = [700, 0, 130, 1000, 333]
    dims = W.LayerDims(num_heads=H, head_k=128, head_v=128)
    b = W.make_prefill_batch(dims, lengths, W.GATE_PER_HEAD, dtype=torch.bfloat16, seed=31, gate="uniform",
                             prefixes=[0, 64, 128, 0, 64], warm=[0, 1, 1, 0, 1], tag="wrap.streams")
    slots, tracks, cu_track = [1, 2, 3, 4, 5], list(range(6, 16)), [0, 2, 4, 6, 8, 10]
    pools = []
    for _ in range(3):
        p = L.StatePool(1, 16, H, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16, device=DEV)
        fill_pool(p, 32)
        pools.append(p)
    ref, _ = _run(pools[0], b, slots, tracks, cu_track, FLAGS | L.LIN_PREFILL_ONE_PIECE)
    args = []
    for pool in pools[1:]:
        out = torch.full((b.total_tokens, H, 128), -7.0, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV), beta=b.beta.to(DEV),
                  out=out, cu_seqlens=b.cu_seqlens.to(DEV), prefix_len=b.prefix_len.to(DEV),
                  slot=_i32(slots), has_initial_state=b.has_initial_state.to(DEV),
                  track_slots=_i32(tracks), cu_track=_i32(cu_track), track_stride=64,
                  gate_mode=b.gate_mode, flags=FLAGS, status=st)
        ws = torch.empty(L.lin_state_prefill_workspace(pool, **kw), dtype=torch.uint8, device=DEV)
        args.append((pool, kw, ws, out, st))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for (pool, kw, ws, out, st), s in zip(args, streams):
        L.lin_state_prefill(pool, workspace=ws, stream=s, **kw)
    torch.cuda.synchronize()
    for pool, kw, ws, out, st in args:
        assert L.lin_state_read_status(st) == 0
        assert torch.equal(out, ref)
        assert torch.equal(pool.temporal, pools[0].temporal)
        assert torch.equal(pool.conv, pools[0].conv)
