"""lin_state_prefill_noalloc: the prefill for callers that cannot allocate
device memory during a step (engines whose pools own all device memory, loops
that must not pay the synchronisation of cudaMalloc / cudaFree). Its scratch is
a fixed array inside the library, so this checks it against the regular
lin_state_prefill (which takes a caller workspace) on two calls in a row, the
second one finding the array filled by the first. This file is collected last
on purpose."""

import pytest
import torch

import linear_attention_state_chunked_gb300 as L
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, fill_pool, max_rel_per_head, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("gate", [W.GATE_PER_HEAD, W.GATE_PER_KEY])
def test_noalloc_prefill_matches_prefill_twice(gate):
    dims = W.LayerDims(num_heads=4, head_k=128, head_v=128)
    tol = TOL_F32 if gate == W.GATE_PER_HEAD else TOL_BF16
    pools = []
    for _ in range(2):
        p = L.StatePool(1, 32, 4, 128, state_dtype=torch.float32, conv_dtype=torch.bfloat16,
                        device=DEV)
        fill_pool(p, 41)
        pools.append(p)
    for call, lengths in enumerate([[300, 64, 1000, 5], [700, 129, 64, 0, 256]]):
        B = len(lengths)
        prefixes = [64 * (i % 2) for i in range(B)]
        warm = [i % 2 for i in range(B)]
        b = W.make_prefill_batch(dims, lengths, gate, dtype=torch.bfloat16, seed=call,
                                 prefixes=prefixes, warm=warm, tag=f"noalloc{call}")
        outs = []
        for k, pool in enumerate(pools):
            out = torch.zeros((b.total_tokens, 4, 128), device=DEV)
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            kw = dict(layer=0, x=b.x.to(DEV), conv_w=b.conv_w.to(DEV), g=b.g.to(DEV),
                      beta=b.beta.to(DEV), out=out, cu_seqlens=b.cu_seqlens.to(DEV),
                      prefix_len=b.prefix_len.to(DEV), slot=_i32(list(range(1, B + 1))),
                      has_initial_state=b.has_initial_state.to(DEV),
                      track_slots=_i32(list(range(8, 8 + 2 * B))),
                      cu_track=_i32(list(range(0, 2 * B + 1, 2))), track_stride=64,
                      gate_mode=gate, status=st)
            if k == 0:
                L.lin_state_prefill(pool, **kw)
            else:
                L.lin_state_prefill_noalloc(pool, **kw)
            assert L.lin_state_read_status(st) == 0
            outs.append(np64(out))
        assert max_rel_per_head(outs[1], outs[0], 1) <= tol
        assert torch.allclose(pools[1].temporal, pools[0].temporal, rtol=0, atol=0) or \
            max_rel_per_head(np64(pools[1].temporal[0]), np64(pools[0].temporal[0]), 1) <= tol
        assert torch.equal(pools[1].conv, pools[0].conv)


def test_noalloc_rejects_batches_above_its_scratch():
    dims = W.LayerDims(num_heads=1, head_k=128, head_v=128)
    B = 4097
    pool = L.StatePool(1, 4, 1, 128, device=DEV)
    x = torch.zeros((B, dims.conv_channels), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(L.LinStateError, match="above the fixed scratch"):
        L.lin_state_prefill_noalloc(
            pool, layer=0, x=x, conv_w=torch.zeros((dims.conv_channels, 4), dtype=torch.bfloat16, device=DEV),
            g=torch.zeros((B, 1, 128), device=DEV), beta=torch.zeros((B, 1), device=DEV),
            out=torch.zeros((B, 1, 128), device=DEV), cu_seqlens=torch.arange(B + 1, dtype=torch.int32, device=DEV),
            prefix_len=torch.zeros(B, dtype=torch.int32, device=DEV),
            slot=torch.full((B,), -1, dtype=torch.int32, device=DEV),
            has_initial_state=torch.zeros(B, dtype=torch.int64, device=DEV))
