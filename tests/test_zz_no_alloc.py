"""pa_decode_noalloc: the decode for callers that cannot allocate device
memory when they run it (a runtime that owns all device memory through its
own pool, a latency-critical loop that cannot risk an allocation's device
synchronisation).  Its split-KV scratch is the library's fixed per-device
array instead of a workspace argument.

Checked through the C ABI against pa_decode (which takes a caller-allocated
workspace) on two calls in a row -- two different batches, so the second
call runs over the scratch the first one left behind -- within the tests'
attention tolerance.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_116_gb300 import workloads as W

from helpers import device_caches, within_tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def _reference_decode(pa, w, kc, vc, bt, lens, mc):
    ws_bytes = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, mc,
                                           W.TORCH_DTYPES[w.dtype])
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
    pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale, workspace=ws)
    return out


def test_noalloc_matches_workspace_decode_twice(pa):
    batches = [
        W.decode_workload("na1", "bf16", 16, 32, 8, 128, W.gqa_batch_lengths(24), seed=11),
        W.decode_workload("na2", "f16", 16, 8, 2, 128, [1, 900, 33, 2048, 16, 470, 5], seed=12),
    ]
    for w in batches:  # two calls in a row on the shared scratch
        kc, vc, bt = device_caches(w, DEV)
        lens = torch.from_numpy(w.seq_lens).to(DEV)
        mc = int(w.seq_lens.max())
        ref = _reference_decode(pa, w, kc, vc, bt, lens, mc)
        got = torch.full_like(ref, float("nan"))
        pa.pa_decode_noalloc(got, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale)
        torch.cuda.synchronize()
        ok, err = within_tol(got.double().cpu().numpy(), ref.double().cpu().numpy(), w.dtype)
        assert ok, "pa_decode_noalloc differs from pa_decode by %.3g (%s)" % (err, w.name)


def test_noalloc_rejects_problems_beyond_its_scratch(pa):
    # 4096 one-token sequences, 16 query heads per KV head: the split scratch
    # this shape asks for (sized as for pa_decode) exceeds the fixed array,
    # so the call must refuse before launching.  The buffers are real and the
    # lengths are 1, so the inputs would be valid even for a launch.
    S, hq, hkv, hd, mc = 4096, 64, 4, 128, 65536
    need = pa.pa_decode_workspace_size(S, hq, hkv, hd, 16, mc, torch.bfloat16)
    assert need > (8 << 20), "shape does not exceed the scratch on this device (%d bytes)" % need
    q = torch.zeros((S, hq, hd), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros_like(q)
    kc = torch.zeros((16, 16, hkv, hd), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((S, 1), dtype=torch.int32, device=DEV)
    lens = torch.ones(S, dtype=torch.int32, device=DEV)
    with pytest.raises(pa.PAError, match="PA_ERR_WORKSPACE"):
        pa.pa_decode_noalloc(out, q, kc, kc, bt, lens, mc, 1.0)
    assert torch.count_nonzero(out).item() == 0  # nothing ran
