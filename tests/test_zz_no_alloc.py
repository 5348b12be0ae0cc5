"""pa_decode_noalloc: the decode for callers that cannot allocate device
memory when they run it (a runtime that owns all device memory through its
own pool, a latency-critical loop that cannot risk an allocation's device
synchronisation).  Its split-KV scratch is the library's fixed per-device
array instead of a workspace argument.

Every case goes through the C ABI and is checked two ways: against the
oracle within the tests' attention tolerance, and bit for bit against
pa_decode (which takes a caller-allocated workspace) on the same inputs --
both launch the same kernel with the same grid, so any difference would be
a scratch-layout slip.  Calls follow one another on the shared array, so
each runs over what the previous one left behind.  This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_116_gb300 import workloads as W

from helpers import device_caches, oracle_attention, within_tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def _inputs(w):
    kc, vc, bt = device_caches(w, DEV)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    return kc, vc, bt, lens, int(w.seq_lens.max())


def _workspace_decode(pa, w, kc, vc, bt, lens, mc):
    ws_bytes = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, mc,
                                           W.TORCH_DTYPES[w.dtype])
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
    pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale, workspace=ws)
    return out


def _noalloc_decode(pa, w, kc, vc, bt, lens, mc):
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
    pa.pa_decode_noalloc(out, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale)
    return out


def _check(pa, w):
    kc, vc, bt, lens, mc = _inputs(w)
    got = _noalloc_decode(pa, w, kc, vc, bt, lens, mc)
    ref = _workspace_decode(pa, w, kc, vc, bt, lens, mc)
    torch.cuda.synchronize()
    pa.pa_device_status(clear=True)  # raises if a bounded wait ran out
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), "pa_decode_noalloc differs from pa_decode (%s)" % w.name
    ok, err = within_tol(got.double().cpu().numpy(), oracle_attention(w), w.dtype)
    assert ok, "pa_decode_noalloc differs from the oracle by %.3g (%s)" % (err, w.name)


# shapes chosen so that each fits the 8 MiB array yet splits units between
# warps: the G <= 8 and G > 8 kernel instances, head_dim 64 / 128 / 256,
# 8- and 32-token blocks
SHAPES = [
    ("g4_hd128_bf16", lambda: W.decode_workload("na_g4", "bf16", 16, 32, 8, 128, W.gqa_batch_lengths(24), seed=11)),
    ("g1_hd128_f16", lambda: W.decode_workload("na_mha", "f16", 16, 8, 8, 128, [1, 900, 33, 2048, 16, 470, 5],
                                               seed=12)),
    ("g12_hd128_f16", lambda: W.decode_workload("na_g12", "f16", 16, 24, 2, 128, [1, 130, 257, 500], seed=13)),
    ("g16_hd64_bf16", lambda: W.decode_workload("na_g16", "bf16", 16, 16, 1, 64, [700, 31, 1, 333], seed=14)),
    ("g4_hd256_bf16", lambda: W.decode_workload("na_hd256", "bf16", 32, 8, 2, 256, [1000, 65, 2, 400], seed=15)),
    ("g8_hd64_bs8_f16", lambda: W.decode_workload("na_bs8", "f16", 8, 16, 2, 64, [9, 800, 17, 1], seed=16)),
]


@pytest.mark.parametrize("name,make", SHAPES)
def test_noalloc_equals_workspace_decode_and_oracle(pa, name, make):
    _check(pa, make())


def test_noalloc_two_calls_in_a_row_over_stale_scratch(pa):
    """The first call splits two long sequences over every warp, so its
    partial records fill the array well past where the second call keeps
    its unit descriptors (1,000 sequences x 8 KV heads x 16 bytes); the
    second call must not be misled by those leftovers."""
    first = W.decode_workload("na_fill", "bf16", 16, 32, 8, 128, [3000, 2500], seed=21)
    second = W.decode_workload("na_after", "bf16", 16, 32, 8, 128, np.random.default_rng(22).integers(1, 40, 1000)
                               .tolist(), seed=22)
    _check(pa, first)
    _check(pa, second)


def test_noalloc_more_sequences_than_one_launch_takes(pa):
    """4,200 one-query sequences at G = 1 run as two launches (4,096 + 104)
    on the same array, one after the other."""
    lens = np.random.default_rng(31).integers(1, 40, 4200).tolist()
    _check(pa, W.decode_workload("na_4200", "bf16", 16, 2, 2, 128, lens, seed=31))


def test_noalloc_check_mode_rejects_bad_tables(pa):
    w = W.decode_workload("na_check", "bf16", 16, 8, 2, 128, [40, 17], seed=51)
    kc, vc, bt, lens, mc = _inputs(w)
    bad = bt.clone()
    bad[1, 0] = w.num_blocks  # outside the pool
    out = torch.zeros((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16, device=DEV)
    pa.pa_set_check_mode(True)
    try:
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_decode_noalloc(out, w.q.to(DEV), kc, vc, bad, lens, mc, w.scale)
        torch.cuda.synchronize()
        assert torch.count_nonzero(out).item() == 0  # nothing ran
        pa.pa_decode_noalloc(out, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale)  # valid tables pass
    finally:
        pa.pa_set_check_mode(False)


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
