"""GPU parity of pa_decode against the oracle.

Tolerance: |gpu - exact| <= atol + rtol * |exact| with atol 1e-5 (fp32) /
1e-2 (bf16, f16) and rtol the output type's unit roundoff (helpers.ATOL /
RTOL).  Unused cache slots are NaN in every case, so a read outside a
sequence's context fails the comparison.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_116_gb300 import workloads as W

from helpers import device_caches, graph_replays_match_eager, oracle_attention, oracle_caches, within_tol

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def run_decode(pa, w, kc, vc, bt, kernel=0, ctas=0, max_context=None):
    pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, kernel)
    pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, ctas)
    try:
        mc = int(w.seq_lens.max()) if max_context is None else max_context
        lens = torch.from_numpy(w.seq_lens).to(DEV)
        ws_bytes = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                               mc, W.TORCH_DTYPES[w.dtype])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype],
                         device=DEV)
        pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, mc, w.scale, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
        return out
    finally:
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, 0)
        pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, 0)


def compare(w, out, exact, rows=None):
    got = out.double().cpu().numpy()
    if rows is not None:
        got, exact = got[rows], exact[rows]
    ok, err = within_tol(got, exact, w.dtype)
    assert ok, "max error %.3g beyond tolerance (%s)" % (err, w.name)
    return err


def test_tiny_decode_fp32(pa):
    w = W.tiny_decode()
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    err = compare(w, run_decode(pa, w, kc, vc, bt), exact)
    assert err < 1e-5


@pytest.mark.parametrize("kernel", [0, 1])
def test_gqa_decode_batch_full(pa, kernel):
    w = W.gqa_decode_batch(device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    compare(w, run_decode(pa, w, kc, vc, bt, kernel=kernel), exact)


def test_long_context_decode_full(pa):
    """8 x 32,768 tokens: every unit is split over many warps and merged;
    all eight sequences' outputs against the oracle."""
    w = W.long_context_decode(device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    compare(w, run_decode(pa, w, kc, vc, bt), exact)


def test_mha_decode_fp16_full(pa):
    w = W.mha_decode(device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    compare(w, run_decode(pa, w, kc, vc, bt), exact)


CASES = []
_r = np.random.default_rng(123)
for _i in range(14):
    _hd = int(_r.choice([64, 128, 256]))
    _g = int(_r.choice([1, 2, 4, 5, 8, 12, 16]))
    _hkv = int(_r.choice([1, 2, 4]))
    _dt = str(_r.choice(["bf16", "f16"]))
    _S = int(_r.integers(1, 9))
    _lens = _r.integers(1, 3 * 16 + 5, _S).tolist()
    _lens[0] = int(_r.choice([1, 16, 32, 48]))  # exactly on a block boundary or a single token
    CASES.append((_dt, _hd, _g, _hkv, _lens, _i))


@pytest.mark.parametrize("dt,hd,g,hkv,lens,seed", CASES)
def test_random_small_decode_both_kernels(pa, dt, hd, g, hkv, lens, seed):
    w = W.decode_workload("rand", dt, 16, g * hkv, hkv, hd, lens, seed=seed)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    for kernel in (1, 2):
        for ctas in (0, 1, 3):
            compare(w, run_decode(pa, w, kc, vc, bt, kernel=kernel, ctas=ctas), exact)


def test_zero_length_sequence_gives_zero_row(pa):
    w = W.decode_workload("z", "bf16", 16, 8, 2, 128, [5, 1, 40], seed=9)
    kc, vc, bt = device_caches(w, DEV)
    w0 = W.decode_workload("z", "bf16", 16, 8, 2, 128, [5, 1, 40], seed=9)
    w0.seq_lens = np.array([5, 0, 40], np.int32)
    exact = oracle_attention(w)
    for kernel in (1, 2):
        out = run_decode(pa, w0, kc, vc, bt, kernel=kernel, max_context=40)
        assert torch.count_nonzero(out[1]).item() == 0
        compare(w, out[[0, 2]], exact[[0, 2]])


@pytest.mark.parametrize("kernel", [1, 2])
def test_permuting_physical_blocks_is_bit_identical(pa, kernel):
    w = W.decode_workload("perm", "bf16", 16, 32, 8, 128, [700, 33, 1, 250, 16], seed=5)
    kc, vc, bt = device_caches(w, DEV)
    base = run_decode(pa, w, kc, vc, bt, kernel=kernel)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_blocks)).to(DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_decode(pa, w, kc2, vc2, bt2, kernel=kernel)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


def test_split_count_invariance_within_tolerance(pa):
    w = W.decode_workload("split", "bf16", 16, 32, 8, 128, [2000, 1500, 37], seed=6)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    outs = [run_decode(pa, w, kc, vc, bt, kernel=2, ctas=c) for c in (1, 2, 7, 40, 300)]
    for o in outs:
        compare(w, o, exact)


def test_check_mode_rejects_bad_tables(pa):
    w = W.decode_workload("chk", "bf16", 16, 8, 2, 128, [20, 40], seed=1)
    kc, vc, bt = device_caches(w, DEV)
    bad = bt.clone()
    bad[1, 1] = w.num_blocks + 3
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.empty(2, 8, 128, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    pa.pa_set_check_mode(True)
    try:
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_decode(out, w.q.to(DEV), kc, vc, bad, lens, 40, w.scale, workspace=ws)
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, 30, w.scale, workspace=ws)  # L > max_context
        pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, 40, w.scale, workspace=ws)
    finally:
        pa.pa_set_check_mode(False)
    with pytest.raises(pa.PAError, match="PA_ERR_WORKSPACE"):
        pa.pa_decode(out, w.q.to(DEV), kc, vc, bt, lens, 40, w.scale, workspace=ws[:16])


# ---------------------------------------------------------------- fused append + decode

APPEND_CASES = [
    ("tiny", lambda: W.tiny_decode()),
    ("gqa24", lambda: W.decode_workload("ap_gqa", "bf16", 16, 32, 8, 128, W.gqa_batch_lengths(24), seed=21)),
    ("mha", lambda: W.decode_workload("ap_mha", "f16", 16, 8, 8, 128, [1, 16, 17, 300, 33], std=0.5, seed=22)),
    ("g12_hd64", lambda: W.decode_workload("ap_g12", "bf16", 16, 24, 2, 64, [1, 2, 15, 16, 47, 129], seed=23)),
    ("hd256", lambda: W.decode_workload("ap_256", "bf16", 16, 8, 2, 256, [5, 64, 200], seed=24)),
]


@pytest.mark.parametrize("name,make", APPEND_CASES)
@pytest.mark.parametrize("kernel", [0, 1])
def test_decode_append_equals_write_then_decode(pa, name, make, kernel):
    """One call writes each sequence's new token at slot(L-1) and attends:
    the pool must equal the oracle's after the write (bit for bit) and the
    output must match the oracle's attention over the written pool."""
    w = make()
    kc, vc, bt = device_caches(w, DEV, after_step=False)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, kernel)
    try:
        ws_bytes = pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                               mc, W.TORCH_DTYPES[w.dtype])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype],
                         device=DEV)
        pa.pa_decode_append(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc, vc,
                            bt, lens, mc, w.scale, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
    finally:
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, 0)
    okc, ovc = oracle_caches(w)
    from helpers import oracle_bits, raw_bits

    assert np.array_equal(raw_bits(kc), oracle_bits(okc)) and np.array_equal(raw_bits(vc), oracle_bits(ovc))
    compare(w, out, oracle_attention(w, okc, ovc))


# ---------------------------------------------------------------- other block sizes

BS_CASES = []
_r3 = np.random.default_rng(321)
# 8 and multiples of 16: TMA boxes; 1, 2, 4, 12, 24: the row gather
for _bs in (1, 2, 4, 8, 12, 24, 32, 64, 128, 256):
    for _i in range(2):
        _hd = int(_r3.choice([64, 128]))
        _g = int(_r3.choice([1, 4, 6]))
        _lens = _r3.integers(1, 3 * _bs + 40, int(_r3.integers(1, 7))).tolist()
        _lens[0] = int(_r3.choice([1, _bs, _bs + 1, 2 * _bs]))
        BS_CASES.append((_bs, _hd, _g, _lens, 400 + 10 * _bs + _i))


@pytest.mark.parametrize("bs,hd,g,lens,seed", BS_CASES)
def test_decode_block_sizes_both_kernels(pa, bs, hd, g, lens, seed):
    w = W.decode_workload("bs", "bf16", bs, 2 * g, 2, hd, lens, seed=seed)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    for kernel in (1, 2):
        for ctas in ((0, 3) if kernel == 2 else (0,)):
            compare(w, run_decode(pa, w, kc, vc, bt, kernel=kernel, ctas=ctas), exact)


@pytest.mark.parametrize("bs", [1, 4, 12])
def test_gathered_block_sizes_are_bit_identical_under_relabelling(pa, bs):
    """The row-gather tiles (block sizes no TMA box fits) read blocks only
    through the table: relabelling physical blocks changes no bit."""
    w = W.decode_workload("gperm", "bf16", bs, 16, 4, 128, [1, 3 * bs + 1, 700, 33], seed=60 + bs)
    kc, vc, bt = device_caches(w, DEV)
    base = run_decode(pa, w, kc, vc, bt, kernel=2)
    perm = torch.from_numpy(np.random.default_rng(bs).permutation(w.num_blocks)).to(DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_decode(pa, w, kc2, vc2, bt2, kernel=2)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("bs", [1, 4, 8, 24, 32, 128])
def test_decode_append_block_sizes(pa, bs):
    w = W.decode_workload("ap_bs", "bf16", bs, 8, 2, 128, [1, max(bs - 1, 2), bs, bs + 1, 3 * bs + 5], seed=bs)
    kc, vc, bt = device_caches(w, DEV, after_step=False)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    ws = torch.empty(max(pa.pa_decode_workspace_size(w.num_seqs, 8, 2, 128, bs, mc, torch.bfloat16), 16),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty((w.num_seqs, 8, 128), dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_append(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc, vc, bt,
                        lens, mc, w.scale, workspace=ws)
    torch.cuda.synchronize()
    okc, ovc = oracle_caches(w)
    from helpers import oracle_bits, raw_bits

    assert np.array_equal(raw_bits(kc), oracle_bits(okc)) and np.array_equal(raw_bits(vc), oracle_bits(ovc))
    compare(w, out, oracle_attention(w, okc, ovc))


# ---------------------------------------------------------------- CUDA-graph replay

def test_graph_replays_of_decode_follow_new_queries(pa):
    w = W.decode_workload("graph", "bf16", 16, 32, 8, 128, [2000, 1500, 37, 700, 16], seed=41)
    kc, vc, bt = device_caches(w, DEV)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    graph_replays_match_eager(
        lambda out, q, ws: pa.pa_decode(out, q, kc, vc, bt, lens, mc, w.scale, workspace=ws), w.q.to(DEV).clone(), DEV)


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_expiry_is_reported_and_the_context_survives(pa):
    """A barrier wait that nothing completes gives up after its bound, the
    kernel sets the timeout bit, pa_device_status reports PA_ERR_TIMEOUT and
    clears it, and the next decode runs normally."""
    pa.pa_device_status(clear=True)
    pa.pa_selftest_wait_timeout(2000)
    with pytest.raises(pa.PAError, match="PA_ERR_TIMEOUT"):
        pa.pa_device_status(clear=True)
    pa.pa_device_status(clear=True)  # cleared: no error now
    w = W.decode_workload("after_timeout", "bf16", 16, 8, 2, 128, [40, 3, 200], seed=81)
    kc, vc, bt = device_caches(w, DEV)
    compare(w, run_decode(pa, w, kc, vc, bt), oracle_attention(w))


# ---------------------------------------------------------------- batches beyond one launch

def test_more_sequences_than_one_launch_takes(pa):
    """5,000 sequences: the library cuts the batch into launches of at most
    4,096 sequences on one workspace; every row matches the oracle, for the
    plain decode and the fused generation step."""
    lens = np.random.default_rng(91).integers(1, 60, 5000).tolist()
    w = W.decode_workload("many", "bf16", 16, 8, 2, 128, lens, seed=91)
    kc, vc, bt = device_caches(w, DEV)
    okc, ovc = oracle_caches(w)
    exact = oracle_attention(w, okc, ovc)
    compare(w, run_decode(pa, w, kc, vc, bt), exact)
    # the generation step from the pre-step pool
    kc2, vc2, _ = device_caches(w, DEV, after_step=False)
    mc = int(w.seq_lens.max())
    ws = torch.empty(max(pa.pa_decode_workspace_size(w.num_seqs, 8, 2, 128, 16, mc, torch.bfloat16), 16),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((w.num_seqs, 8, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_append(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc2, vc2,
                        bt, torch.from_numpy(w.seq_lens).to(DEV), mc, w.scale, workspace=ws)
    torch.cuda.synchronize()
    from helpers import oracle_bits, raw_bits

    assert np.array_equal(raw_bits(kc2), oracle_bits(okc)) and np.array_equal(raw_bits(vc2), oracle_bits(ovc))
    compare(w, out, exact)
