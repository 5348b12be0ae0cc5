"""GPU parity of the quantized (FP8 E4M3) cache: pa_write_kv_fp8 against the
oracle's quantizing write (codes and scales bit for bit, NaN canaries in the
untouched slots included), pa_decode_fp8 against the oracle's attention over
the codes' exact values (tolerance of the query type: |gpu - exact| <= atol +
rtol |exact|, helpers.ATOL / RTOL), and the copy-on-write block copy of code
and scale pools.  Both decode kernels (tensor-core and CUDA-core) are run.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_116_gb300 import workloads as W

from helpers import (FP8_NAN_CODE, device_fp8_caches, graph_replays_match_eager, oracle_fp8_attention,
                     oracle_fp8_caches, within_tol)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=0, ctas=0, lens=None, max_context=None):
    pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, kernel)
    pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, ctas)
    try:
        seq_lens = w.seq_lens if lens is None else lens
        mc = int(seq_lens.max()) if max_context is None else max_context
        ws_bytes = pa.pa_decode_fp8_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                   w.block_size, mc, W.TORCH_DTYPES[w.dtype])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype],
                         device=DEV)
        pa.pa_decode_fp8(out, w.q.to(DEV), kc, vc, ks, vs, bt, torch.from_numpy(seq_lens).to(DEV), mc, w.scale,
                         workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
        return out
    finally:
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, 0)
        pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, 0)


def compare(w, out, exact):
    ok, err = within_tol(out.double().cpu().numpy(), exact, w.dtype)
    assert ok, "max error %.3g beyond tolerance (%s)" % (err, w.name)
    return err


def assert_pools_equal(dev_pools, ora_pools):
    kc, vc, ks, vs = dev_pools
    okc, ovc, oks, ovs = ora_pools
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))


# ---------------------------------------------------------------- the quantizing write

WRITE_CASES = [
    ("tiny_f32", lambda: W.tiny_decode()),
    ("bf16_g4", lambda: W.decode_workload("w_bf16", "bf16", 16, 32, 8, 128, [1, 15, 16, 17, 300], seed=31)),
    ("f16_mha", lambda: W.decode_workload("w_f16", "f16", 16, 8, 8, 128, [40, 3], std=0.5, seed=32)),
    ("bs8_hd64", lambda: W.decode_workload("w_bs8", "bf16", 8, 4, 2, 64, [9, 8, 1, 30], seed=33)),
    ("bs32_hd96", lambda: W.decode_workload("w_bs32", "f16", 32, 6, 3, 96, [70, 33], seed=34)),
    ("hd256", lambda: W.decode_workload("w_256", "bf16", 16, 4, 1, 256, [20, 48], std=3.0, seed=35)),
]


@pytest.mark.parametrize("name,make", WRITE_CASES)
def test_write_kv_fp8_matches_oracle_bit_for_bit(pa, name, make):
    w = make()
    kc, vc, ks, vs, _ = device_fp8_caches(w, DEV)
    torch.cuda.synchronize()
    assert_pools_equal((kc, vc, ks, vs), oracle_fp8_caches(w))


def test_write_kv_fp8_special_rows(pa):
    """An all-zero row keeps scale 1 and zero codes; beside a huge (or a
    unit) element the rest of a row rounds to small or signed-zero codes;
    negative slots write nothing."""
    hkv, hd, bs, nb = 2, 128, 16, 4
    k = torch.randn(5, hkv, hd, dtype=torch.float32)
    v = torch.randn(5, hkv, hd, dtype=torch.float32)
    k[0] = 0.0
    v[1, 0, 7] = 3.0e4
    k[3, 1] = -1e-30  # next to 1.0 these round to (signed) zero codes
    k[3, 1, 0] = 1.0
    slots = torch.tensor([3, 17, -1, 63, 40], dtype=torch.int64)
    dk = torch.full((nb, bs, hkv, hd), FP8_NAN_CODE, dtype=torch.uint8, device=DEV)
    dv = torch.full_like(dk, FP8_NAN_CODE)
    dks = torch.full((nb, hkv, bs), float("nan"), device=DEV)
    dvs = torch.full_like(dks, float("nan"))
    pa.pa_write_kv_fp8(k.to(DEV), v.to(DEV), slots.to(DEV), dk, dv, dks, dvs)
    torch.cuda.synchronize()
    ok = np.full((nb, bs, hkv, hd), FP8_NAN_CODE, np.uint8)
    ov = ok.copy()
    oks = np.full((nb, hkv, bs), np.nan, np.float32)
    ovs = oks.copy()
    oracle.write_kv_fp8(k.numpy(), v.numpy(), "f32", slots.numpy(), ok, ov, oks, ovs)
    assert_pools_equal((dk, dv, dks, dvs), (ok, ov, oks, ovs))
    assert oks[0, 0, 3] == 1.0 and np.all(ok[0, 3, 0] == 0)
    assert np.all(ok[3, 15, 1, 1:] == 0x80) and ok[3, 15, 1, 0] == 0x7E  # slot 63


def test_write_kv_fp8_check_mode(pa):
    dk = torch.zeros((4, 16, 2, 128), dtype=torch.uint8, device=DEV)
    dv = torch.zeros_like(dk)
    dks = torch.zeros((4, 2, 16), device=DEV)
    dvs = torch.zeros_like(dks)
    k = torch.randn(2, 2, 128, device=DEV, dtype=torch.bfloat16)
    pa.pa_set_check_mode(True)
    try:
        for bad in ([5, 5], [0, 64]):
            with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
                pa.pa_write_kv_fp8(k, k, torch.tensor(bad, device=DEV), dk, dv, dks, dvs)
        pa.pa_write_kv_fp8(k, k, torch.tensor([0, 63], device=DEV), dk, dv, dks, dvs)
    finally:
        pa.pa_set_check_mode(False)


# ---------------------------------------------------------------- decode over the quantized cache

def test_gqa_decode_batch_fp8_full(pa):
    """The 64-sequence GQA batch (bf16 queries, Hq 32, Hkv 8, head_dim 128,
    block size 16) over an FP8 cache, every output element."""
    w = W.gqa_decode_batch(device=DEV)
    pools = device_fp8_caches(w, DEV)
    kc, vc, ks, vs, bt = pools
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    exact = oracle_fp8_attention(w, *opools)
    for kernel in (0, 1):
        compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=kernel), exact)


def test_mha_decode_fp8_full(pa):
    """The 13B-style MHA batch (f16, Hq = Hkv = 40, N(0, 0.5) values, all 128
    sequences of its lognormal length mix) over an FP8 cache."""
    w = W.mha_decode(device=DEV)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    exact = oracle_fp8_attention(w, *opools)
    compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt), exact)


@pytest.mark.parametrize("pair", [1, 2])
def test_long_context_decode_fp8_full(pa, pair):
    """8 x 32,768 tokens over an FP8 cache, all eight sequences, with the
    32-token pair step off (1) and on (2)."""
    w = W.long_context_decode(device=DEV)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, pair)
    try:
        compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt), exact)
    finally:
        pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 0)


def test_tiny_decode_fp8_fp32_queries(pa):
    """fp32 queries run on the CUDA-core kernel and meet the fp32 bound."""
    w = W.tiny_decode()
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    assert compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt), exact) < 1e-5


FP8_CASES = []
_r = np.random.default_rng(808)
for _i in range(12):
    _hd = int(_r.choice([128, 256, 64]))
    _g = int(_r.choice([1, 2, 4, 6, 8, 12, 16]))
    _hkv = int(_r.choice([1, 2, 4]))
    _dt = str(_r.choice(["bf16", "f16"]))
    _bs = int(_r.choice([8, 16, 16, 32, 64]))
    _lens = _r.integers(1, 3 * _bs + 9, int(_r.integers(1, 8))).tolist()
    _lens[0] = int(_r.choice([1, _bs, _bs + 1, 2 * _bs]))
    FP8_CASES.append((_dt, _hd, _g, _hkv, _bs, _lens, 900 + _i))


@pytest.mark.parametrize("dt,hd,g,hkv,bs,lens,seed", FP8_CASES)
def test_random_small_fp8_decode_both_kernels(pa, dt, hd, g, hkv, bs, lens, seed):
    w = W.decode_workload("fp8_rand", dt, bs, g * hkv, hkv, hd, lens, seed=seed)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    exact = oracle_fp8_attention(w, *opools)
    tc_ok = hd in (128, 256)
    for kernel in ((1, 2) if tc_ok else (1,)):
        for ctas in ((0, 1, 5) if kernel == 2 else (0,)):
            compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=kernel, ctas=ctas), exact)
    if not tc_ok:
        with pytest.raises(pa.PAError, match="PA_ERR_UNSUPPORTED"):
            run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=2)


@pytest.mark.parametrize("bs", [8, 32, 128, 256])
def test_fp8_decode_block_sizes(pa, bs):
    w = W.decode_workload("fp8_bs", "bf16", bs, 16, 4, 128, [1, bs - 1, bs, bs + 1, 3 * bs + 5], seed=bs + 7)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    for kernel in (1, 2):
        compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=kernel), exact)


def test_fp8_zero_length_sequence_gives_zero_row(pa):
    w = W.decode_workload("fp8_z", "bf16", 16, 8, 2, 128, [5, 1, 40], seed=19)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    lens0 = np.array([5, 0, 40], np.int32)
    for kernel in (1, 2):
        out = run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=kernel, lens=lens0, max_context=40)
        assert torch.count_nonzero(out[1]).item() == 0
        ok, err = within_tol(out[[0, 2]].double().cpu().numpy(), exact[[0, 2]], "bf16")
        assert ok, err


def test_fp8_permuting_physical_blocks_is_bit_identical(pa):
    w = W.decode_workload("fp8_perm", "bf16", 16, 32, 8, 128, [700, 33, 1, 250, 16], seed=15)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    base = run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=2)
    perm = torch.from_numpy(np.random.default_rng(2).permutation(w.num_blocks)).to(DEV)
    moved = []
    for t in (kc, vc, ks, vs):
        u = torch.empty_like(t)
        u[perm] = t
        moved.append(u)
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_decode_fp8(pa, w, *moved, bt2, kernel=2)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


def test_fp8_split_count_invariance_within_tolerance(pa):
    w = W.decode_workload("fp8_split", "f16", 16, 32, 8, 128, [2000, 1500, 37], seed=16)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    for c in (1, 2, 7, 40, 300):
        compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=2, ctas=c), exact)


def test_fp8_decode_rejects_misaligned_scales(pa):
    w = W.decode_workload("fp8_al", "bf16", 16, 8, 2, 128, [20], seed=17)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    flat = torch.zeros(ks.numel() + 1, device=DEV)
    bad = flat[1:].view(ks.shape)  # 4-byte offset
    with pytest.raises(pa.PAError, match="PA_ERR_INVALID_ARG"):
        run_decode_fp8(pa, w, kc, vc, bad, vs, bt)


# ---------------------------------------------------------------- copy-on-write of a quantized pool

def test_copy_blocks_of_fp8_pools_is_bit_exact(pa):
    """Code pools copy as PA_FP8_E4M3 blocks, scale pools as fp32 blocks of
    head_dim 1; two layers; compared with the oracle's block copy."""
    w = W.decode_workload("fp8_cow", "bf16", 16, 8, 2, 128, [40, 17, 100], seed=18)
    layers = [device_fp8_caches(w, DEV) for _ in range(2)]
    opools = oracle_fp8_caches(w)
    pairs = np.array([[int(w.block_tables[0, 0]), int(w.block_tables[1, 1])],
                      [int(w.block_tables[2, 3]), int(w.block_tables[0, 2])]], np.int64)
    # destinations must not be read elsewhere in this call: they are not sources
    assert not set(pairs[:, 1]) & set(pairs[:, 0])
    dp = torch.from_numpy(pairs).to(DEV)
    pa.pa_copy_blocks([l[0] for l in layers], [l[1] for l in layers], dp)
    pa.pa_copy_blocks([l[2] for l in layers], [l[3] for l in layers], dp)
    torch.cuda.synchronize()
    okc, ovc, oks, ovs = (a.copy() for a in opools)
    oracle.copy_blocks([okc], [ovc], pairs)
    oracle.copy_blocks([oks], [ovs], pairs)
    for l in layers:
        assert_pools_equal(l[:4], (okc, ovc, oks, ovs))


def test_graph_replays_of_fp8_decode_follow_new_queries(pa):
    w = W.decode_workload("fp8_graph", "bf16", 16, 32, 8, 128, [2000, 1500, 37, 700, 16], seed=42)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    graph_replays_match_eager(
        lambda out, q, ws: pa.pa_decode_fp8(out, q, kc, vc, ks, vs, bt, lens, mc, w.scale, workspace=ws),
        w.q.to(DEV).clone(), DEV)


# ---------------------------------------------------------------- the generation step over a quantized cache

APPEND_FP8_CASES = [
    ("gqa24_bf16", lambda: W.decode_workload("ap8_gqa", "bf16", 16, 32, 8, 128, W.gqa_batch_lengths(24), seed=61)),
    ("mha_f16", lambda: W.decode_workload("ap8_mha", "f16", 16, 8, 8, 128, [1, 16, 17, 300, 33], std=0.5, seed=62)),
    ("g12_bs8", lambda: W.decode_workload("ap8_g12", "bf16", 8, 24, 2, 128, [1, 7, 8, 9, 47, 129], seed=63)),
    ("bs32", lambda: W.decode_workload("ap8_bs32", "bf16", 32, 8, 2, 128, [1, 31, 32, 33, 100], seed=64)),
    ("hd256", lambda: W.decode_workload("ap8_256", "bf16", 16, 8, 2, 256, [5, 64, 200], seed=65)),
    ("hd64", lambda: W.decode_workload("ap8_64", "f16", 16, 8, 2, 64, [3, 40], seed=66)),
    ("tiny_f32", lambda: W.tiny_decode()),
]


@pytest.mark.parametrize("name,make", APPEND_FP8_CASES)
@pytest.mark.parametrize("kernel", [0, 1])
def test_decode_append_fp8_equals_quantizing_write_then_decode(pa, name, make, kernel):
    """One call quantizes each sequence's new token into the slot of position
    L-1 and attends: the code and scale pools must equal the oracle's after
    its quantizing write (bit for bit, untouched slots included) and the
    output must match the oracle's attention over them."""
    w = make()
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV, after_step=False)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, kernel)
    try:
        ws_bytes = pa.pa_decode_fp8_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                   w.block_size, mc, W.TORCH_DTYPES[w.dtype])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=W.TORCH_DTYPES[w.dtype],
                         device=DEV)
        pa.pa_decode_append_fp8(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc,
                                vc, ks, vs, bt, lens, mc, w.scale, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
    finally:
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, 0)
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    compare(w, out, oracle_fp8_attention(w, *opools))


def test_decode_append_fp8_zero_length_sequence(pa):
    w = W.decode_workload("ap8_z", "bf16", 16, 8, 2, 128, [5, 1, 40], seed=67)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV, after_step=False)
    before = [t.clone() for t in (kc, vc, ks, vs)]
    lens0 = torch.tensor([5, 0, 40], dtype=torch.int32, device=DEV)
    ws = torch.empty(max(pa.pa_decode_fp8_workspace_size(3, 8, 2, 128, 16, 40, torch.bfloat16), 16),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((3, 8, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_append_fp8(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc, vc, ks,
                            vs, bt, lens0, 40, w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]).item() == 0
    # sequence 1 wrote nothing: its block (and every other untouched slot) is as before
    blk = int(w.block_tables[1, 0])
    assert torch.equal(kc[blk], before[0][blk]) and torch.equal(ks[blk].view(torch.int32),
                                                                before[2][blk].view(torch.int32))


@pytest.mark.parametrize("ctas", [1, 5, 37, 200])
def test_decode_append_fp8_any_split(pa, ctas):
    """The fused step with the batch cut at many places: whichever warp ends
    up owning a unit's last tile quantizes and writes the new rows."""
    w = W.decode_workload("ap8_split", "bf16", 16, 16, 4, 128, [1, 2, 3, 4, 5, 40, 47, 48, 49, 300, 1000], seed=71)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV, after_step=False)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, ctas)
    try:
        ws = torch.empty(max(pa.pa_decode_fp8_workspace_size(w.num_seqs, 16, 4, 128, 16, mc, torch.bfloat16), 16),
                         dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, 16, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        pa.pa_decode_append_fp8(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc,
                                vc, ks, vs, bt, lens, mc, w.scale, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
    finally:
        pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, 0)
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    compare(w, out, oracle_fp8_attention(w, *opools))


# ---------------------------------------------------------------- the 32-token pair step

PAIR_CASES = [
    # (dtype, block_size, G, Hkv, lengths): odd and even tile counts, a last
    # tile of 1..16 tokens, one-tile units, 8-token blocks
    ("bf16", 16, 4, 8, [1, 16, 17, 31, 32, 33, 48, 300, 2047, 3360]),
    ("f16", 16, 1, 8, [2, 15, 64, 65, 129, 1000]),
    ("bf16", 8, 8, 2, [1, 7, 8, 9, 16, 17, 40, 257]),
    ("f16", 32, 6, 2, [31, 32, 33, 95, 96, 97, 500]),
    ("bf16", 64, 2, 4, [1, 63, 64, 65, 700]),
]


@pytest.mark.parametrize("dt,bs,g,hkv,lens", PAIR_CASES)
def test_fp8_pair_step_never_and_always_match_oracle(pa, dt, bs, g, hkv, lens):
    """The code-cache kernel with and without the pair step (head_dim 128,
    G <= 8), over several splits of the batch, against the oracle."""
    w = W.decode_workload("fp8_pair", dt, bs, g * hkv, hkv, 128, lens, seed=bs * 31 + g)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    try:
        for mode in (1, 2):
            pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, mode)
            for ctas in (0, 1, 5, 37):
                compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=2, ctas=ctas), exact)
    finally:
        pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 0)


@pytest.mark.parametrize("ctas", [0, 1, 5, 37])
def test_fp8_pair_step_with_the_new_token(pa, ctas):
    """The fused generation step with pair steps forced: the tile the new
    token goes to is worked alone, the pools match the oracle bit for bit."""
    w = W.decode_workload("ap8_pair", "bf16", 16, 32, 8, 128, [1, 2, 16, 17, 33, 300, 1001, 2048], seed=73)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV, after_step=False)
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    mc = int(w.seq_lens.max())
    pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 2)
    pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, ctas)
    try:
        ws = torch.empty(max(pa.pa_decode_fp8_workspace_size(w.num_seqs, 32, 8, 128, 16, mc, torch.bfloat16), 16),
                         dtype=torch.uint8, device=DEV)
        out = torch.full((w.num_seqs, 32, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        pa.pa_decode_append_fp8(out, w.q.to(DEV), w.new_k.to(DEV).contiguous(), w.new_v.to(DEV).contiguous(), kc,
                                vc, ks, vs, bt, lens, mc, w.scale, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)
    finally:
        pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 0)
        pa.pa_set_option(pa.PA_OPT_DECODE_CTAS, 0)
    opools = oracle_fp8_caches(w)
    assert_pools_equal((kc, vc, ks, vs), opools)
    compare(w, out, oracle_fp8_attention(w, *opools))


def test_fp8_pair_step_permuting_physical_blocks_is_bit_identical(pa):
    w = W.decode_workload("fp8_pperm", "bf16", 16, 32, 8, 128, [700, 33, 1, 250, 16, 2500], seed=74)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 2)
    try:
        base = run_decode_fp8(pa, w, kc, vc, ks, vs, bt, kernel=2)
        perm = torch.from_numpy(np.random.default_rng(3).permutation(w.num_blocks)).to(DEV)
        moved = []
        for t in (kc, vc, ks, vs):
            u = torch.empty_like(t)
            u[perm] = t
            moved.append(u)
        bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
        again = run_decode_fp8(pa, w, *moved, bt2, kernel=2)
    finally:
        pa.pa_set_option(pa.PA_OPT_FP8_PAIR_STEP, 0)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


def test_fp8_decode_more_sequences_than_one_launch_takes(pa):
    lens = np.random.default_rng(92).integers(1, 60, 5000).tolist()
    w = W.decode_workload("many8", "bf16", 16, 8, 2, 128, lens, seed=92)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    exact = oracle_fp8_attention(w, *oracle_fp8_caches(w))
    compare(w, run_decode_fp8(pa, w, kc, vc, ks, vs, bt), exact)


# ---------------------------------------------------------------- varlen over the quantized cache

def run_varlen_fp8(pa, w, pools, causal=None, kernel=0, planned=False):
    """kernel: 0 automatic, 1 CUDA-core, 2 tcgen05; planned: pass the workspace
    that lets the tcgen05 kernel run its work longest first."""
    kc, vc, ks, vs, bt = pools
    out = torch.full(tuple(w.q.shape), float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
    mq, mc = int(w.query_lens.max()), int(w.seq_lens.max())
    pa.pa_set_option(pa.PA_OPT_VARLEN_KERNEL, kernel)
    try:
        ws = None
        if planned:
            n = pa.pa_varlen_fp8_workspace_size(w.num_seqs, int(w.query_lens.sum()), mq, w.num_heads, w.num_kv_heads,
                                                w.head_dim, w.block_size, mc, W.TORCH_DTYPES[w.dtype])
            ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
        pa.pa_varlen_fp8(out, w.q.to(DEV), kc, vc, ks, vs, bt, torch.from_numpy(w.seq_lens).to(DEV),
                         torch.from_numpy(w.query_start_loc).to(DEV), mq, mc, w.scale,
                         causal=w.causal if causal is None else causal, workspace=ws)
        torch.cuda.synchronize()
        pa.pa_device_status(clear=True)  # raises if a bounded wait ran out
    finally:
        pa.pa_set_option(pa.PA_OPT_VARLEN_KERNEL, 0)
    return out


def varlen_fp8_kernels(w):
    """(kernel, planned) pairs that apply to w: the CUDA-core kernel always;
    the tcgen05 kernel (with and without the plan) for bf16/f16 queries,
    head_dim 128 and block size 8 or a multiple of 16."""
    runs = [(1, False)]
    if w.dtype in ("bf16", "f16") and w.head_dim == 128 and (w.block_size == 8 or w.block_size % 16 == 0):
        runs += [(2, False), (2, True)]
    return runs


def oracle_varlen_fp8(w, opools, causal):
    kc, vc, ks, vs = opools
    return oracle.paged_attention_fp8(W.raw_numpy(w.q), w.dtype, kc, vc, ks, vs, w.block_tables, w.seq_lens,
                                      w.query_start_loc, w.scale, causal)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_fp8_handbook_layout(pa, dtype):
    """The handbook's three requests (a decode, a full prefill, a chunk after
    cached context) over an FP8 cache, causal and not."""
    w = W.handbook_check(dtype=dtype)
    pools = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal(pools[:4], opools)
    for causal in (True, False):
        exact = oracle_varlen_fp8(w, opools, causal)
        for kernel, planned in varlen_fp8_kernels(w):
            err = compare(w, run_varlen_fp8(pa, w, pools, causal=causal, kernel=kernel, planned=planned), exact)
            if dtype == "f32":
                assert err < 1e-5


def test_varlen_fp8_mixed_step_with_cow_full(pa):
    """The mixed varlen step (16 prefill chunks after cached context, 240
    decode rows of 60 sampling groups sharing a prompt, the copy-on-write of
    the shared tails) over an FP8 cache: codes and scales bit-exact after
    the step's quantizing writes and block copies, attention against the
    oracle with num_new > 1."""
    w = W.mixed_varlen(device=DEV)
    pools = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal(pools[:4], opools)
    exact = oracle_varlen_fp8(w, opools, True)
    for kernel, planned in varlen_fp8_kernels(w):
        compare(w, run_varlen_fp8(pa, w, pools, kernel=kernel, planned=planned), exact)


VARLEN_FP8_CASES = []
_r4 = np.random.default_rng(909)
for _i in range(8):
    _bs = int(_r4.choice([1, 4, 16, 32]))
    _hd = int(_r4.choice([64, 96, 128]))
    _g = int(_r4.choice([1, 3, 6, 12]))
    _hkv = int(_r4.choice([1, 2]))
    _dt = str(_r4.choice(["f32", "bf16", "f16"]))
    _S = int(_r4.integers(1, 6))
    _lens = _r4.integers(1, 3 * _bs + 60, _S)
    _q = np.minimum(_lens, _r4.integers(1, 50, _S))
    _q[_r4.random(_S) < 0.3] = 1
    VARLEN_FP8_CASES.append((_dt, _bs, _hd, _g, _hkv, _lens.tolist(), _q.tolist(), 950 + _i))


@pytest.mark.parametrize("dt,bs,hd,g,hkv,lens,qlens,seed", VARLEN_FP8_CASES)
def test_random_varlen_fp8(pa, dt, bs, hd, g, hkv, lens, qlens, seed):
    w = W.varlen_workload("vfp8", dt, bs, g * hkv, hkv, hd, lens, qlens, seed=seed)
    pools = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal(pools[:4], opools)
    for causal in (True, False):
        exact = oracle_varlen_fp8(w, opools, causal)
        for kernel, planned in varlen_fp8_kernels(w):
            compare(w, run_varlen_fp8(pa, w, pools, causal=causal, kernel=kernel, planned=planned), exact)


TC_VARLEN_FP8_CASES = []
_r5 = np.random.default_rng(919)
for _i in range(8):
    _bs = int(_r5.choice([8, 16, 32, 64]))
    _g = int(_r5.choice([1, 2, 3, 6, 8, 12]))
    _hkv = int(_r5.choice([1, 2, 4]))
    _dt = str(_r5.choice(["bf16", "f16"]))
    _S = int(_r5.integers(1, 7))
    _q = _r5.integers(1, 300, _S)
    _q[_r5.random(_S) < 0.4] = 1  # decode rows mixed in
    _cached = _r5.integers(0, 400, _S)
    TC_VARLEN_FP8_CASES.append((_dt, _bs, _g, _hkv, (_cached + _q).tolist(), _q.tolist(), 970 + _i))


@pytest.mark.parametrize("dt,bs,g,hkv,lens,qlens,seed", TC_VARLEN_FP8_CASES)
def test_random_varlen_fp8_tensor_core(pa, dt, bs, g, hkv, lens, qlens, seed):
    """head_dim 128 shapes the tcgen05 kernel takes over a code cache: several
    128-key tiles, both query tiles of a pair, partial last tiles."""
    w = W.varlen_workload("vfp8tc", dt, bs, g * hkv, hkv, 128, lens, qlens, seed=seed)
    pools = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    for causal in (True, False):
        exact = oracle_varlen_fp8(w, opools, causal)
        for kernel, planned in varlen_fp8_kernels(w):
            compare(w, run_varlen_fp8(pa, w, pools, causal=causal, kernel=kernel, planned=planned), exact)


def test_varlen_fp8_permutation_bit_identical(pa):
    w = W.varlen_workload("perm_vfp8", "bf16", 16, 12, 2, 128, [300, 81, 17, 1000], [1, 81, 5, 130], seed=3)
    kc, vc, ks, vs, bt = device_fp8_caches(w, DEV)
    base = run_varlen_fp8(pa, w, (kc, vc, ks, vs, bt), kernel=2, planned=True)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(w.num_blocks)).to(DEV)
    pools2 = []
    for t in (kc, vc, ks, vs):
        t2 = torch.empty_like(t)
        t2[perm] = t
        pools2.append(t2)
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_varlen_fp8(pa, w, (*pools2, bt2), kernel=2, planned=True)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))



def test_varlen_fp8_long_contexts(pa):
    """Over the quantized cache: a chunk after 20,000 cached tokens and
    decode rows over 17,000 and 33,000 tokens (several table windows of the
    producers and of a decode warp), every kernel that applies."""
    w = W.varlen_workload("long_vfp8", "bf16", 16, 12, 2, 128, [20032, 17000, 33000, 150], [32, 1, 1, 150],
                          seed=77)
    pools = device_fp8_caches(w, DEV)
    opools = oracle_fp8_caches(w)
    assert_pools_equal(pools[:4], opools)
    exact = oracle_varlen_fp8(w, opools, True)
    for kernel, planned in varlen_fp8_kernels(w):
        compare(w, run_varlen_fp8(pa, w, pools, kernel=kernel, planned=planned), exact)
