"""GPU parity of pa_varlen (mixed prefill chunks and decode rows, causal or
not) against the oracle, including the copy-on-write mixed step."""
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


def run_varlen(pa, w, kc, vc, bt, causal=None, kernel=0, routed=False):
    """routed: pass a workspace of pa_varlen_workspace_size bytes (the
    library must accept both that and none)."""
    pa.pa_set_option(pa.PA_OPT_VARLEN_KERNEL, kernel)
    try:
        out = torch.full(tuple(w.q.shape), float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
        mq, mc = int(w.query_lens.max()), int(w.seq_lens.max())
        ws = None
        if routed:
            n = pa.pa_varlen_workspace_size(w.num_seqs, int(w.query_lens.sum()), mq, w.num_heads, w.num_kv_heads,
                                            w.head_dim, w.block_size, mc, W.TORCH_DTYPES[w.dtype])
            ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
        pa.pa_varlen(out, w.q.to(DEV), kc, vc, bt, torch.from_numpy(w.seq_lens).to(DEV),
                     torch.from_numpy(w.query_start_loc).to(DEV), mq, mc,
                     w.scale, causal=w.causal if causal is None else causal, workspace=ws)
        torch.cuda.synchronize()
        return out
    finally:
        pa.pa_set_option(pa.PA_OPT_VARLEN_KERNEL, 0)


def compare(w, out, exact):
    ok, err = within_tol(out.double().cpu().numpy(), exact, w.dtype)
    assert ok, "max error %.3g beyond tolerance (%s)" % (err, w.name)
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_handbook_layout(pa, dtype):
    w = W.handbook_check(dtype=dtype)
    kc, vc, bt = device_caches(w, DEV)
    for causal in (True, False):
        exact = oracle_attention(w, causal=causal)
        err = compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal), exact)
        if dtype == "f32":
            assert err < 1e-5


def test_mixed_varlen_with_cow_full(pa):
    w = W.mixed_varlen(device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    compare(w, run_varlen(pa, w, kc, vc, bt), exact)


CASES = []
_r = np.random.default_rng(77)
for _i in range(10):
    _bs = int(_r.choice([1, 4, 16, 32]))
    _hd = int(_r.choice([32, 64, 128]))
    _g = int(_r.choice([1, 3, 6]))
    _hkv = int(_r.choice([1, 2]))
    _dt = str(_r.choice(["f32", "bf16", "f16"]))
    _S = int(_r.integers(1, 6))
    _lens = _r.integers(1, 3 * _bs + 40, _S)
    _q = np.minimum(_lens, _r.integers(1, 70, _S))
    CASES.append((_dt, _bs, _hd, _g, _hkv, _lens.tolist(), _q.tolist(), _i))


@pytest.mark.parametrize("dt,bs,hd,g,hkv,lens,qlens,seed", CASES)
def test_random_small_varlen(pa, dt, bs, hd, g, hkv, lens, qlens, seed):
    w = W.varlen_workload("rand", dt, bs, g * hkv, hkv, hd, lens, qlens, seed=seed)
    kc, vc, bt = device_caches(w, DEV)
    for causal in (True, False):
        compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal), oracle_attention(w, causal=causal))


def test_check_mode_rejects_bad_cu_seqlens(pa):
    w = W.handbook_check()
    kc, vc, bt = device_caches(w, DEV)
    out = torch.empty(tuple(w.q.shape), device=DEV)
    cu = torch.from_numpy(w.query_start_loc).to(DEV)
    bad = cu.clone()
    bad[2] = bad[1] + 6  # request 1 would have 6 new tokens but context 5
    bad[3] = bad[2] + 8
    lens = torch.from_numpy(w.seq_lens).to(DEV)
    pa.pa_set_check_mode(True)
    try:
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_varlen(out, w.q.to(DEV), kc, vc, bt, lens, bad, 8, 37, w.scale)
        pa.pa_varlen(out, w.q.to(DEV), kc, vc, bt, lens, cu, 8, 37, w.scale)
    finally:
        pa.pa_set_check_mode(False)


TC_CASES = []
_r2 = np.random.default_rng(2024)
for _i in range(12):
    _hd = int(_r2.choice([64, 128]))
    _g = int(_r2.choice([1, 2, 3, 6, 8, 12]))
    _hkv = int(_r2.choice([1, 2, 4]))
    _dt = str(_r2.choice(["bf16", "f16"]))
    _S = int(_r2.integers(1, 9))
    _q = _r2.integers(1, 200, _S)
    _q[_r2.random(_S) < 0.4] = 1  # decode rows mixed in
    _cached = _r2.integers(0, 300, _S)
    _cached[0] = 0 if _S > 1 else _cached[0]  # a full prefill with no cached context
    TC_CASES.append((_dt, _hd, _g, _hkv, (_cached + _q).tolist(), _q.tolist(), _i))


@pytest.mark.parametrize("dt,hd,g,hkv,lens,qlens,seed", TC_CASES)
def test_random_varlen_tensor_core_kernels(pa, dt, hd, g, hkv, lens, qlens, seed):
    """The tcgen05 kernel (option 2), with and without a workspace argument."""
    w = W.varlen_workload("rand_tc", dt, 16, g * hkv, hkv, hd, lens, qlens, seed=100 + seed)
    kc, vc, bt = device_caches(w, DEV)
    for causal in (True, False):
        exact = oracle_attention(w, causal=causal)
        compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal, kernel=2), exact)
        compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal, kernel=2, routed=True), exact)


def test_varlen_kernels_agree_on_mixed_step(pa):
    w = W.mixed_varlen(num_chunks=4, num_groups=6, device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    for kernel in (1, 2):
        got = run_varlen(pa, w, kc, vc, bt, kernel=kernel).double().cpu().numpy()
        assert within_tol(got, exact, w.dtype)[0], "kernel %d" % kernel


def test_mixed_varlen_full_tcgen05(pa):
    w = W.mixed_varlen(device=DEV)
    kc, vc, bt = device_caches(w, DEV)
    compare(w, run_varlen(pa, w, kc, vc, bt, kernel=2, routed=True), oracle_attention(w))
    pa.pa_device_status(clear=True)  # raises if a kernel recorded a timeout


@pytest.mark.parametrize("kernel,routed", [(1, False), (2, False), (2, True)])
def test_varlen_permutation_bit_identical(pa, kernel, routed):
    w = W.varlen_workload("perm_v", "bf16", 16, 12, 2, 128, [300, 81, 17, 1000], [1, 81, 5, 130], seed=3)
    kc, vc, bt = device_caches(w, DEV)
    base = run_varlen(pa, w, kc, vc, bt, kernel=kernel, routed=routed)
    perm = torch.from_numpy(np.random.default_rng(4).permutation(w.num_blocks)).to(DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_varlen(pa, w, kc2, vc2, bt2, kernel=kernel, routed=routed)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
def test_varlen_tcgen05_block_sizes(pa, bs):
    rng = np.random.default_rng(bs)
    S = 5
    q = rng.integers(1, 150, S)
    q[1] = 1
    lens = q + rng.integers(0, 3 * bs, S)
    w = W.varlen_workload("vl_bs", "bf16", bs, 12, 2, 128, lens.tolist(), q.tolist(), seed=bs)
    kc, vc, bt = device_caches(w, DEV)
    for causal in (True, False):
        exact = oracle_attention(w, causal=causal)
        for routed in (False, True):
            compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal, kernel=2, routed=routed), exact)


HD256_CASES = []
_r3 = np.random.default_rng(256)
for _i in range(8):
    _g = int(_r3.choice([1, 2, 3, 4, 8, 12, 16]))
    _hkv = int(_r3.choice([1, 2]))
    _dt = str(_r3.choice(["bf16", "f16"]))
    _bs = int(_r3.choice([16, 32]))
    _S = int(_r3.integers(1, 7))
    _q = _r3.integers(1, 200, _S)
    _q[_r3.random(_S) < 0.4] = 1  # decode rows (the prefill path takes them at this head dim)
    _cached = _r3.integers(0, 300, _S)
    HD256_CASES.append((_dt, _bs, _g, _hkv, (_cached + _q).tolist(), _q.tolist(), _i))


@pytest.mark.parametrize("dt,bs,g,hkv,lens,qlens,seed", HD256_CASES)
def test_varlen_tcgen05_head_dim_256(pa, dt, bs, g, hkv, lens, qlens, seed):
    """head_dim 256 on the tensor cores: one query tile per CTA (S and O take
    384 tensor-memory columns) and one-slot K / V rings."""
    w = W.varlen_workload("hd256", dt, bs, g * hkv, hkv, 256, lens, qlens, seed=300 + seed)
    kc, vc, bt = device_caches(w, DEV)
    for causal in (True, False):
        exact = oracle_attention(w, causal=causal)
        for routed in (False, True):
            compare(w, run_varlen(pa, w, kc, vc, bt, causal=causal, kernel=2, routed=routed), exact)
    pa.pa_device_status(clear=True)  # raises if a kernel recorded a timeout


def test_varlen_head_dim_256_relabelling_bit_identical(pa):
    w = W.varlen_workload("perm_256", "bf16", 16, 8, 2, 256, [300, 81, 17, 700], [1, 81, 5, 130], seed=7)
    kc, vc, bt = device_caches(w, DEV)
    base = run_varlen(pa, w, kc, vc, bt, kernel=2, routed=True)
    compare(w, base, oracle_attention(w))
    perm = torch.from_numpy(np.random.default_rng(8).permutation(w.num_blocks)).to(DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    again = run_varlen(pa, w, kc2, vc2, bt2, kernel=2, routed=True)
    assert torch.equal(base.view(torch.int16), again.view(torch.int16))


def test_varlen_head_dim_256_block_size_8_takes_the_cuda_core_path(pa):
    w = W.varlen_workload("hd256_bs8", "bf16", 8, 4, 2, 256, [40, 9, 70], [12, 1, 30], seed=9)
    kc, vc, bt = device_caches(w, DEV)
    compare(w, run_varlen(pa, w, kc, vc, bt, kernel=0), oracle_attention(w))


# Parallel-sampling layouts: runs of decode rows forked from one prompt
# (their tables share the prompt's full blocks, each has its own blocks from
# the partial tail on, some with more cached tokens of their own), lone decode
# rows and prefill chunks between them.  (dtype, block size, head dim, G, Hkv)
FORK_CASES = [
    ("bf16", 16, 128, 6, 2),
    ("f16", 16, 128, 4, 2),
    ("bf16", 8, 64, 2, 3),
    ("bf16", 8, 128, 4, 1),
    ("bf16", 32, 128, 8, 1),
    ("f16", 16, 64, 1, 4),
    ("bf16", 64, 128, 3, 2),
    ("bf16", 16, 128, 12, 1),
]
FORK_LAYOUT = [("chunk", 40, 20), ("group", 37, [0, 5, 21, 3]), ("single", 50), ("group", 16, [0, 0, 17]),
               ("group", 7, [2, 9]), ("chunk", 3, 0), ("group", 300, [0, 0, 0, 0, 0]),
               ("group", 130, [40, 0, 77, 1, 2, 3, 4]), ("single", 1), ("group", 33, [0, 1])]


def decode_rows(w):
    return torch.from_numpy(w.query_start_loc[:-1][w.query_lens == 1].astype(np.int64)).to(DEV)


@pytest.mark.parametrize("dt,bs,hd,g,hkv", FORK_CASES)
def test_varlen_forked_decode_rows(pa, dt, bs, hd, g, hkv):
    """Forked samples' decode rows against the oracle with the plan
    (workspace given), and bit for bit against the same launch without it:
    the plan changes which CTA works a row, not its arithmetic."""
    w = W.forked_decode_mix(FORK_LAYOUT, dt, bs, g * hkv, hkv, hd, seed=bs + hd + g)
    kc, vc, bt = device_caches(w, DEV)
    planned = run_varlen(pa, w, kc, vc, bt, kernel=2, routed=True)
    compare(w, planned, oracle_attention(w))
    unplanned = run_varlen(pa, w, kc, vc, bt, kernel=2, routed=False)
    rows = decode_rows(w)
    assert torch.equal(planned[rows].view(torch.int16), unplanned[rows].view(torch.int16))
    pa.pa_device_status(clear=True)


def test_varlen_forked_decode_rows_many_requests(pa):
    """Over a thousand decode rows in runs of forked samples, with chunks and
    lone rows between runs (more requests than the plan kernel's threads)."""
    rng = np.random.default_rng(7)
    layout = [("chunk", 70, 30)]
    while sum(len(x[2]) if x[0] == "group" else 1 for x in layout) < 1300:
        k = int(rng.integers(1, 8))
        layout.append(("group", int(rng.integers(1, 60)), rng.integers(0, 20, k).tolist()))
        if rng.random() < 0.1:
            layout.append(("single", int(rng.integers(1, 40))))
    w = W.forked_decode_mix(layout, "bf16", 16, 4, 1, 64, seed=11)
    kc, vc, bt = device_caches(w, DEV)
    planned = run_varlen(pa, w, kc, vc, bt, kernel=2, routed=True)
    compare(w, planned, oracle_attention(w))
    unplanned = run_varlen(pa, w, kc, vc, bt, kernel=2, routed=False)
    rows = decode_rows(w)
    assert torch.equal(planned[rows].view(torch.int16), unplanned[rows].view(torch.int16))
    pa.pa_device_status(clear=True)


@pytest.mark.parametrize("bs", [8, 16, 256])
def test_varlen_long_contexts(pa, bs):
    """Contexts past one block-table window of the prefill producers (512
    16-token groups, 8,192 tokens) and of a decode warp (32 tiles): a chunk
    of 32 after 20,000 cached tokens, decode rows over 17,000 and 33,000
    tokens, a short full prefill; with and without the plan, and on the
    CUDA-core kernel."""
    w = W.varlen_workload("long_vl", "bf16", bs, 12, 2, 128, [20032, 17000, 33000, 150], [32, 1, 1, 150],
                          seed=40 + bs)
    kc, vc, bt = device_caches(w, DEV)
    exact = oracle_attention(w)
    for kernel, routed in ((2, False), (2, True), (1, False)):
        compare(w, run_varlen(pa, w, kc, vc, bt, kernel=kernel, routed=routed), exact)
    pa.pa_device_status(clear=True)
