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


def run_varlen(pa, w, kc, vc, bt, causal=None, kernel=0):
    pa.pa_set_option(pa.PA_OPT_VARLEN_KERNEL, kernel)
    try:
        out = torch.full(tuple(w.q.shape), float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=DEV)
        pa.pa_varlen(out, w.q.to(DEV), kc, vc, bt, torch.from_numpy(w.seq_lens).to(DEV),
                     torch.from_numpy(w.query_start_loc).to(DEV), int(w.query_lens.max()), int(w.seq_lens.max()),
                     w.scale, causal=w.causal if causal is None else causal)
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
