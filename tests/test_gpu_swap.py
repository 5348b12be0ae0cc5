"""GPU parity of the block swap between the device pool and a pinned host
pool (preemption: blocks go out to CPU memory and come back, the xxqk.cn
PagedAttention article, §显存不够时的调度).  Bit-exact against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_116_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def _same(a, b):
    """Bit equality (random fp32 bit patterns include NaNs)."""
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


def _random_pools(layers, nb, bs, hkv, hd, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.float32:
        mk = lambda: torch.randint(-2 ** 31, 2 ** 31 - 1, (nb, bs, hkv, hd), generator=g,  # noqa: E731
                                   dtype=torch.int32).view(torch.float32)
    else:
        mk = lambda: torch.randint(-32768, 32767, (nb, bs, hkv, hd), generator=g,  # noqa: E731
                                   dtype=torch.int16).view(dtype)
    return [mk() for _ in range(layers)], [mk() for _ in range(layers)]


@pytest.mark.parametrize("dtype,bs,hkv,hd", [(torch.bfloat16, 16, 8, 128), (torch.float32, 1, 1, 4),
                                             (torch.float16, 8, 2, 64)])
def test_swap_out_and_in_bit_exact(pa, dtype, bs, hkv, hd):
    layers, nb_dev, nb_host = 3, 37, 29
    dk, dv = _random_pools(layers, nb_dev, bs, hkv, hd, dtype, seed=1)
    hk, hv = _random_pools(layers, nb_host, bs, hkv, hd, dtype, seed=2)
    out_pairs = np.array([[3, 0], [36, 28], [0, 5], [17, 6], [18, 7], [9, 13]], np.int64)
    # oracle on host copies
    odk = [W.raw_numpy(t).copy() for t in dk]
    odv = [W.raw_numpy(t).copy() for t in dv]
    ohk = [W.raw_numpy(t).copy() for t in hk]
    ohv = [W.raw_numpy(t).copy() for t in hv]
    oracle.swap_blocks(odk, odv, ohk, ohv, out_pairs)
    # device pool on the GPU, host pool pinned; pairs on the device
    gdk = [t.to(DEV) for t in dk]
    gdv = [t.to(DEV) for t in dv]
    ghk = [t.pin_memory() for t in hk]
    ghv = [t.pin_memory() for t in hv]
    pa.pa_swap_blocks(gdk, gdv, ghk, ghv, torch.from_numpy(out_pairs).to(DEV))
    torch.cuda.synchronize()
    for l in range(layers):
        assert _same(W.raw_numpy(ghk[l]), ohk[l])
        assert _same(W.raw_numpy(ghv[l]), ohv[l])
        assert _same(W.raw_numpy(gdk[l]), odk[l])  # the source is left as it was
    # back in, to other device blocks; pairs in pinned host memory this time
    in_pairs = np.array([[0, 20], [28, 1], [5, 2], [6, 30], [7, 31], [13, 4]], np.int64)
    oracle.swap_blocks(ohk, ohv, odk, odv, in_pairs)
    pa.pa_swap_blocks(ghk, ghv, gdk, gdv, torch.from_numpy(in_pairs).pin_memory())
    torch.cuda.synchronize()
    for l in range(layers):
        assert _same(W.raw_numpy(gdk[l]), odk[l])
        assert _same(W.raw_numpy(gdv[l]), odv[l])
    # out and back: device block 3 now lives again in block 20, 36 in 1, ...
    for (s, h), (h2, d) in zip(out_pairs, in_pairs):
        assert h == h2
        for l in range(layers):
            assert _same(W.raw_numpy(gdk[l][d]), W.raw_numpy(dk[l][s]))
            assert _same(W.raw_numpy(gdv[l][d]), W.raw_numpy(dv[l][s]))


def test_swap_device_to_device_and_empty(pa):
    dk, dv = _random_pools(2, 10, 16, 2, 64, torch.bfloat16, seed=3)
    ek, ev = _random_pools(2, 12, 16, 2, 64, torch.bfloat16, seed=4)
    a = ([t.to(DEV) for t in dk], [t.to(DEV) for t in dv])
    b = ([t.to(DEV) for t in ek], [t.to(DEV) for t in ev])
    before = [W.raw_numpy(t).copy() for t in b[0]]
    pa.pa_swap_blocks(a[0], a[1], b[0], b[1], torch.empty((0, 2), dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    assert all(_same(W.raw_numpy(t), x) for t, x in zip(b[0], before))
    pairs = np.array([[9, 11], [0, 0]], np.int64)
    ok = [W.raw_numpy(t).copy() for t in ek]
    ov = [W.raw_numpy(t).copy() for t in ev]
    oracle.swap_blocks([W.raw_numpy(t).copy() for t in dk], [W.raw_numpy(t).copy() for t in dv], ok, ov, pairs)
    pa.pa_swap_blocks(a[0], a[1], b[0], b[1], torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    for l in range(2):
        assert _same(W.raw_numpy(b[0][l]), ok[l])
        assert _same(W.raw_numpy(b[1][l]), ov[l])


def test_swap_rejects_pageable_host_memory(pa):
    dk = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
    hk = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16)  # pageable, not pinned
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device=DEV)
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(dk, dk.clone(), hk, hk.clone(), pairs)
    # through the C ABI itself: an unregistered host pool is refused before any launch
    arr = lambda t: (ctypes.c_void_p * 1)(t.data_ptr())  # noqa: E731
    hv = hk.clone()
    st = pa.lib().pa_swap_blocks(arr(dk), arr(dk), arr(hk), arr(hv), 1, ctypes.c_void_p(pairs.data_ptr()), 1, 4, 4,
                                 16, 1, 64, pa.PA_BF16, None)
    assert st != 0
    assert np.count_nonzero(W.raw_numpy(hk).view(np.uint16)) == 0


def test_swap_check_mode_rejects_bad_pairs(pa):
    dk = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
    hk = torch.zeros((6, 16, 1, 64), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pa.pa_set_check_mode(True)
    try:
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_swap_blocks(dk, dk, hk, hv, torch.tensor([[4, 0]], device=DEV))  # source beyond its pool
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_swap_blocks(dk, dk, hk, hv, torch.tensor([[0, 6]], device=DEV))  # destination beyond
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_swap_blocks(dk, dk, hk, hv, torch.tensor([[0, 5], [1, 5]], device=DEV))  # repeated destination
        pa.pa_swap_blocks(dk, dk, hk, hv, torch.tensor([[3, 5], [1, 0]], device=DEV))  # valid
        torch.cuda.synchronize()
    finally:
        pa.pa_set_check_mode(False)
