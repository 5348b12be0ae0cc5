"""GPU parity of the byte-moving kernels: slot translation, K/V write and the
copy-on-write block copy must equal the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_116_gb300 import workloads as W

from helpers import device_caches, golden, oracle_bits, oracle_caches, raw_bits

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    return pa


def test_slot_mapping_printed_examples(pa):
    for case in golden("slot_translation.json")["cases"]:
        bt = torch.tensor([case["block_table"]], dtype=torch.int32, device=DEV)
        pos = torch.tensor(case["positions"], dtype=torch.int64, device=DEV)
        got = pa.pa_slot_mapping(bt, torch.zeros_like(pos, dtype=torch.int32), pos, case["block_size"])
        assert got.cpu().tolist() == case["slots"]


@pytest.mark.parametrize("bs", [1, 4, 16, 32])
def test_slot_mapping_random_matches_oracle(pa, bs):
    rng = np.random.default_rng(bs)
    S, maxb, n = 37, 50, 5000
    bt = rng.integers(0, 100000, (S, maxb)).astype(np.int32)
    seq = rng.integers(0, S, n).astype(np.int32)
    pos = rng.integers(-3, maxb * bs, n).astype(np.int64)
    exp = oracle.slot_mapping(bt, seq, pos, bs)
    got = pa.pa_slot_mapping(torch.from_numpy(bt).to(DEV), torch.from_numpy(seq).to(DEV),
                             torch.from_numpy(pos).to(DEV), bs).cpu().numpy()
    assert np.array_equal(got, exp)


@pytest.mark.parametrize("make", [W.tiny_decode, W.handbook_check,
                                  lambda: W.mixed_varlen(num_chunks=3, num_groups=5),
                                  lambda: W.decode_workload("w", "f16", 16, 40, 40, 128, [5, 40, 17], seed=2)])
def test_write_and_copy_bit_exact(pa, make):
    w = make()
    kc, vc, _ = device_caches(w, DEV)
    okc, ovc = oracle_caches(w)
    # the whole pool, NaN canaries included, bit for bit
    assert np.array_equal(raw_bits(kc), oracle_bits(okc))
    assert np.array_equal(raw_bits(vc), oracle_bits(ovc))


def test_write_skips_negative_slots_and_keeps_canaries(pa):
    hkv, hd = 2, 64
    kc = torch.full((8, 4, hkv, hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    before = raw_bits(kc).copy()
    k = torch.randn(5, hkv, hd, device=DEV).bfloat16()
    v = torch.randn(5, hkv, hd, device=DEV).bfloat16()
    slots = torch.tensor([3, -1, 31, -7, 0], dtype=torch.int64, device=DEV)
    pa.pa_write_kv(k, v, slots, kc, vc)
    flat = kc.view(32, hkv, hd)
    for i, s in enumerate([3, -1, 31, -7, 0]):
        if s >= 0:
            assert torch.equal(flat[s].view(torch.int16), k[i].view(torch.int16))
    after = raw_bits(kc).reshape(32, -1)
    untouched = [r for r in range(32) if r not in (3, 31, 0)]
    assert np.array_equal(after[untouched], before.reshape(32, -1)[untouched])


def test_copy_blocks_multi_layer(pa):
    g = torch.Generator().manual_seed(4)
    layers, nb, bs, hkv, hd = 5, 40, 16, 2, 128
    ks = [torch.randint(-30000, 30000, (nb, bs, hkv, hd), generator=g, dtype=torch.int16).view(torch.bfloat16)
          for _ in range(layers)]
    vs = [torch.randint(-30000, 30000, (nb, bs, hkv, hd), generator=g, dtype=torch.int16).view(torch.bfloat16)
          for _ in range(layers)]
    pairs = np.array([[1, 30], [7, 2], [39, 0], [5, 5], [12, 13]], np.int64)
    oks = [W.raw_numpy(k).copy() for k in ks]
    ovs = [W.raw_numpy(v).copy() for v in vs]
    oracle.copy_blocks(oks, ovs, pairs)
    dks = [k.to(DEV) for k in ks]
    dvs = [v.to(DEV) for v in vs]
    pa.pa_copy_blocks(dks, dvs, torch.from_numpy(pairs).to(DEV))
    for l in range(layers):
        assert np.array_equal(W.raw_numpy(dks[l]), oks[l])
        assert np.array_equal(W.raw_numpy(dvs[l]), ovs[l])


def test_cow_keeps_the_sharer_intact_on_device(pa):
    """The fork/append table on the device: B's append copies the shared
    tail (pa_copy_blocks) and writes into the copy; A's rows stay."""
    from oracle import blocks as B

    bs = 4
    pool = B.CountingPool(bs)
    a = B.Sequence(pool, bs)
    for t in range(6):
        a.append(t)
    b = a.fork()
    ev = b.append(6)
    assert ev[0] == "cow"
    kc = torch.full((4, bs, 1, 16), float("nan"), dtype=torch.float32, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    rows = torch.arange(7 * 16, dtype=torch.float32, device=DEV).view(7, 1, 16)
    bt_a = torch.tensor([a.blocks], dtype=torch.int32, device=DEV)
    s = pa.pa_slot_mapping(bt_a, torch.zeros(6, dtype=torch.int32, device=DEV), torch.arange(6, device=DEV), bs)
    pa.pa_write_kv(rows[:6], rows[:6], s, kc, vc)
    pa.pa_copy_blocks(kc, vc, torch.tensor([[ev[1], ev[2]]], device=DEV))
    bt_b = torch.tensor([b.blocks], dtype=torch.int32, device=DEV)
    s = pa.pa_slot_mapping(bt_b, torch.zeros(1, dtype=torch.int32, device=DEV), torch.tensor([6], device=DEV), bs)
    pa.pa_write_kv(rows[6:], rows[6:], s, kc, vc)
    host = kc.cpu().numpy()
    assert np.array_equal(oracle.gather(host, a.blocks, 6, "f32"), rows[:6].cpu().numpy().astype(np.float64))
    assert np.array_equal(oracle.gather(host, b.blocks, 7, "f32"), rows.cpu().numpy().astype(np.float64))


def test_check_mode_rejects_bad_indices(pa):
    kc = torch.zeros((4, 4, 1, 16), dtype=torch.float32, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.zeros((2, 1, 16), device=DEV)
    pa.pa_set_check_mode(True)
    try:
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_write_kv(k, k, torch.tensor([3, 3], device=DEV), kc, vc)  # duplicate slot
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_write_kv(k, k, torch.tensor([3, 16], device=DEV), kc, vc)  # beyond the pool
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_copy_blocks(kc, vc, torch.tensor([[0, 4]], device=DEV))
        with pytest.raises(pa.PAError, match="PA_ERR_INDEX"):
            pa.pa_copy_blocks(kc, vc, torch.tensor([[0, 1], [1, 2]], device=DEV))
        pa.pa_write_kv(k, k, torch.tensor([3, -1], device=DEV), kc, vc)  # valid
    finally:
        pa.pa_set_check_mode(False)
