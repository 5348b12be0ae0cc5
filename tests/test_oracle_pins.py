"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle routine to something other than itself: values the
pages print (tests/golden/, each with its source), a library routine
(torch's scaled_dot_product_attention, torch's dtype conversions), closed
forms, invariants, or brute force on tiny inputs.  The sensitivity tests at
the end feed the oracle inputs that reproduce a plausible mistake (wrong GQA
head mapping, causal offset off by one, wrong scale, transposed operands)
and check that the pins notice.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import blocks as B
from paged_kv_cache_116_gb300 import workloads as W

from helpers import golden, nan_cache, oracle_attention, oracle_caches

# ------------------------------------------------------------------ slots


def test_slot_translation_matches_printed_examples():
    for case in golden("slot_translation.json")["cases"]:
        bt = np.array([case["block_table"]], np.int32)
        pos = np.array(case["positions"], np.int64)
        got = oracle.slot_mapping(bt, np.zeros(len(pos), np.int32), pos, case["block_size"])
        assert got.tolist() == case["slots"], case["source"]


def test_slot_mapping_padding_and_multi_sequence():
    bt = np.array([[7, 3, -1], [0, 5, 2]], np.int32)
    seq = np.array([0, 1, 1, 0, 1], np.int32)
    pos = np.array([5, 0, 9, -1, 4], np.int64)
    got = oracle.slot_mapping(bt, seq, pos, 4)
    # brute force: walk the positions block by block
    exp = []
    for s, p in zip(seq, pos):
        if p < 0:
            exp.append(-1)
            continue
        block, off = 0, int(p)
        while off >= 4:
            block, off = block + 1, off - 4
        exp.append(int(bt[s][block]) * 4 + off)
    assert got.tolist() == exp


# ------------------------------------------------------------------ block bookkeeping


def test_block_pool_fifo_doctest():
    g = golden("block_pool.json")["fifo_doctest"]
    pool = B.BlockPool(g["num_blocks"])
    table = pool.allocate(3)
    assert table == g["first_allocate_3"] and pool.num_free() == g["free_after_first"]
    pool.allocate(2)
    pool.free(table)
    assert pool.allocate(4) == g["second_allocate_2_then_free_first_then_allocate_4"]
    assert pool.allocate(10) is None  # short: the page returns None


def test_block_pool_run_py():
    g = golden("block_pool.json")["run_py"]
    pool = B.BlockPool(g["num_blocks"])
    got = pool.allocate(g["allocate"])
    assert got == g["blocks"] and pool.num_free() == g["free_after"]
    pool.free(got)
    assert pool.num_free() == g["free_after_release"]


def test_round_robin_tables():
    g = golden("block_pool.json")["round_robin_tables"]
    assert B.round_robin_tables(g["seq_lens"], g["block_size"], g["num_blocks"]) == g["tables"]
    # the workload generator's own allocator gives the same layout
    w = W.handbook_check()
    for row, t in zip(w.block_tables.tolist(), g["tables"]):
        assert row[: len(t)] == t


def test_append_slot_block_counts():
    g = golden("block_pool.json")["append_slot"]
    for n, b in zip(g["token_counts"], g["blocks"]):
        assert B.blocks_needed(n, g["block_size"]) == b


def test_cow_table():
    g = golden("cow_table.json")
    pool = B.CountingPool(g["block_size"])
    a = B.Sequence(pool, g["block_size"])
    for t in g["a_tokens"]:
        a.append(t)
    snaps = []
    b = a.fork()
    snaps.append((a.blocks[:], b.blocks[:], len(pool.ref), dict(pool.ref)))
    ev = b.append(g["b_appends"])
    assert ev[0] == "cow" and ev[1] == 1 and ev[2] == 2
    assert a.tokens() == g["a_tokens_after"] and b.tokens() == g["b_tokens_after"]
    snaps.append((a.blocks[:], b.blocks[:], len(pool.ref), dict(pool.ref)))
    a.close()
    snaps.append((a.blocks[:], b.blocks[:], len(pool.ref), dict(pool.ref)))
    b.close()
    snaps.append((a.blocks[:], b.blocks[:], len(pool.ref), dict(pool.ref)))
    for (ab, bb, live, refs), step in zip(snaps, g["steps"]):
        assert ab == step["a"] and bb == step["b"] and live == step["live"], step["step"]
        assert {str(k): v for k, v in refs.items()} == step["refs"], step["step"]


def test_cow_boundary_needs_no_copy():
    # Appending exactly at a block boundary opens a new block; the full shared
    # block is never copied.
    pool = B.CountingPool(4)
    a = B.Sequence(pool, 4)
    for t in range(8):
        a.append(t)
    b = a.fork()
    assert b.append(8)[0] == "new"
    assert a.tokens() == list(range(8)) and b.tokens() == list(range(9))


def test_parallel_sampling_counts():
    g = golden("sharing_counts.json")
    for row in g["rows"]:
        unshared, shared = B.parallel_sampling_blocks(g["prompt_len"], g["gen_len"], row["n"], g["block_size"])
        assert (unshared, shared) == (row["unshared"], row["shared"])
        assert round(100.0 * (1 - shared / unshared), 1) == row["saving_pct"]


def test_mixed_workload_cow_pairs_match_oracle_bookkeeping():
    """The mixed step's copy list (from the generator's own pool) is what the
    oracle's Sequence/BlockPool give for the same allocation order."""
    w = W.mixed_varlen()
    n_chunks, groups, gsize, prompt = 16, 60, 4, 300
    pool = B.BlockPool(w.num_blocks)
    pool.free_queue = __import__("collections").deque(
        torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(0)).tolist())
    for i in range(n_chunks):
        assert pool.allocate(B.blocks_needed(int(w.seq_lens[i]), 16)) == \
            w.block_tables[i, : B.blocks_needed(int(w.seq_lens[i]), 16)].tolist()
    pairs, row = [], n_chunks
    for _ in range(groups):
        owner = B.Sequence(pool, 16)
        for _t in range(prompt):
            owner.append()
        samples = [owner] + [owner.fork() for _ in range(gsize - 1)]
        pairs += B.cow_step([samples], 16, pool)
        for s in samples:
            assert w.block_tables[row, : len(s.blocks)].tolist() == s.blocks
            row += 1
    assert [tuple(p) for p in w.cow_pairs.tolist()] == pairs
    assert len(pairs) == groups * (gsize - 1)  # the 18 + 7n reading: the last sample writes in place


# ------------------------------------------------------------------ sizes


def test_utilisation_generator():
    g = golden("sizes.json")["utilisation"]
    lens = W.gqa_batch_lengths(g["num_requests"], 0)
    used = int(lens.sum())
    assert round(100 * used / (g["num_requests"] * g["max_len"]), 1) == g["prealloc_pct"]
    for bs, pct in g["paged_pct"].items():
        alloc = sum(B.blocks_needed(int(L), int(bs)) * int(bs) for L in lens)
        assert round(100 * used / alloc, 1) == pct


def test_tail_waste_and_kv_bytes():
    g = golden("sizes.json")["tail_waste"]
    nb = B.blocks_needed(g["tokens"], g["block_size"])
    assert nb == g["blocks"] and nb * g["block_size"] == g["slots"]
    assert nb * g["block_size"] - g["tokens"] == g["tail_slots"]
    assert g["tokens"] * g["kib_per_token"] / 1024 == g["logical_mib"]
    assert g["slots"] * g["kib_per_token"] / 1024 == g["allocated_mib"]
    assert g["tail_slots"] * g["kib_per_token"] / 1024 == g["tail_mib"]
    k = golden("sizes.json")["kv_bytes"]
    # bytes per token per layer and head read by a decode = 2 (K,V) * head_dim * elt
    per_token = 2 * k["layers"] * 8 * k["head_dim"] * k["elt"]
    assert per_token == k["per_token_bytes_gqa8"]
    for hkv, mib in k["mib"].items():
        assert 2 * k["layers"] * int(hkv) * k["head_dim"] * k["tokens"] * k["elt"] // 2 ** 20 == mib


# ------------------------------------------------------------------ element decoding


def test_decode_all_f16_and_bf16_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint16)
    for name, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        ours = oracle.decode(bits, name)
        ref = torch.from_numpy(bits.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(ours), nan)
        assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------------------ write / copy / gather


def test_write_places_rows_at_printed_slots():
    # the [7, 3] example: tokens 0..5 land in rows 28..31, 12, 13; the rest stay NaN
    cache_k = np.full((8, 4, 1, 2), np.nan, np.float32)
    cache_v = np.full((8, 4, 1, 2), np.nan, np.float32)
    k = np.arange(12, dtype=np.float32).reshape(6, 1, 2)
    v = -k
    slots = oracle.slot_mapping(np.array([[7, 3]], np.int32), np.zeros(6, np.int32), np.arange(6), 4)
    oracle.write_kv(k, v, slots, cache_k, cache_v)
    flat_k = cache_k.reshape(32, 1, 2)
    for i, s in enumerate([28, 29, 30, 31, 12, 13]):
        assert np.array_equal(flat_k[s], k[i]) and np.array_equal(cache_v.reshape(32, 1, 2)[s], v[i])
    untouched = np.setdiff1d(np.arange(32), [28, 29, 30, 31, 12, 13])
    assert np.all(np.isnan(flat_k[untouched]))


def test_write_then_gather_round_trip_and_skip_negative():
    w = W.tiny_decode()
    kc, vc = oracle_caches(w)
    all_k = np.concatenate([W.raw_numpy(w.pre_k), W.raw_numpy(w.new_k)])
    seq = np.concatenate([w.pre_seq_idx, w.new_seq_idx])
    pos = np.concatenate([w.pre_pos, w.new_pos])
    for s, L in enumerate(w.seq_lens):
        got = oracle.gather(kc, w.block_tables[s], int(L), "f32")
        rows = all_k[seq == s][np.argsort(pos[seq == s])]
        assert np.array_equal(got, rows.astype(np.float64))
    before = kc.copy()
    oracle.write_kv(np.ones((1, 2, 32), np.float32), np.ones((1, 2, 32), np.float32), np.array([-1]), kc, vc)
    assert np.array_equal(np.isnan(before), np.isnan(kc)) and np.array_equal(before[~np.isnan(before)],
                                                                              kc[~np.isnan(kc)])


def test_copy_blocks_whole_blocks_every_layer():
    rng = np.random.default_rng(1)
    layers = 3
    ks = [rng.integers(0, 65535, (10, 4, 2, 8), dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 65535, (10, 4, 2, 8), dtype=np.uint16) for _ in range(layers)]
    k0, v0 = [k.copy() for k in ks], [v.copy() for v in vs]
    pairs = np.array([[1, 7], [4, 2], [9, 0]], np.int64)
    oracle.copy_blocks(ks, vs, pairs)
    for l in range(layers):
        for src, dst in pairs:
            assert np.array_equal(ks[l][dst], k0[l][src]) and np.array_equal(vs[l][dst], v0[l][src])
        untouched = [b for b in range(10) if b not in pairs[:, 1]]
        assert np.array_equal(ks[l][untouched], k0[l][untouched])
        assert np.array_equal(vs[l][untouched], v0[l][untouched])


def test_cow_copy_then_write_keeps_sharer_intact():
    """The cache-level version of the fork/append table: B's append copies
    the shared tail and writes into the copy, A still reads 0..5."""
    bs, pool = 4, B.CountingPool(4)
    kc = np.full((4, bs, 1, 2), np.nan, np.float32)
    vc = kc.copy()
    tok = np.arange(14, dtype=np.float32).reshape(7, 1, 2)
    a = B.Sequence(pool, bs)
    for t in range(6):
        a.append(t)
    bt_a = np.array([a.blocks], np.int32)
    oracle.write_kv(tok[:6], tok[:6], oracle.slot_mapping(bt_a, np.zeros(6, np.int32), np.arange(6), bs), kc, vc)
    b = a.fork()
    ev = b.append(6)
    oracle.copy_blocks([kc], [vc], np.array([[ev[1], ev[2]]]))
    bt_b = np.array([b.blocks], np.int32)
    oracle.write_kv(tok[6:], tok[6:], oracle.slot_mapping(bt_b, np.zeros(1, np.int32), np.array([6]), bs), kc, vc)
    assert np.array_equal(oracle.gather(kc, a.blocks, 6, "f32"), tok[:6].astype(np.float64))
    assert np.array_equal(oracle.gather(kc, b.blocks, 7, "f32"), tok.astype(np.float64))


# ------------------------------------------------------------------ attention


def _sdpa_reference(w, kc, vc, causal=True, scale=None):
    """torch's scaled_dot_product_attention over each request's contiguous
    K/V in float64 (GQA through the library's own enable_gqa)."""
    out = []
    qsl = w.query_start_loc
    q_all = torch.from_numpy(oracle.decode(W.raw_numpy(w.q), w.dtype))
    for i, (L, n) in enumerate(zip(w.seq_lens, w.query_lens)):
        k = torch.from_numpy(oracle.gather(kc, w.block_tables[i], int(L), w.dtype))
        v = torch.from_numpy(oracle.gather(vc, w.block_tables[i], int(L), w.dtype))
        q = q_all[qsl[i]: qsl[i + 1]]
        mask = torch.ones(int(n), int(L), dtype=torch.bool).tril(diagonal=int(L - n)) if causal else None
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                           attn_mask=mask, scale=scale, enable_gqa=True)
        out.append(o.transpose(0, 1))
    return torch.cat(out).numpy()


def test_attention_matches_sdpa_on_handbook_layout():
    g = golden("attention_check.json")
    w = W.handbook_check()
    assert w.seq_lens.tolist() == g["seq_lens"] and w.query_lens.tolist() == g["query_lens"]
    kc, vc = oracle_caches(w)
    ours = oracle_attention(w, kc, vc)
    ref = _sdpa_reference(w, kc, vc)  # default scale = head_dim ** -0.5, as the page passes
    qsl = w.query_start_loc
    for i in range(3):
        err = np.abs(ours[qsl[i]: qsl[i + 1]] - ref[qsl[i]: qsl[i + 1]]).max()
        assert err < g["bound"]
        assert err < 1e-12  # both sides in float64


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_attention_matches_sdpa_random_shapes(dtype):
    rng = np.random.default_rng(7)
    for trial in range(6):
        bs = int(rng.choice([1, 4, 16]))
        hkv = int(rng.choice([1, 2]))
        g = int(rng.choice([1, 3, 4]))
        hd = int(rng.choice([8, 32]))
        S = int(rng.integers(1, 5))
        lens = rng.integers(1, 3 * bs + 3, S)
        qlens = np.minimum(lens, rng.integers(1, 6, S))
        w = W.varlen_workload("rand", dtype, bs, hkv * g, hkv, hd, lens, qlens, seed=trial)
        kc, vc = oracle_caches(w)
        for causal in (True, False):
            ours = oracle_attention(w, kc, vc, causal=causal)
            # the library's scale argument is a float: give SDPA the same value
            ref = _sdpa_reference(w, kc, vc, causal=causal, scale=float(np.float32(w.scale)))
            assert np.abs(ours - ref).max() < 1e-12


def test_decode_single_token_returns_v():
    w = W.tiny_decode()
    kc, vc = oracle_caches(w)
    out = oracle_attention(w, kc, vc)
    s = int(np.where(w.seq_lens == 1)[0][0])
    v = oracle.gather(vc, w.block_tables[s], 1, "f32")[0]  # [Hkv, hd]
    rep = w.num_heads // w.num_kv_heads
    for h in range(w.num_heads):
        assert np.array_equal(out[s, h], v[h // rep])


def test_equal_keys_give_mean_of_values():
    w = W.decode_workload("eq", "f32", 4, 4, 2, 16, [9, 1, 16], num_blocks=12, seed=3)
    k_const = np.ones_like(W.raw_numpy(w.pre_k)) * 0.25
    w.pre_k = torch.from_numpy(k_const)
    w.new_k = torch.from_numpy(np.ones_like(W.raw_numpy(w.new_k)) * 0.25)
    kc, vc = oracle_caches(w)
    out = oracle_attention(w, kc, vc)
    rep = w.num_heads // w.num_kv_heads
    for s, L in enumerate(w.seq_lens):
        v = oracle.gather(vc, w.block_tables[s], int(L), "f32")
        for h in range(w.num_heads):
            assert np.allclose(out[s, h], v[:, h // rep].mean(axis=0), rtol=0, atol=1e-14)


def test_full_prefill_first_row_is_first_value():
    w = W.varlen_workload("pf", "f32", 4, 4, 2, 16, [7], [7], seed=5)
    kc, vc = oracle_caches(w)
    out = oracle_attention(w, kc, vc)
    v0 = oracle.gather(vc, w.block_tables[0], 1, "f32")[0]
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // 2])


def test_permuting_physical_blocks_leaves_output_unchanged():
    w = W.varlen_workload("perm", "bf16", 4, 6, 2, 32, [13, 4, 9], [1, 4, 3], seed=11)
    kc, vc = oracle_caches(w)
    base = oracle_attention(w, kc, vc)
    perm = np.random.default_rng(2).permutation(w.num_blocks)  # old id b -> new id perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    w.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    assert np.array_equal(oracle_attention(w, kc2, vc2), base)


def test_unselected_sequences_are_untouched():
    w = W.tiny_decode()
    kc, vc = oracle_caches(w)
    full = oracle_attention(w, kc, vc)
    part = oracle_attention(w, kc, vc, seq_select=np.array([0, 1, 0, 1], np.uint8))
    assert np.array_equal(part[[1, 3]], full[[1, 3]]) and np.all(np.isnan(part[[0, 2]]))


# ------------------------------------------------------------------ the pins notice plausible mistakes


def test_pins_detect_wrong_gqa_mapping():
    w = W.handbook_check()
    kc, vc = oracle_caches(w)
    ref = _sdpa_reference(w, kc, vc)
    # h % Hkv instead of h // (Hq/Hkv): same as permuting the query heads
    hq, hkv = w.num_heads, w.num_kv_heads
    rep = hq // hkv
    wrong = [(h % hkv) * rep + h // hkv for h in range(hq)]
    q = W.raw_numpy(w.q)[:, wrong]
    out = oracle.paged_attention(q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.scale, "f32")
    out_back = np.empty_like(out)
    out_back[:, wrong] = out
    assert np.abs(out_back - ref).max() > 1e-3


def test_pins_detect_causal_offset_and_scale_mistakes():
    w = W.handbook_check()
    kc, vc = oracle_caches(w)
    ref = _sdpa_reference(w, kc, vc)
    # one more visible key per new row: the same as seq_lens + 1 with an extra
    # (NaN-free) key -- emulate with a non-causal pass on the prefill rows
    nc = oracle_attention(w, kc, vc, causal=False)
    assert np.abs(nc - ref)[1:].max() > 1e-3
    bad_scale = oracle.paged_attention(W.raw_numpy(w.q), kc, vc, w.block_tables, w.seq_lens,
                                       w.query_start_loc, 1.0, "f32")
    assert np.abs(bad_scale - ref).max() > 1e-3


def test_pins_detect_swapped_k_and_v():
    w = W.handbook_check()
    kc, vc = oracle_caches(w)
    ref = _sdpa_reference(w, kc, vc)
    swapped = oracle.paged_attention(W.raw_numpy(w.q), vc, kc, w.block_tables, w.seq_lens,
                                     w.query_start_loc, w.scale, "f32")
    assert np.abs(swapped - ref).max() > 1e-3


def test_swap_out_and_back_is_identity_and_moves_whole_blocks():
    rng = np.random.default_rng(9)
    dev_k = [rng.integers(0, 65535, (12, 4, 2, 8), dtype=np.uint16) for _ in range(2)]
    dev_v = [rng.integers(0, 65535, (12, 4, 2, 8), dtype=np.uint16) for _ in range(2)]
    host_k = [np.zeros((6, 4, 2, 8), np.uint16) for _ in range(2)]
    host_v = [np.zeros((6, 4, 2, 8), np.uint16) for _ in range(2)]
    k0, v0 = [k.copy() for k in dev_k], [v.copy() for v in dev_v]
    out_pairs = np.array([[3, 0], [11, 5], [7, 2]], np.int64)  # device block -> host slot
    oracle.swap_blocks(dev_k, dev_v, host_k, host_v, out_pairs)
    for l in range(2):
        for d, h in out_pairs:
            assert np.array_equal(host_k[l][h], k0[l][d]) and np.array_equal(host_v[l][h], v0[l][d])
        assert np.all(host_k[l][[1, 3, 4]] == 0)
    # the blocks are freed on the device and come back into other physical blocks
    for l in range(2):
        dev_k[l][[3, 11, 7]] = 0
        dev_v[l][[3, 11, 7]] = 0
    in_pairs = np.array([[0, 9], [5, 1], [2, 4]], np.int64)  # host slot -> new device block
    oracle.swap_blocks(host_k, host_v, dev_k, dev_v, in_pairs)
    for l in range(2):
        for (d_old, h), (_, d_new) in zip(out_pairs, in_pairs):
            assert np.array_equal(dev_k[l][d_new], k0[l][d_old]) and np.array_equal(dev_v[l][d_new], v0[l][d_old])


# ---- quantized cache (FP8 E4M3 codes, one scale per token and KV head,
#      scales laid out [num_blocks, num_kv_heads, block_size]) ----

def _torch_fp8():
    import torch

    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn")
    return torch


def test_e4m3_values_of_all_256_codes_match_torch():
    """The code table against torch's own float8_e4m3fn decoding (a library
    routine): every finite value and the two NaN codes."""
    torch = _torch_fp8()
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.isnan(ours).sum() == 2 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range_and_ties_go_to_even():
    """Rounding against torch's conversion (round to nearest even) on random
    values and on every midpoint between neighbouring codes; out of range
    (where torch gives NaN) the format's largest finite value is kept."""
    torch = _torch_fp8()
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))  # 0 .. 448 increasing
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(8)
    rand = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32)
    x = np.concatenate([mids, -mids, rand[np.abs(rand) <= 448], grid.astype(np.float32)])
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # ties: the even mantissa wins (1.0625 -> 1.0, 1.1875 -> 1.25, 232 -> 224)
    assert oracle.e4m3_decode(oracle.e4m3_encode(np.array([1.0625, 1.1875, 232.0], np.float32))).tolist() == \
        [1.0, 1.25, 224.0]
    big = oracle.e4m3_encode(np.array([449.0, 464.0, 1e6, -3e38, np.inf], np.float32))
    assert big.tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_quant_rows_scale_max_code_and_error_bound():
    """scale = max|x| / 448 (fp32), the largest element encodes to +-448, and
    every element comes back within half a code step: 2^-4 relative for
    normal codes, 2^-10 x scale below them; an all-zero row keeps scale 1."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * np.exp2(rng.integers(-8, 8, (64, 1)))).astype(np.float32)
    x[5] = 0.0
    codes, scales = oracle.quant_rows(x, "f32")
    amax = np.abs(x).max(axis=1)
    want = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(scales, want)
    dq = oracle.e4m3_decode(codes) * scales[:, None].astype(np.float64)
    big = np.argmax(np.abs(x), axis=1)
    for r in range(64):
        if amax[r] > 0:
            assert abs(oracle.e4m3_decode(codes[r, big[r]])) == 448.0
    err = np.abs(dq - x.astype(np.float64))
    bound = np.exp2(-4) * np.abs(x) + np.exp2(-10) * scales[:, None] + 1e-6 * np.abs(x)
    assert np.all(err <= bound)
    assert np.all(codes[5] == 0) and scales[5] == 1.0


def _grid_pool(rng, nb, bs, hkv, hd):
    """K/V values on the E4M3 grid times a power-of-two row scale, each row
    holding +-448 x scale: quantizing them is lossless."""
    codes = rng.integers(0, 0x7F, (nb, bs, hkv, hd)).astype(np.uint8)
    codes |= (rng.integers(0, 2, codes.shape).astype(np.uint8) << 7)
    codes[..., 0] = np.where(rng.integers(0, 2, codes.shape[:-1]) == 1, 0x7E, 0xFE)
    scales = np.exp2(rng.integers(-9, -2, (nb, hkv, bs))).astype(np.float32)  # [NB, Hkv, bs]
    vals = (oracle.e4m3_decode(codes) * scales.transpose(0, 2, 1)[..., None]).astype(np.float32)
    return codes, scales, vals


def test_fp8_write_and_attention_are_lossless_on_grid_values():
    """On values a quantized cache holds exactly, the quantizing write
    reproduces the codes and scales, and attention over the codes equals the
    pinned attention over the same values stored as fp32, bit for bit; a
    swapped K/V scale changes the result."""
    rng = np.random.default_rng(5)
    nb, bs, hkv, hd, hq = 12, 4, 2, 16, 6
    kcodes, kscales, kvals = _grid_pool(rng, nb, bs, hkv, hd)
    vcodes, vscales, vvals = _grid_pool(rng, nb, bs, hkv, hd)
    # the write: tokens in slot order
    slots = np.arange(nb * bs, dtype=np.int64)
    wk = np.zeros_like(kcodes)
    wv = np.zeros_like(vcodes)
    wks = np.zeros_like(kscales)
    wvs = np.zeros_like(vscales)
    oracle.write_kv_fp8(kvals.reshape(-1, hkv, hd), vvals.reshape(-1, hkv, hd), "f32", slots, wk, wv, wks, wvs)
    assert np.array_equal(wk, kcodes) and np.array_equal(wv, vcodes)
    assert np.array_equal(wks, kscales) and np.array_equal(wvs, vscales)
    lens = np.array([7, 1, 20], np.int32)
    qlens = np.array([3, 1, 20], np.int32)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((3, 6), -1, np.int32)
    tables[0, :2], tables[1, :1], tables[2, :5] = perm[:2], perm[2:3], perm[3:8]
    q = rng.standard_normal((int(qlens.sum()), hq, hd)).astype(np.float32)
    for causal in (True, False):
        got = oracle.paged_attention_fp8(q, "f32", kcodes, vcodes, kscales, vscales, tables, lens, qsl, 0.25,
                                         causal=causal)
        exact = oracle.paged_attention(q, kvals, vvals, tables, lens, qsl, 0.25, "f32", causal=causal)
        assert np.array_equal(got, exact)
        wrong = oracle.paged_attention_fp8(q, "f32", kcodes, vcodes, vscales, kscales, tables, lens, qsl, 0.25,
                                           causal=causal)
        assert not np.allclose(wrong, exact)
