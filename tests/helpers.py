"""Shared test helpers: oracle-side caches built from a workload, and the
attention tolerance.  Test infrastructure; the product never imports this."""
import json
import os

import numpy as np

import oracle
from paged_kv_cache_116_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}

# Attention tolerance: |gpu - exact| <= ATOL + RTOL * |exact|.  ATOL is the
# stated max-abs bound (1e-5 for fp32, 1e-2 for 16-bit types with fp32
# accumulation); RTOL is the unit roundoff of the output type, the error
# that storing the exact value in that type may add by itself.
ATOL = {"f32": 1e-5, "bf16": 1e-2, "f16": 1e-2}
RTOL = {"f32": 2.0 ** -24, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def nan_cache(w):
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    if w.dtype == "f32":
        return np.full(shape, np.nan, dtype=np.float32)
    return np.full(shape, NAN_BITS[w.dtype], dtype=np.uint16)


def oracle_caches(w, after_step=True):
    """Oracle K/V caches of a workload: NaN everywhere, the cached rows
    written through the pre-step tables, then (after_step) the step's block
    copies and new rows."""
    kc, vc = nan_cache(w), nan_cache(w)
    slots = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, w.block_size)
    oracle.write_kv(W.raw_numpy(w.pre_k), W.raw_numpy(w.pre_v), slots, kc, vc)
    if after_step:
        if w.cow_pairs.shape[0]:
            oracle.copy_blocks([kc], [vc], w.cow_pairs)
        slots = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, w.block_size)
        oracle.write_kv(W.raw_numpy(w.new_k), W.raw_numpy(w.new_v), slots, kc, vc)
    return kc, vc


def oracle_attention(w, kc=None, vc=None, seq_select=None, causal=None):
    if kc is None:
        kc, vc = oracle_caches(w)
    return oracle.paged_attention(W.raw_numpy(w.q), kc, vc, w.block_tables, w.seq_lens, w.query_start_loc,
                                  w.scale, w.dtype, w.causal if causal is None else causal,
                                  seq_select=seq_select)


def within_tol(got, exact, dtype):
    err = np.abs(got - exact)
    bound = ATOL[dtype] + RTOL[dtype] * np.abs(exact)
    return bool(np.all(err <= bound)), float(np.nanmax(err)) if err.size else 0.0


def device_caches(w, dev, after_step=True):
    """Device K/V caches of a workload built through the library itself:
    NaN everywhere, cached rows via pa_slot_mapping + pa_write_kv on the
    pre-step tables, then (after_step) pa_copy_blocks and the step's rows."""
    import torch
    import paged_kv_cache_116_gb300 as pa

    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=W.TORCH_DTYPES[w.dtype], device=dev)
    vc = torch.full_like(kc, float("nan"))
    if w.pre_pos.shape[0]:
        slots = pa.pa_slot_mapping(torch.from_numpy(w.pre_block_tables).to(dev),
                                   torch.from_numpy(w.pre_seq_idx).to(dev), torch.from_numpy(w.pre_pos).to(dev),
                                   w.block_size)
        pa.pa_write_kv(w.pre_k.to(dev), w.pre_v.to(dev), slots, kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    if after_step:
        if w.cow_pairs.shape[0]:
            pa.pa_copy_blocks(kc, vc, torch.from_numpy(w.cow_pairs).to(dev))
        slots = pa.pa_slot_mapping(bt, torch.from_numpy(w.new_seq_idx).to(dev), torch.from_numpy(w.new_pos).to(dev),
                                   w.block_size)
        pa.pa_write_kv(w.new_k.to(dev), w.new_v.to(dev), slots, kc, vc)
    return kc, vc, bt


def raw_bits(t):
    """Bit patterns of a cache (host numpy, uint32 for fp32 else uint16)."""
    a = W.raw_numpy(t)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def oracle_bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


# ---- quantized (FP8 E4M3) cache -------------------------------------------

FP8_NAN_CODE = 0x7F


def oracle_fp8_caches(w):
    """Oracle code pools [NB, bs, Hkv, hd] (NaN code everywhere) and scale
    pools [NB, Hkv, bs] (NaN everywhere) after the quantizing write of the
    workload's cached rows, the step's block copies, and its new rows."""
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    sshape = (w.num_blocks, w.num_kv_heads, w.block_size)
    kc = np.full(shape, FP8_NAN_CODE, np.uint8)
    vc = kc.copy()
    ks = np.full(sshape, np.nan, np.float32)
    vs = ks.copy()
    slots = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, w.block_size)
    oracle.write_kv_fp8(W.raw_numpy(w.pre_k), W.raw_numpy(w.pre_v), w.dtype, slots, kc, vc, ks, vs)
    if w.cow_pairs.shape[0]:
        oracle.copy_blocks([kc], [vc], w.cow_pairs)
        oracle.copy_blocks([ks], [vs], w.cow_pairs)
    slots = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, w.block_size)
    oracle.write_kv_fp8(W.raw_numpy(w.new_k), W.raw_numpy(w.new_v), w.dtype, slots, kc, vc, ks, vs)
    return kc, vc, ks, vs


def device_fp8_caches(w, dev, after_step=True):
    """The same pools built on the device through pa_slot_mapping and
    pa_write_kv_fp8 (without the step's new rows unless after_step)."""
    import torch
    import paged_kv_cache_116_gb300 as pa

    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    sshape = (w.num_blocks, w.num_kv_heads, w.block_size)
    kc = torch.full(shape, FP8_NAN_CODE, dtype=torch.uint8, device=dev)
    vc = torch.full_like(kc, FP8_NAN_CODE)
    ks = torch.full(sshape, float("nan"), dtype=torch.float32, device=dev)
    vs = torch.full_like(ks, float("nan"))
    bt = torch.from_numpy(w.block_tables).to(dev)
    if w.pre_pos.shape[0]:
        slots = pa.pa_slot_mapping(torch.from_numpy(w.pre_block_tables).to(dev),
                                   torch.from_numpy(w.pre_seq_idx).to(dev), torch.from_numpy(w.pre_pos).to(dev),
                                   w.block_size)
        pa.pa_write_kv_fp8(w.pre_k.to(dev), w.pre_v.to(dev), slots, kc, vc, ks, vs)
    if after_step:
        if w.cow_pairs.shape[0]:
            pairs = torch.from_numpy(w.cow_pairs).to(dev)
            pa.pa_copy_blocks(kc, vc, pairs)
            pa.pa_copy_blocks(ks, vs, pairs)
        slots = pa.pa_slot_mapping(bt, torch.from_numpy(w.new_seq_idx).to(dev), torch.from_numpy(w.new_pos).to(dev),
                                   w.block_size)
        pa.pa_write_kv_fp8(w.new_k.to(dev), w.new_v.to(dev), slots, kc, vc, ks, vs)
    return kc, vc, ks, vs, bt


def oracle_fp8_attention(w, kc, vc, ks, vs, seq_select=None):
    out = oracle.paged_attention_fp8(W.raw_numpy(w.q), w.dtype, kc, vc, ks, vs, w.block_tables, w.seq_lens,
                                     w.query_start_loc, w.scale, w.causal)
    if seq_select is not None:
        out = out[np.asarray(seq_select, bool)]
    return out


# ---- CUDA-graph replay -------------------------------------------------

def graph_replays_match_eager(decode_fn, q, dev):
    """decode_fn(out, q, ws) captured once in a CUDA graph and replayed with
    new queries each time must give, bit for bit, what an eager call gives:
    units split across warps have to be merged on every replay, not only on
    the first."""
    import torch

    out = torch.empty_like(q)
    ref = torch.empty_like(q)
    ws_graph = torch.empty(1 << 24, dtype=torch.uint8, device=dev)
    ws_eager = torch.empty(1 << 24, dtype=torch.uint8, device=dev)
    decode_fn(out, q, ws_graph)  # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        decode_fn(out, q, ws_graph)
    gen = torch.Generator(device=dev).manual_seed(77)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, generator=gen, device=dev).to(q.dtype))
        g.replay()
        decode_fn(ref, q, ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
