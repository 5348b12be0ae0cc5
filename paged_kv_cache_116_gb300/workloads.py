"""Seeded synthetic inputs for the paged-KV hot path.

This module holds no arithmetic of the method: it draws lengths and values,
hands out physical block ids, and lists which (sequence, position) rows exist
before a step and which arrive in it.  Turning positions into slots, writing,
copying and attending are left to the library (and, in the tests, to the
oracle), so both sides start from the same inputs and nothing else.

Every workload is a ``Workload``:

- geometry: dtype ("f32" | "bf16" | "f16"), block_size, num_blocks,
  num_heads (Hq), num_kv_heads (Hkv), head_dim, scale, causal;
- per request i: seq_lens[i] (context after the step), query_lens[i] (new
  tokens this step; 1 for decode), block_tables[i] (padded with -1 past the
  blocks it holds; these entries are never read);
- ``pre_*``: the context already cached before the step, as rows with the
  request (row of ``pre_block_tables``) and the position they belong to;
- ``new_*`` / ``q``: the step's new tokens (request, position, K/V row, query),
  ordered by request, so request i's queries are rows
  [query_start_loc[i], query_start_loc[i+1]);
- ``cow_pairs``: the (src, dst) block copies the step makes before writing,
  from a reference-counted FIFO pool (empty for the decode configurations).

Unused cache slots are meant to be filled with NaN by whoever materialises
the cache, so that a kernel reading outside a sequence's context shows up.
"""
from __future__ import annotations

import math
import random
from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
ELT_BYTES = {"f32": 4, "bf16": 2, "f16": 2}
PAD = -1


@dataclass
class Workload:
    name: str
    dtype: str
    block_size: int
    num_blocks: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    causal: bool
    seq_lens: np.ndarray
    query_lens: np.ndarray
    block_tables: np.ndarray
    pre_block_tables: np.ndarray
    pre_seq_idx: np.ndarray
    pre_pos: np.ndarray
    pre_k: torch.Tensor
    pre_v: torch.Tensor
    new_seq_idx: np.ndarray
    new_pos: np.ndarray
    new_k: torch.Tensor
    new_v: torch.Tensor
    q: torch.Tensor
    cow_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    seed: int = 0
    notes: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.query_lens)]).astype(np.int32)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elt(self) -> int:
        return ELT_BYTES[self.dtype]

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.query_lens == 1))

    def kv_bytes_read(self) -> int:
        """Bytes of K and V the step's attention reads: every request's
        context once per KV head (the shared prompt blocks count once per
        reader)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 2 * self.elt


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(g, shape, std: float, dtype: str) -> torch.Tensor:
    """N(0, std^2) values drawn in fp32 on the generator's device, then
    rounded to the element type."""
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=g.device)
    if std != 1.0:
        t.mul_(std)
    return t.to(TORCH_DTYPES[dtype])


def _pad_tables(tables, width=None) -> np.ndarray:
    width = width or max(1, max(len(t) for t in tables))
    out = np.full((len(tables), width), PAD, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, : len(t)] = t
    return out


def _blocks_for(n_tokens: int, bs: int) -> int:
    return -(-n_tokens // bs)


def _shuffled_tables(lens, bs: int, num_blocks: int, seed: int) -> np.ndarray:
    """Consecutive slices of a seeded permutation of the physical ids."""
    perm = torch.randperm(num_blocks, generator=_gen(seed)).numpy()
    tables, at = [], 0
    for L in lens:
        n = _blocks_for(int(L), bs)
        tables.append(perm[at : at + n].tolist())
        at += n
    return _pad_tables(tables)


def _rows_for(lens_before) -> tuple[np.ndarray, np.ndarray]:
    """(request index, position) of every cached row, request by request."""
    seq = np.repeat(np.arange(len(lens_before), dtype=np.int32), np.asarray(lens_before, dtype=np.int64))
    pos = np.concatenate([np.arange(int(n), dtype=np.int64) for n in lens_before]) if len(lens_before) else \
        np.zeros(0, np.int64)
    return seq, pos


def decode_workload(name, dtype, block_size, num_heads, num_kv_heads, head_dim, lens, *, std=1.0,
                    num_blocks=None, slack=0.10, seed=0, scale=None, tables=None, notes="",
                    device="cpu") -> Workload:
    """One new token per sequence at position L-1; positions 0..L-2 cached.
    Values are drawn by torch's seeded generator on `device` (the CPU and
    CUDA generators give different, each reproducible, streams)."""
    lens = np.asarray(lens, dtype=np.int32)
    S = lens.shape[0]
    need = sum(_blocks_for(int(L), block_size) for L in lens)
    if num_blocks is None:
        num_blocks = int(math.ceil(need * (1.0 + slack)))
    if tables is None:
        tables = _shuffled_tables(lens, block_size, num_blocks, seed)
    g = _gen(seed + 1, device)
    q = _normal(g, (S, num_heads, head_dim), std, dtype)
    pre_seq, pre_pos = _rows_for(lens - 1)
    pre_k = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), std, dtype)
    pre_v = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), std, dtype)
    new_k = _normal(g, (S, num_kv_heads, head_dim), std, dtype)
    new_v = _normal(g, (S, num_kv_heads, head_dim), std, dtype)
    return Workload(
        name=name, dtype=dtype, block_size=block_size, num_blocks=num_blocks, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim,
        scale=float(scale if scale is not None else head_dim ** -0.5), causal=True,
        seq_lens=lens, query_lens=np.ones(S, np.int32), block_tables=tables, pre_block_tables=tables,
        pre_seq_idx=pre_seq, pre_pos=pre_pos, pre_k=pre_k, pre_v=pre_v,
        new_seq_idx=np.arange(S, dtype=np.int32), new_pos=(lens - 1).astype(np.int64),
        new_k=new_k, new_v=new_v, q=q, seed=seed, notes=notes)


# ---------------------------------------------------------------- configurations


def tiny_decode(seed: int = 0) -> Workload:
    """fp32, block_size 4, 32 blocks, Hq 4, Hkv 2, head_dim 32, contexts
    [6, 13, 1, 20]; tables are consecutive slices of a seeded permutation of
    the 32 blocks."""
    return decode_workload("tiny_decode_fp32_bs4", "f32", 4, 4, 2, 32, [6, 13, 1, 20], num_blocks=32,
                           seed=seed, scale=32 ** -0.5,
                           notes="contexts [6,13,1,20]; unused slots NaN")


def gqa_batch_lengths(n: int = 64, seed: int = 0) -> np.ndarray:
    """Context lengths prompt + output with prompt ~ randint(100, 2000) and
    output ~ randint(20, 1500), drawn in that order from Python's `random`
    seeded with `seed` (the handbook's utilisation workload)."""
    rnd = random.Random(seed)
    pairs = [(rnd.randint(100, 2000), rnd.randint(20, 1500)) for _ in range(n)]
    return np.array([p + o for p, o in pairs], dtype=np.int32)


def gqa_decode_batch(seed: int = 0, num_seqs: int = 64, device="cpu", block_size: int = 16) -> Workload:
    """bf16, block_size 16 (or another size for the block-size sweep), Hq 32,
    Hkv 8, head_dim 128, 64 sequences, shuffled physical blocks, 10 % slack."""
    name = "gqa_decode_bf16_64seq" + ("" if block_size == 16 else "_bs%d" % block_size)
    return decode_workload(name, "bf16", block_size, 32, 8, 128, gqa_batch_lengths(num_seqs, seed),
                           seed=seed, notes="L = randint(100,2000)+randint(20,1500), random.seed(0)",
                           device=device)


def long_context_decode(seed: int = 0, num_seqs: int = 8, context: int = 32768, device="cpu") -> Workload:
    """bf16, block_size 16, Hq 32, Hkv 8, head_dim 128, 8 sequences of 32768."""
    return decode_workload("long_decode_bf16_8x32k", "bf16", 16, 32, 8, 128, [context] * num_seqs, seed=seed,
                           notes="8 x 32768 tokens", device=device)


def mha_lengths(n: int = 128, seed: int = 0, mean: float = 480.0, sigma: float = 1.0) -> np.ndarray:
    """Lognormal totals with the given mean (mu = ln(mean) - sigma^2/2),
    rounded and clipped to [1, 2048], from numpy's default_rng(seed)."""
    rng = np.random.default_rng(seed)
    mu = math.log(mean) - sigma * sigma / 2
    return np.clip(np.rint(rng.lognormal(mu, sigma, n)), 1, 2048).astype(np.int32)


def mha_decode(seed: int = 0, num_seqs: int = 128, device="cpu") -> Workload:
    """fp16, block_size 16, Hq = Hkv = 40, head_dim 128, 128 sequences,
    values ~ N(0, 0.5^2)."""
    return decode_workload("mha_decode_fp16_128seq", "f16", 16, 40, 40, 128, mha_lengths(num_seqs, seed), std=0.5,
                           seed=seed, notes="lognormal lengths sigma=1 mean 480 clip [1,2048]; std 0.5",
                           device=device)


class _FifoRefPool:
    """Reference-counted FIFO block pool used to lay out the mixed step."""

    def __init__(self, order):
        self.free = deque(int(b) for b in order)
        self.ref = {}

    def take(self) -> int:
        b = self.free.popleft()
        self.ref[b] = 1
        return b


def mixed_varlen(seed: int = 0, num_chunks: int = 16, num_groups: int = 60, group_size: int = 4,
                 prompt_len: int = 300, chunk_range=(64, 1024), cached_range=(0, 1024), device="cpu") -> Workload:
    """bf16, block_size 16, Hq 12, Hkv 2, head_dim 128.

    Requests 0..num_chunks-1 are prefill chunks: n new tokens ~ U[64, 1024]
    after `cached` ~ U[0, 1024] tokens already in their blocks.  Then
    num_groups parallel-sampling groups of group_size samples share one
    prompt of prompt_len tokens (the first sample owns it, the others fork
    it); each sample appends one token at position prompt_len.  A shared
    partial tail is copied to a fresh block before a sample writes it, so in
    each group all samples but the last copy the tail and the last writes in
    place.
    """
    bs, hq, hkv, hd, dtype = 16, 12, 2, 128, "bf16"
    rng = np.random.default_rng(seed)
    n_new = rng.integers(chunk_range[0], chunk_range[1] + 1, num_chunks)
    cached = rng.integers(cached_range[0], cached_range[1] + 1, num_chunks)
    chunk_lens = cached + n_new
    prompt_blocks = _blocks_for(prompt_len, bs)
    need = sum(_blocks_for(int(L), bs) for L in chunk_lens) + num_groups * prompt_blocks
    need += num_groups * group_size * 2  # room for tail copies and new blocks
    num_blocks = int(math.ceil(need * 1.10))
    pool = _FifoRefPool(torch.randperm(num_blocks, generator=_gen(seed)).numpy())

    pre_tables, post_tables = [], []
    for L in chunk_lens:
        t = [pool.take() for _ in range(_blocks_for(int(L), bs))]
        pre_tables.append(t)
        post_tables.append(t)
    pairs = []
    for _ in range(num_groups):
        owner = [pool.take() for _ in range(prompt_blocks)]
        for b in owner:
            pool.ref[b] = group_size  # owner + (group_size - 1) forks
        for _s in range(group_size):
            pre_tables.append(list(owner))
            table = list(owner)
            if prompt_len % bs == 0:
                table.append(pool.take())
            elif pool.ref[table[-1]] > 1:
                old = table[-1]
                table[-1] = pool.take()
                pool.ref[old] -= 1
                pairs.append((old, table[-1]))
            post_tables.append(table)

    S = num_chunks + num_groups * group_size
    seq_lens = np.concatenate([chunk_lens, np.full(num_groups * group_size, prompt_len + 1)]).astype(np.int32)
    query_lens = np.concatenate([n_new, np.ones(num_groups * group_size, np.int64)]).astype(np.int32)
    width = max(len(t) for t in post_tables + pre_tables)
    pre_bt, post_bt = _pad_tables(pre_tables, width), _pad_tables(post_tables, width)

    # rows cached before the step: each chunk's first `cached` tokens, and
    # each group's prompt written once through its owner (first sample)
    pre_seq = [np.full(int(c), i, np.int32) for i, c in enumerate(cached)]
    pre_pos = [np.arange(int(c), dtype=np.int64) for c in cached]
    for gi in range(num_groups):
        owner_row = num_chunks + gi * group_size
        pre_seq.append(np.full(prompt_len, owner_row, np.int32))
        pre_pos.append(np.arange(prompt_len, dtype=np.int64))
    pre_seq, pre_pos = np.concatenate(pre_seq), np.concatenate(pre_pos)
    new_seq = np.repeat(np.arange(S, dtype=np.int32), query_lens.astype(np.int64))
    new_pos = np.concatenate([np.arange(int(seq_lens[i] - query_lens[i]), int(seq_lens[i]), dtype=np.int64)
                              for i in range(S)])
    g = _gen(seed + 1, device)
    N = int(query_lens.sum())
    q = _normal(g, (N, hq, hd), 1.0, dtype)
    pre_k = _normal(g, (pre_pos.shape[0], hkv, hd), 1.0, dtype)
    pre_v = _normal(g, (pre_pos.shape[0], hkv, hd), 1.0, dtype)
    new_k = _normal(g, (N, hkv, hd), 1.0, dtype)
    new_v = _normal(g, (N, hkv, hd), 1.0, dtype)
    return Workload(
        name="mixed_varlen_cow_bf16", dtype=dtype, block_size=bs, num_blocks=num_blocks, num_heads=hq,
        num_kv_heads=hkv, head_dim=hd, scale=hd ** -0.5, causal=True, seq_lens=seq_lens, query_lens=query_lens,
        block_tables=post_bt, pre_block_tables=pre_bt, pre_seq_idx=pre_seq, pre_pos=pre_pos, pre_k=pre_k,
        pre_v=pre_v, new_seq_idx=new_seq, new_pos=new_pos, new_k=new_k, new_v=new_v, q=q,
        cow_pairs=np.array(pairs, dtype=np.int64).reshape(-1, 2), seed=seed,
        notes=f"{num_chunks} chunks n~U{list(chunk_range)} cached~U{list(cached_range)}; "
              f"{num_groups}x{group_size} samples share a {prompt_len}-token prompt")


def forked_decode_mix(layout, dtype="bf16", block_size=16, num_heads=12, num_kv_heads=2, head_dim=128,
                      seed=0, device="cpu") -> Workload:
    """A varlen step whose decode rows include parallel-sampling groups.

    layout: a list of requests in order, each
      ("chunk", n_new, cached)        a prefill chunk after `cached` tokens;
      ("single", L)                   a decode row over L tokens (own blocks);
      ("group", prompt_len, extras)   len(extras) samples forked from one
                                      prompt: they share its full blocks, each
                                      has its own blocks from the prompt's
                                      partial tail on, holding extras[j] more
                                      cached tokens of its own, and appends
                                      one token (L = prompt_len + extras[j] + 1).
    Cached rows are written before the step (the shared prompt rows once,
    through the first sample's table); the new rows by the step.  Physical
    blocks come from a shuffled free list."""
    bs = block_size
    rng = np.random.default_rng(seed)
    lens, qlens, cached_of, tables, pre_rows = [], [], [], [], []
    need = 0
    for item in layout:
        if item[0] == "chunk":
            need += _blocks_for(int(item[1]) + int(item[2]), bs)
        elif item[0] == "single":
            need += _blocks_for(int(item[1]), bs)
        else:
            shared = int(item[1]) // bs
            need += shared + sum(_blocks_for(int(item[1]) + int(e) + 1, bs) - shared for e in item[2])
    num_blocks = max(1, int(math.ceil(need * 1.1)) + 4)
    free = list(rng.permutation(num_blocks))
    for item in layout:
        if item[0] in ("chunk", "single"):
            L = int(item[1]) + int(item[2]) if item[0] == "chunk" else int(item[1])
            n = int(item[1]) if item[0] == "chunk" else 1
            t = [int(free.pop()) for _ in range(_blocks_for(L, bs))]
            lens.append(L)
            qlens.append(n)
            tables.append(t)
            pre_rows.append((len(tables) - 1, 0, L - n))
        else:
            prompt, extras = int(item[1]), [int(e) for e in item[2]]
            shared = [int(free.pop()) for _ in range(prompt // bs)]
            for j, e in enumerate(extras):
                L = prompt + e + 1
                t = shared + [int(free.pop()) for _ in range(_blocks_for(L, bs) - len(shared))]
                lens.append(L)
                qlens.append(1)
                tables.append(t)
                # the shared rows once (first sample), every sample's own rows
                pre_rows.append((len(tables) - 1, 0 if j == 0 else len(shared) * bs, L - 1))
    S = len(lens)
    seq_lens, query_lens = np.asarray(lens, np.int32), np.asarray(qlens, np.int32)
    bt = _pad_tables(tables)
    pre_seq = np.concatenate([np.full(b - a, i, np.int32) for i, a, b in pre_rows])
    pre_pos = np.concatenate([np.arange(a, b, dtype=np.int64) for i, a, b in pre_rows])
    new_seq = np.repeat(np.arange(S, dtype=np.int32), query_lens.astype(np.int64))
    new_pos = np.concatenate([np.arange(int(seq_lens[i] - query_lens[i]), int(seq_lens[i]), dtype=np.int64)
                              for i in range(S)])
    g = _gen(seed + 1, device)
    N = int(query_lens.sum())
    q = _normal(g, (N, num_heads, head_dim), 1.0, dtype)
    pre_k = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), 1.0, dtype)
    pre_v = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), 1.0, dtype)
    new_k = _normal(g, (N, num_kv_heads, head_dim), 1.0, dtype)
    new_v = _normal(g, (N, num_kv_heads, head_dim), 1.0, dtype)
    return Workload(
        name="forked_decode_mix", dtype=dtype, block_size=bs, num_blocks=num_blocks, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, scale=head_dim ** -0.5, causal=True, seq_lens=seq_lens,
        query_lens=query_lens, block_tables=bt, pre_block_tables=bt, pre_seq_idx=pre_seq, pre_pos=pre_pos,
        pre_k=pre_k, pre_v=pre_v, new_seq_idx=new_seq, new_pos=new_pos, new_k=new_k, new_v=new_v, q=q, seed=seed,
        notes="layout %r" % (layout,))


def handbook_check(seed: int = 0, dtype: str = "f32") -> Workload:
    """The handbook's verification layout: contexts [37, 5, 20] with [1, 5, 8]
    new tokens (a decode, a full prefill, the second half of a chunked
    prefill), Hq 8, Hkv 2, head_dim 64, block_size 4, 32 blocks handed out
    one per request in turn."""
    seq_lens = np.array([37, 5, 20], np.int32)
    qlens = np.array([1, 5, 8], np.int32)
    return varlen_workload("handbook_check", dtype, 4, 8, 2, 64, seq_lens, qlens, num_blocks=32,
                           tables=_pad_tables(_round_robin(seq_lens, 4, 32)), seed=seed)


def _round_robin(seq_lens, bs, num_blocks):
    free = deque(range(num_blocks))
    tables = [[] for _ in seq_lens]
    while any(len(t) * bs < s for t, s in zip(tables, seq_lens)):
        for t, s in zip(tables, seq_lens):
            if len(t) * bs < s:
                t.append(free.popleft())
    return tables


def varlen_workload(name, dtype, block_size, num_heads, num_kv_heads, head_dim, seq_lens, query_lens, *,
                    num_blocks=None, tables=None, std=1.0, seed=0, causal=True, slack=0.10,
                    device="cpu") -> Workload:
    """Request i has seq_lens[i] tokens after the step, the last query_lens[i]
    of them new; the earlier ones are cached."""
    seq_lens = np.asarray(seq_lens, np.int32)
    query_lens = np.asarray(query_lens, np.int32)
    assert np.all(query_lens <= seq_lens)
    S = seq_lens.shape[0]
    need = sum(_blocks_for(int(L), block_size) for L in seq_lens)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * (1.0 + slack))))
    if tables is None:
        tables = _shuffled_tables(seq_lens, block_size, num_blocks, seed)
    g = _gen(seed + 1, device)
    N = int(query_lens.sum())
    cached = seq_lens - query_lens
    pre_seq, pre_pos = _rows_for(cached)
    new_seq = np.repeat(np.arange(S, dtype=np.int32), query_lens.astype(np.int64))
    new_pos = np.concatenate([np.arange(int(cached[i]), int(seq_lens[i]), dtype=np.int64) for i in range(S)]) \
        if S else np.zeros(0, np.int64)
    q = _normal(g, (N, num_heads, head_dim), std, dtype)
    pre_k = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), std, dtype)
    pre_v = _normal(g, (pre_pos.shape[0], num_kv_heads, head_dim), std, dtype)
    new_k = _normal(g, (N, num_kv_heads, head_dim), std, dtype)
    new_v = _normal(g, (N, num_kv_heads, head_dim), std, dtype)
    return Workload(
        name=name, dtype=dtype, block_size=block_size, num_blocks=num_blocks, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, scale=head_dim ** -0.5, causal=causal, seq_lens=seq_lens,
        query_lens=query_lens, block_tables=tables, pre_block_tables=tables, pre_seq_idx=pre_seq, pre_pos=pre_pos,
        pre_k=pre_k, pre_v=pre_v, new_seq_idx=new_seq, new_pos=new_pos, new_k=new_k, new_v=new_v, q=q, seed=seed)


CONFIGS = {
    "tiny_decode": tiny_decode,
    "gqa_decode_batch": gqa_decode_batch,
    "long_context_decode": long_context_decode,
    "mha_decode": mha_decode,
    "mixed_varlen": mixed_varlen,
}


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Host copy of a tensor's elements as numpy: float32 stays float32,
    16-bit types become their uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)
