"""Splitting a batch of paged-attention requests across GPUs (host side).

Requests are independent, and so are the KV heads within a request (every
query head reads only its own KV head: "分页 KV Cache", §分页注意力,
`paged_attention`), so a batch shards with no exchange on the data path:

- by sequence: each rank takes a contiguous run of requests and holds only
  their blocks, in a block pool of its own;
- by KV head: each rank takes an equal share of the KV heads (and their
  query heads) of every request; the block tables stay as they are, and each
  rank's pool holds its heads' part of every token row.

The pages fix no policy for this; they only note that how a cache is sharded
changes what each device must hold ("KV cache：容量推导、分页与回收",
§输入放得下，输出还要留空间).  The readings here:

- Requests that share a block (a forked prompt, its copy-on-write tail) stay
  on one rank, so a shard never needs a block another rank writes: the cut
  falls between connected groups of requests (requests joined by any block
  id in their tables before or after the step, or by a copy).
- The cut balances the (query, key) pairs each rank attends -- for request
  i, n_i * L_i - n_i (n_i - 1) / 2 with n_i new tokens and L_i the context
  after the step -- by giving each group to the rank whose share of the
  running total its midpoint falls in.  It depends on the lengths only.
- A rank's pool holds the blocks its requests use, numbered in the order of
  their global ids (so a shuffled global pool stays shuffled).

Nothing here does arithmetic of the method: it selects rows and renumbers
block ids.  The shards' outputs, put back in order, are the batch's output.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np

from .workloads import PAD, Workload


def attended_pairs(seq_lens, query_lens) -> np.ndarray:
    """(query, key) pairs request i attends in a causal step: its n_i new
    tokens see L_i - n_i + 1, ..., L_i keys."""
    L = np.asarray(seq_lens, np.int64)
    n = np.asarray(query_lens, np.int64)
    return n * L - n * (n - 1) // 2


def request_groups(w: Workload) -> list[list[int]]:
    """Requests joined by a shared block id (in the tables before or after
    the step, or through a copy pair), as sorted lists in request order."""
    S = w.num_seqs
    parent = list(range(S))

    def find(a):
        while parent[a] != a:
            parent[a] = parent[parent[a]]
            a = parent[a]
        return a

    owner = {}
    copy_src = {int(d): int(s) for s, d in w.cow_pairs.reshape(-1, 2)} if w.cow_pairs.size else {}
    for tables in (w.pre_block_tables, w.block_tables):
        for i in range(S):
            for b in tables[i]:
                b = int(b)
                if b == PAD:
                    continue
                for key in (b, copy_src.get(b, b)):
                    if key in owner:
                        ra, rb = find(i), find(owner[key])
                        if ra != rb:
                            parent[max(ra, rb)] = min(ra, rb)
                    else:
                        owner[key] = i
    groups = {}
    for i in range(S):
        groups.setdefault(find(i), []).append(i)
    return sorted(groups.values(), key=lambda g: g[0])


def split_sequences(w: Workload, world: int) -> list[np.ndarray]:
    """Request indices of each rank (ascending); groups of requests that
    share blocks are never cut, and ranks are balanced by attended pairs."""
    if world < 1:
        raise ValueError("world must be positive")
    groups = request_groups(w)
    pairs = attended_pairs(w.seq_lens, w.query_lens)
    weight = np.array([pairs[g].sum() for g in groups], np.float64)
    total = weight.sum()
    mids = np.cumsum(weight) - weight / 2
    owner = np.minimum((mids * world / total).astype(np.int64), world - 1) if total > 0 else \
        np.minimum(np.arange(len(groups)) * world // max(len(groups), 1), world - 1)
    shards = [[] for _ in range(world)]
    for g, r in zip(groups, owner):
        shards[int(r)].extend(g)
    return [np.array(sorted(s), np.int64) for s in shards]


def split_kv_heads(num_kv_heads: int, world: int) -> list[range]:
    """KV heads of each rank: equal contiguous shares."""
    if world < 1 or num_kv_heads % world:
        raise ValueError("num_kv_heads (%d) must be a multiple of the number of ranks (%d)" % (num_kv_heads, world))
    h = num_kv_heads // world
    return [range(r * h, (r + 1) * h) for r in range(world)]


def _query_rows(w: Workload, sel: np.ndarray) -> np.ndarray:
    qsl = w.query_start_loc
    return np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in sel]).astype(np.int64) if len(sel) else \
        np.zeros(0, np.int64)


def shard_by_sequence(w: Workload, sel) -> Workload:
    """The part of w that requests `sel` (ascending) make up, with a block
    pool of their blocks only."""
    sel = np.asarray(sel, np.int64)
    used = set()
    for tables in (w.pre_block_tables, w.block_tables):
        for i in sel:
            used.update(int(b) for b in tables[i] if b != PAD)
    pairs = [(int(s), int(d)) for s, d in w.cow_pairs.reshape(-1, 2) if int(d) in used]
    used.update(s for s, _ in pairs)
    order = sorted(used)
    local = {b: k for k, b in enumerate(order)}
    remap = np.vectorize(lambda b: local[int(b)] if b != PAD else PAD, otypes=[np.int32])

    def tables_of(t):
        sub = t[sel]
        return remap(sub) if sub.size else sub.astype(np.int32)

    seq_local = np.full(w.num_seqs, -1, np.int64)
    seq_local[sel] = np.arange(len(sel))
    pre_mask = np.isin(w.pre_seq_idx, sel)
    new_mask = np.isin(w.new_seq_idx, sel)
    rows = _query_rows(w, sel)
    return replace(
        w, name="%s_shard" % w.name, num_blocks=max(len(order), 1), seq_lens=w.seq_lens[sel],
        query_lens=w.query_lens[sel], block_tables=tables_of(w.block_tables),
        pre_block_tables=tables_of(w.pre_block_tables),
        pre_seq_idx=seq_local[w.pre_seq_idx[pre_mask]].astype(np.int32), pre_pos=w.pre_pos[pre_mask],
        pre_k=w.pre_k[_index(pre_mask, w.pre_k)], pre_v=w.pre_v[_index(pre_mask, w.pre_v)],
        new_seq_idx=seq_local[w.new_seq_idx[new_mask]].astype(np.int32), new_pos=w.new_pos[new_mask],
        new_k=w.new_k[_index(new_mask, w.new_k)], new_v=w.new_v[_index(new_mask, w.new_v)],
        q=w.q[_index(rows, w.q)],
        cow_pairs=np.array([(local[s], local[d]) for s, d in pairs], np.int64).reshape(-1, 2))


def shard_by_kv_head(w: Workload, heads: range) -> Workload:
    """KV heads `heads` of every request of w, with their query heads; the
    pool keeps every block and holds only these heads of each token row."""
    G = w.num_heads // w.num_kv_heads
    h0, h1 = heads.start, heads.stop
    return replace(
        w, name="%s_heads%d_%d" % (w.name, h0, h1), num_heads=(h1 - h0) * G, num_kv_heads=h1 - h0,
        pre_k=w.pre_k[:, h0:h1].contiguous(), pre_v=w.pre_v[:, h0:h1].contiguous(),
        new_k=w.new_k[:, h0:h1].contiguous(), new_v=w.new_v[:, h0:h1].contiguous(),
        q=w.q[:, h0 * G:h1 * G].contiguous())


def shard(w: Workload, rank: int, world: int, by: str = "sequence") -> Workload:
    """Rank `rank`'s part of w when it is split `world` ways."""
    if by == "sequence":
        return shard_by_sequence(w, split_sequences(w, world)[rank])
    if by == "kv_head":
        return shard_by_kv_head(w, split_kv_heads(w.num_kv_heads, world)[rank])
    raise ValueError("by must be 'sequence' or 'kv_head'")


def _index(mask_or_rows, t):
    """numpy mask or row indices -> an index for tensor t (on t's device)."""
    import torch

    return torch.as_tensor(np.asarray(mask_or_rows), device=t.device)
