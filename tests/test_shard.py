"""Splitting a batch across ranks (paged_kv_cache_116_gb300.shard), on CPU.

Checked: every (sequence, KV head) lands on exactly one rank; each shard's
block tables are valid for its own pool and keep the batch's sharing pattern
(two table entries name one block in the shard exactly when they did in the
batch); and -- on two gloo ranks -- the shards' oracle outputs, put back in
order, equal the oracle's output for the whole batch bit for bit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from paged_kv_cache_116_gb300 import shard as SH  # noqa: E402
from paged_kv_cache_116_gb300 import workloads as W  # noqa: E402


def _small_batches():
    return {
        "gqa": W.gqa_decode_batch(num_seqs=10),
        "mixed": W.mixed_varlen(num_chunks=3, num_groups=4, chunk_range=(20, 60), cached_range=(0, 40)),
        "mha": W.decode_workload("mha_small", "f16", 16, 8, 8, 64, W.mha_lengths(9, 0) // 4 + 1, std=0.5, seed=3),
    }


def _check_tables(whole, part, sel):
    """The shard's tables are valid for its pool and name the same blocks
    (up to renumbering) as the batch's rows `sel`."""
    bs = part.block_size
    for tables_p, tables_w in ((part.block_tables, whole.block_tables), (part.pre_block_tables, whole.pre_block_tables)):
        assert tables_p.shape[0] == len(sel)
        seen = {}
        for k, i in enumerate(sel):
            nb = (int(whole.seq_lens[i]) + bs - 1) // bs
            row_p, row_w = tables_p[k], tables_w[i]
            assert np.all(row_p[row_w == W.PAD] == W.PAD)
            for b_p, b_w in zip(row_p[row_w != W.PAD], row_w[row_w != W.PAD]):
                assert 0 <= b_p < part.num_blocks
                assert seen.setdefault(int(b_w), int(b_p)) == int(b_p)  # one global block -> one local block
            if tables_p is part.block_tables:
                assert np.all(row_p[:nb] != W.PAD)
        assert len(set(seen.values())) == len(seen)  # and no two global blocks share a local one


@pytest.mark.parametrize("name", ["gqa", "mixed", "mha"])
@pytest.mark.parametrize("world", [2, 3, 4])
def test_sequence_split_covers_every_unit_once_with_valid_tables(name, world):
    w = _small_batches()[name]
    shards = SH.split_sequences(w, world)
    assert sorted(np.concatenate(shards).tolist()) == list(range(w.num_seqs))
    for r, sel in enumerate(shards):
        part = SH.shard(w, r, world)
        assert part.num_seqs == len(sel)
        _check_tables(w, part, sel)
        assert part.q.shape[0] == int(w.query_lens[sel].sum())


def test_sharing_groups_stay_together_and_the_cut_balances_work():
    w = W.mixed_varlen(num_chunks=4, num_groups=6)
    groups = SH.request_groups(w)
    # 4 lone chunks, then 6 groups of the 4 samples that share a prompt
    assert [len(g) for g in groups] == [1] * 4 + [4] * 6
    for world in (2, 3):
        shards = SH.split_sequences(w, world)
        for g in groups:
            assert sum(set(g) <= set(s.tolist()) for s in shards) == 1
    w = W.gqa_decode_batch(num_seqs=64)
    pairs = SH.attended_pairs(w.seq_lens, w.query_lens)
    loads = [pairs[s].sum() for s in SH.split_sequences(w, 4)]
    assert max(loads) - min(loads) <= pairs.max()  # within one request of even


def test_kv_head_split_covers_every_head_once():
    w = _small_batches()["gqa"]
    for world in (1, 2, 4, 8):
        heads = SH.split_kv_heads(w.num_kv_heads, world)
        assert sorted(h for r in heads for h in r) == list(range(w.num_kv_heads))
        part = SH.shard(w, 0, world, by="kv_head")
        assert part.num_kv_heads * world == w.num_kv_heads and part.num_heads * world == w.num_heads
        assert np.array_equal(part.block_tables, w.block_tables)
    with pytest.raises(ValueError):
        SH.split_kv_heads(8, 3)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    from helpers import oracle_attention

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for name, w in _small_batches().items():
            for by in ("sequence", "kv_head"):
                part = SH.shard(w, rank, world, by=by)
                got = oracle_attention(part) if part.num_seqs else np.zeros((0, part.num_heads, w.head_dim))
                gathered = [None] * world
                dist.all_gather_object(gathered, got)
                if rank == 0:
                    axis = 0 if by == "sequence" else 1
                    out[(name, by)] = bool(np.array_equal(np.concatenate(gathered, axis=axis), oracle_attention(w)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_single_rank_oracle_output_bit_for_bit():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert len(res) == 6 and all(res.values()), res
