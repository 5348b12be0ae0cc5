"""CPU checks of the seeded input layouts the GPU parity tests use: the
forked-sample varlen batch writes every cached and new row to its own slot,
shares exactly the prompt's full blocks inside a group, and gives each
sample its own blocks from the partial tail on."""
import numpy as np

import oracle
from paged_kv_cache_116_gb300 import workloads as W

LAYOUT = [("chunk", 40, 20), ("group", 37, [0, 5, 21, 3]), ("single", 50), ("group", 16, [0, 0, 17]),
          ("group", 7, [2, 9]), ("group", 300, [0, 0, 0, 0, 0])]


def _requests(layout):
    """(kind, prompt_len, extra) per request, in order."""
    out = []
    for item in layout:
        if item[0] == "group":
            out += [("group", item[1], e) for e in item[2]]
        else:
            out.append((item[0], None, None))
    return out


def test_forked_decode_mix_slots_are_distinct_and_in_range():
    for bs in (8, 16, 32):
        w = W.forked_decode_mix(LAYOUT, "bf16", bs, 8, 2, 64, seed=bs)
        pre = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, bs)
        new = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, bs)
        slots = np.concatenate([pre, new])
        assert np.all(slots >= 0) and np.all(slots < w.num_blocks * bs)
        assert len(np.unique(slots)) == len(slots)
        # every request's rows 0 .. L-1 are written exactly once (shared rows once per group)
        assert new.shape[0] == int(w.query_lens.sum())


def test_forked_decode_mix_shares_the_prompts_full_blocks_only():
    bs = 8
    w = W.forked_decode_mix(LAYOUT, "bf16", bs, 8, 2, 64, seed=3)
    reqs = _requests(LAYOUT)
    assert len(reqs) == w.num_seqs
    i = 0
    for item in LAYOUT:
        if item[0] != "group":
            i += 1
            continue
        prompt, extras = item[1], item[2]
        members = list(range(i, i + len(extras)))
        shared = prompt // bs
        for j, r in enumerate(members):
            L = int(w.seq_lens[r])
            assert L == prompt + extras[j] + 1 and int(w.query_lens[r]) == 1
            nb = -(-L // bs)
            row = w.block_tables[r]
            assert np.all(row[:nb] >= 0) and np.all(row[nb:] == W.PAD)
            # the full prompt blocks are the first member's; the rest are the member's own
            assert np.array_equal(row[:shared], w.block_tables[members[0]][:shared])
            for r2 in members:
                if r2 != r:
                    assert not set(row[shared:nb].tolist()) & set(w.block_tables[r2][:-(-int(w.seq_lens[r2]) // bs)].tolist())
        i += len(extras)
