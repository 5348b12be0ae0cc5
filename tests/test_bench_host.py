"""Host-side arithmetic of bench.py (CPU): the unique K/V bytes of a batch
whose requests share blocks, and the split of the varlen flops into parts."""
import os
import sys
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_116_gb300 import workloads as W  # noqa: E402


def test_unique_bytes_count_a_shared_block_once_with_its_longest_reader():
    # block 5 is full in both requests and read by a third for 10 tokens;
    # 7 and 9 are private tails of 4 and 2 tokens
    w = SimpleNamespace(num_seqs=3, block_size=16, num_kv_heads=2, head_dim=8, elt=2,
                        seq_lens=np.array([20, 18, 10]),
                        block_tables=np.array([[5, 7], [5, 9], [5, -1]]))
    row = 2 * 8 * 2 * 2  # Hkv x hd x (K, V) x bytes
    assert bench.unique_kv_bytes(w) == (16 + 4 + 2) * row


def test_unique_bytes_of_the_mixed_batch_are_below_the_per_reader_bytes():
    w = W.mixed_varlen()
    per_reader = int(w.seq_lens.sum()) * w.num_kv_heads * w.head_dim * 2 * w.elt
    uniq = bench.unique_kv_bytes(w)
    # 60 groups of 4 samples share a 300-token prompt's 18 full blocks
    shared = 60 * 3 * 18 * 16 * w.num_kv_heads * w.head_dim * 2 * w.elt
    assert uniq == per_reader - shared


def test_varlen_flops_of_the_parts_add_up():
    w = W.mixed_varlen()
    pre = np.where(w.query_lens > 1)[0]
    dec = np.where(w.query_lens == 1)[0]
    total = bench.varlen_flops(w)
    assert abs(bench.varlen_flops(w, pre) + bench.varlen_flops(w, dec) - total) <= 1e-9 * total
    # a decode row attends to all L keys: 4 Hq hd L flops
    i = int(dec[0])
    assert bench.varlen_flops(w, [i]) == 4.0 * w.num_heads * w.head_dim * int(w.seq_lens[i])


def test_reference_arm_prints_the_contract_line(capsys):
    """The reference arm (the CPU oracle, rank 0) prints one JSON line with
    the GPU arm's metric, unit and workload name, and no host copies."""
    import json

    class Args:
        workload = "tiny_decode"
        kv_dtype = "native"
        steps = 2
        warmup = 1

    bench.run_reference(Args(), rank=0)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] == W.tiny_decode().name
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
