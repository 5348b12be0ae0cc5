"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1).

Each rank works its shard of the batch (the sequences are independent,
there is no data-path collective), so the only cross-rank steps are the
barrier, the max of the ranks' times and the sum of their units; the
whole-job rate is every rank's units over the slowest rank's time.  The
reference arm runs on rank 0 only; the other ranks exit without work.  The
shards themselves are checked in test_shard.py, and bench.py's workload on
two ranks here."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank])
        units = bench.sum_over_ranks(1000 + 500 * rank)  # shards of unequal size
        w = bench.make_workload("gqa_decode_batch", "cpu", 16, rank, world)
        seqs = bench.sum_over_ranks(w.num_seqs)
        out[rank] = (ms, bench.whole_job_rate(units, 10, ms), seqs, w.seq_lens.tolist())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    times = [12.5, 20.0]  # ms over the timed steps, rank 1 is slower
    with mp.get_context("spawn").Manager() as m:  # no fork of a threaded test process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, rate, seqs, _ = res[r]
        assert ms == 20.0
        assert rate == pytest.approx((1000 + 1500) * 10 / 0.020)
        assert seqs == 128  # two ranks: a batch twice the 64-sequence configuration
    # the two shards hold the 128 sequences of the doubled batch, in order
    sys.path.insert(0, ROOT)
    from paged_kv_cache_116_gb300 import workloads as W

    assert res[0][3] + res[1][3] == W.gqa_batch_lengths(128).tolist()


def test_without_a_process_group_the_time_is_the_rank_own():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.25) == 7.25
    assert bench.sum_over_ranks(64) == 64
    assert bench.whole_job_rate(64, 100, 50.0) == pytest.approx(64 * 100 / 0.05)


def test_reference_arm_on_a_nonzero_rank_exits_without_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload = "gqa_decode_batch"
        kv_dtype = "native"
        steps = 1
        warmup = 0

    bench.run_reference(Args(), rank=1)
    assert capsys.readouterr().out == ""
