"""Benchmark of the paged-KV hot path (default: the 64-sequence GQA decode batch).

A step is one pass of the path over one batch, through the C ABI:
  decode workloads: pa_decode_append -- each sequence's new token is written
                    at its translated slot and the batch is decoded, in one
                    launch (--unfused: pa_slot_mapping -> pa_write_kv ->
                    pa_decode, three launches; both times are reported)
  mixed_varlen:     pa_copy_blocks (copy-on-write of the shared tails) ->
                    pa_slot_mapping -> pa_write_kv (every new token) ->
                    pa_varlen (prefill chunks + decode rows)
  --kv-dtype fp8:   a workload over the quantized cache (E4M3 codes, one
                    fp32 scale per token and KV head); decode: pa_decode_append_fp8
                    (the new rows quantized into their slots, then the decode;
                    --unfused: pa_slot_mapping -> pa_write_kv_fp8 ->
                    pa_decode_fp8); mixed_varlen: the block copies move code
                    and scale blocks, pa_write_kv_fp8, pa_varlen_fp8; its
                    K/V bytes are the codes plus the scales
Inputs are resident in HBM.  Enough copies of the K/V pool to exceed twice
the 129 MB L2 alternate between steps, so no step reads a pool the previous
one left in L2.  The step is captured once per pool copy as a CUDA graph and
replayed (what a serving loop does); `eager_ms_per_step` is the same calls
issued one by one.

Prints ONE JSON line (rank 0).  `value` is the algorithmic K/V bytes the
step's attention reads over the step's device time (GB/s); `roofline` is the
dominant kernel timed alone (its own graph, same rotation) against the
measured HBM copy bandwidth (decode) or the measured bf16 tensor rate
(varlen); `e2e` is the step with its inputs copied from pinned host memory
and its output copied back inside the timed region, pipelined as a serving
loop runs it (two buffer sets and two copy streams, so a step's copies
overlap its neighbours' kernels); `cpu_baseline` is the
CPU oracle on a bounded sample.  `--impl reference` times that oracle alone
as the reference arm.

Multi-GPU (torchrun, N ranks): the batch is N times the configuration,
drawn by the same generators, and each rank takes its shard -- a
length-balanced cut by sequence, the rank holding only its requests' blocks
(weak scaling, no data-path collective); `value` sums all ranks' bytes over
the slowest rank's time.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (fraction of HBM peak) and sequences/s, 1×GB300"
L2_BYTES = 129 * 10 ** 6
WORKLOADS = ("gqa_decode_batch", "long_context_decode", "mha_decode", "tiny_decode", "mixed_varlen")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="gqa_decode_batch")
    ap.add_argument("--no-rotate", action="store_true", help="one pool copy (for profiling)")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, clocks and cpu_baseline")
    ap.add_argument("--block-size", type=int, default=16,
                    help="block size of the GQA decode batch (the block-size sweep); other workloads keep theirs")
    ap.add_argument("--swap", action="store_true",
                    help="measure pa_swap_blocks (device pool <-> pinned host pool) instead of the attention step")
    ap.add_argument("--unfused", action="store_true",
                    help="decode step as pa_slot_mapping + pa_write_kv + pa_decode instead of pa_decode_append")
    ap.add_argument("--kv-dtype", choices=["native", "fp8"], default="native",
                    help="fp8: the workload over an FP8 E4M3 cache (queries keep the workload's type)")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def traffic_key(workload, fp8, block_size):
    """Key of a workload's record in the committed ncu traffic table: the
    workload, then "_fp8" over a quantized cache, then "_bs<n>" for a block
    size other than 16."""
    return workload + ("_fp8" if fp8 else "") + ("" if block_size == 16 else "_bs%d" % block_size)


def traffic_record(workload, kernel_file):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary of this workload, if it was taken on the current kernel source."""
    if workload is None:
        return None
    src = os.path.join(ROOT, "paged_kv_cache_116_gb300", "csrc", kernel_file)
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload, {})
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("source_sha256") == sha:
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# ---------------------------------------------------------------- ranks

def max_over_ranks(x, device=None):
    """The largest of every rank's x (the slowest rank's time); x itself
    without a process group.  Collective: every rank must call it."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, device=None):
    """The sum of every rank's x; x itself without a process group.
    Collective: every rank must call it."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_rate(units_per_step_all_ranks, steps, ms):
    """Units per second over the whole job: every rank's units of a step
    (each rank holds its shard of the batch) over the slowest rank's time."""
    return units_per_step_all_ranks * steps / (ms / 1e3)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + q, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", os.environ.get("LOCAL_RANK", "0")],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workloads


def make_workload(name, device, block_size=16, rank=0, world=1):
    """The named configuration (one GPU), or -- on `world` ranks -- rank's
    shard of a batch `world` times as large drawn by the same generators
    (weak scaling): requests split by a length-balanced cut, each rank
    holding only its requests' blocks (paged_kv_cache_116_gb300.shard)."""
    from paged_kv_cache_116_gb300 import shard as SH
    from paged_kv_cache_116_gb300 import workloads as W

    n = world
    if name == "tiny_decode":
        w = W.tiny_decode() if n == 1 else W.decode_workload(
            "tiny_decode_fp32_bs4", "f32", 4, 4, 2, 32, [6, 13, 1, 20] * n, num_blocks=32 * n, scale=32 ** -0.5)
    elif name == "gqa_decode_batch":
        w = W.gqa_decode_batch(num_seqs=64 * n, device=device, block_size=block_size)
    elif name == "long_context_decode":
        w = W.long_context_decode(num_seqs=8 * n, device=device)
    elif name == "mha_decode":
        w = W.mha_decode(num_seqs=128 * n, device=device)
    else:
        w = W.mixed_varlen(num_chunks=16 * n, num_groups=60 * n, device=device)
    return w if n == 1 else SH.shard(w, rank, n, by="sequence")


def varlen_flops(w, select=None):
    """2 x the multiply-adds of Q K^T and P V over the causal (or full) key ranges
    (of the requests in `select`, default all)."""
    total = 0.0
    idx = range(w.num_seqs) if select is None else select
    for i in idx:
        n, L = int(w.query_lens[i]), int(w.seq_lens[i])
        total += n * (L - n) + n * (n + 1) / 2 if w.causal else n * L
    return 4.0 * w.num_heads * w.head_dim * total


def unique_kv_bytes(w):
    """K/V bytes of the distinct pool rows the step's attention reads: a block
    shared by several requests (a forked prompt) counts once, with the most
    tokens any reader uses of it."""
    used = {}
    for i in range(w.num_seqs):
        L = int(w.seq_lens[i])
        for j in range((L + w.block_size - 1) // w.block_size):
            b = int(w.block_tables[i, j])
            used[b] = max(used.get(b, 0), min(w.block_size, L - j * w.block_size))
    return sum(used.values()) * w.num_kv_heads * w.head_dim * 2 * w.elt


def oracle_setup(w):
    """Oracle-side pool of a (host) workload after the step's copies and writes."""
    import numpy as np

    import oracle
    from paged_kv_cache_116_gb300 import workloads as W

    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    if w.dtype == "f32":
        kc = np.full(shape, np.nan, np.float32)
    else:
        kc = np.full(shape, 0x7FC0 if w.dtype == "bf16" else 0x7E00, np.uint16)
    vc = kc.copy()
    s = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, w.block_size)
    oracle.write_kv(W.raw_numpy(w.pre_k), W.raw_numpy(w.pre_v), s, kc, vc)
    if w.cow_pairs.shape[0]:
        oracle.copy_blocks([kc], [vc], w.cow_pairs)
    s = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, w.block_size)
    oracle.write_kv(W.raw_numpy(w.new_k), W.raw_numpy(w.new_v), s, kc, vc)
    return kc, vc, W.raw_numpy(w.q)


def oracle_step(w, kc, vc, q, num_threads=0):
    import oracle

    return oracle.paged_attention(q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.scale, w.dtype,
                                  w.causal, num_threads=num_threads)


def oracle_setup_fp8(w):
    """Oracle-side quantized pool (codes and scales) of a host workload after its step's writes and copies."""
    import numpy as np

    import oracle
    from paged_kv_cache_116_gb300 import workloads as W

    kc = np.full((w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), 0x7F, np.uint8)
    vc = kc.copy()
    ks = np.full((w.num_blocks, w.num_kv_heads, w.block_size), np.nan, np.float32)
    vs = ks.copy()
    s = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, w.block_size)
    oracle.write_kv_fp8(W.raw_numpy(w.pre_k), W.raw_numpy(w.pre_v), w.dtype, s, kc, vc, ks, vs)
    if w.cow_pairs.shape[0]:
        oracle.copy_blocks([kc], [vc], w.cow_pairs)
        oracle.copy_blocks([ks], [vs], w.cow_pairs)
    s = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, w.block_size)
    oracle.write_kv_fp8(W.raw_numpy(w.new_k), W.raw_numpy(w.new_v), w.dtype, s, kc, vc, ks, vs)
    return (kc, vc, ks, vs), W.raw_numpy(w.q)


def oracle_step_fp8(w, pools, q, num_threads=0):
    import oracle

    return oracle.paged_attention_fp8(q, w.dtype, *pools, w.block_tables, w.seq_lens, w.query_start_loc, w.scale,
                                      w.causal, num_threads=num_threads)


def fp8_kv_bytes(w):
    """Bytes of the quantized cache a decode step reads: per context token and
    KV head, head_dim codes and one fp32 scale, for K and for V."""
    return int(w.seq_lens.astype("int64").sum()) * w.num_kv_heads * 2 * (w.head_dim + 4)


def host_sample_workload(name):
    """A bounded sample of a workload with the same generators, values drawn
    on the host: its first requests (or, for the mixed step, fewer chunks and
    sampling groups)."""
    from paged_kv_cache_116_gb300 import workloads as W

    return {"gqa_decode_batch": lambda: W.gqa_decode_batch(num_seqs=8),
            "long_context_decode": lambda: W.long_context_decode(num_seqs=1),
            "mha_decode": lambda: W.mha_decode(num_seqs=16),
            "tiny_decode": W.tiny_decode,
            "mixed_varlen": lambda: W.mixed_varlen(num_chunks=1, num_groups=4)}[name]()


def oracle_runner(w, fp8):
    """(one oracle step as a callable taking a thread count, 0 = all cores;
    K/V bytes it reads) for a host workload."""
    if fp8:
        pools, q = oracle_setup_fp8(w)
        return (lambda nt=0: oracle_step_fp8(w, pools, q, nt)), fp8_kv_bytes(w)
    kc, vc, q = oracle_setup(w)
    return (lambda nt=0: oracle_step(w, kc, vc, q, nt)), w.kv_bytes_read()


def cpu_sample(name, budget_s=10.0, fp8=False):
    """The oracle (as it stands) on a bounded sample of the workload,
    repeated for about budget_s seconds."""
    import oracle

    w = host_sample_workload(name)
    run, per_step = oracle_runner(w, fp8)
    cores = oracle.max_threads()

    def timed_reps(nt, budget):
        reps, t = 0, time.perf_counter()
        while True:
            run(nt)
            reps += 1
            el = time.perf_counter() - t
            if el >= budget:
                return reps, el

    reps, el = timed_reps(0, budget_s)
    # then one core (last: the oracle's thread count persists in the process)
    reps1, el1 = timed_reps(1, budget_s / 3)
    return {"value": per_step * reps / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d requests of the same generators (%d context tokens) x %d, fp64 C oracle with OpenMP%s, "
                      "%.1f s" % (w.num_seqs, int(w.seq_lens.sum()), reps, ", FP8 cache" if fp8 else "", el),
            "seq_per_s": w.num_seqs * reps / el,
            "single_core": {"value": per_step * reps1 / el1 / 1e9, "unit": "GB/s",
                            "seq_per_s": w.num_seqs * reps1 / el1, "reps": reps1}}


def run_reference(args, rank):
    """Reference arm: the CPU oracle on a bounded sample of the workload per
    step (rank 0 only)."""
    if rank != 0:
        return
    import oracle

    fp8 = args.kv_dtype == "fp8"
    w = host_sample_workload(args.workload)
    run, step_bytes = oracle_runner(w, fp8)
    for _ in range(args.warmup):
        run()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t
    value = step_bytes * args.steps / dt / 1e9
    desc = "%d requests of the %s generators per step, fp64 C oracle with OpenMP%s" % (
        w.num_seqs, args.workload, " over an FP8 cache" if fp8 else "")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + ("_fp8cache" if fp8 else ""), "sample_requests": w.num_seqs},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------- the GPU arm


def run_swap(args):
    """Preemption traffic: blocks of the GQA batch's geometry (16 tokens x 8
    KV heads x 128 x bf16 = 32 KiB per K or V block) across 8 layers move
    from the device pool to a pinned host pool and back, one pa_swap_blocks
    call per direction.  Beside it: the same blocks moved by one
    cudaMemcpyAsync per block and layer (torch copies, graph-captured), and
    one contiguous copy of the same byte count (the copy engines' rate, the
    denominator of frac)."""
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_116_gb300 as pa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers, nb_dev, nb_host, n, bs, hkv, hd = 8, 4096, 1024, 1024, 16, 8, 128
    g = torch.Generator(device=dev).manual_seed(0)
    mk = lambda nb: torch.randint(-32768, 32767, (nb, bs, hkv, hd), generator=g, dtype=torch.int16,  # noqa: E731
                                  device=dev).view(torch.bfloat16)
    dk = [mk(nb_dev) for _ in range(layers)]
    dv = [mk(nb_dev) for _ in range(layers)]
    hk = [torch.empty((nb_host, bs, hkv, hd), dtype=torch.bfloat16).pin_memory() for _ in range(layers)]
    hv = [torch.empty((nb_host, bs, hkv, hd), dtype=torch.bfloat16).pin_memory() for _ in range(layers)]
    rng = np.random.default_rng(0)
    picked = rng.choice(nb_dev, 2 * n, replace=False)  # blocks that go out, blocks they come back to
    src, back = picked[:n], picked[n:]
    dst = rng.permutation(nb_host)[:n]
    out_pairs = torch.from_numpy(np.stack([src, dst], 1).astype(np.int64)).to(dev)
    in_pairs = torch.from_numpy(np.stack([dst, back], 1).astype(np.int64)).to(dev)
    block_bytes = bs * hkv * hd * 2
    moved = 2 * layers * n * block_bytes  # K and V, one direction

    def graph(fn):
        fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, capture_error_mode="thread_local"):
            fn()
        return gr

    def per_block(a_k, a_v, b_k, b_v, pairs):
        pl = pairs.cpu().tolist()

        def fn():
            for l in range(layers):
                for s_, d_ in pl:
                    b_k[l][d_].copy_(a_k[l][s_], non_blocking=True)
                    b_v[l][d_].copy_(a_v[l][s_], non_blocking=True)
        return fn

    bulk_d = torch.empty(moved, dtype=torch.uint8, device=dev)
    bulk_h = torch.empty(moved, dtype=torch.uint8).pin_memory()
    gs = {
        "swap_out": graph(lambda: pa.pa_swap_blocks(dk, dv, hk, hv, out_pairs, stream=torch.cuda.current_stream())),
        "swap_in": graph(lambda: pa.pa_swap_blocks(hk, hv, dk, dv, in_pairs, stream=torch.cuda.current_stream())),
        "memcpy_out": graph(per_block(dk, dv, hk, hv, out_pairs)),
        "memcpy_in": graph(per_block(hk, hv, dk, dv, in_pairs)),
        "bulk_out": graph(lambda: bulk_h.copy_(bulk_d, non_blocking=True)),
        "bulk_in": graph(lambda: bulk_d.copy_(bulk_h, non_blocking=True)),
    }
    reps = max(args.steps if args.steps < 20000 else 20, 3)
    res = {}
    for name, gr in gs.items():
        for _ in range(max(args.warmup if args.warmup < 20 else 3, 3)):
            gr.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            gr.replay()
        b.record()
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / reps
    # parity of what was timed: the last swap-in brought the out-swapped blocks back
    for l in (0, layers - 1):
        assert torch.equal(dk[l][torch.from_numpy(back).to(dev)].view(torch.int16),
                           dk[l][torch.from_numpy(src).to(dev)].view(torch.int16))
    gbs = {k: moved / (v / 1e3) / 1e9 for k, v in res.items()}
    line = {
        "metric": "block swap GB/s, device pool <-> pinned host pool", "value": gbs["swap_out"], "unit": "GB/s",
        "n_gpus": 1, "steps": reps, "warmup": 3, "ms_per_step": res["swap_out"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (moved as bytes)", "data": "synthetic",
        "config": {"workload": "swap_blocks", "layers": layers, "blocks_per_direction": n, "block_size": bs,
                   "num_kv_heads": hkv, "head_dim": hd, "bytes_per_direction": moved,
                   "step": "one pa_swap_blocks call (all layers, K and V), replayed as a CUDA graph"},
        "swap_in_gbs": gbs["swap_in"],
        "per_block_memcpy_gbs": {"out": gbs["memcpy_out"], "in": gbs["memcpy_in"],
                                 "copies_per_direction": 2 * layers * n},
        "roofline": {"bound": "link", "kernel": "swap_blocks_kernel", "achieved": gbs["swap_out"],
                     "peak": gbs["bulk_out"], "unit": "GB/s", "frac": gbs["swap_out"] / gbs["bulk_out"],
                     "peak_kind": "measured here: one contiguous cudaMemcpyAsync of the same bytes, same direction",
                     "in": {"achieved": gbs["swap_in"], "peak": gbs["bulk_in"],
                            "frac": gbs["swap_in"] / gbs["bulk_in"]},
                     "traffic": None},
        "gpu_launches": reps,
        "ms": res,
    }
    print(json.dumps(line))




def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.swap:
        if rank == 0:
            run_swap(args)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__

    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import paged_kv_cache_116_gb300 as pa
    from paged_kv_cache_116_gb300 import workloads as W

    w = make_workload(args.workload, dev, args.block_size, rank, world)
    tdt = W.TORCH_DTYPES[w.dtype]
    S, hq, hkv, hd, bs = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    decode = w.is_decode and w.cow_pairs.shape[0] == 0
    fp8 = args.kv_dtype == "fp8"
    max_ctx, max_q = int(w.seq_lens.max()), int(w.query_lens.max())
    kv_bytes = fp8_kv_bytes(w) if fp8 else w.kv_bytes_read()
    N = int(w.query_lens.sum())

    # resident pools, filled through the library; enough copies to defeat L2
    pool_bytes = 2 * w.num_blocks * bs * hkv * (hd + 4 if fp8 else hd * w.elt)
    copies = 1 if args.no_rotate else min(16, max(2, math.ceil(2 * L2_BYTES / pool_bytes)))
    l2_note = ("inputs larger than L2: %d pool copies of %.3f GB alternate between steps" % (copies, pool_bytes / 1e9)
               if copies * pool_bytes > L2_BYTES else
               "pool of %.6f GB x %d copies stays in L2 (launch-bound case)" % (pool_bytes / 1e9, copies))
    pools = []
    pre_slots = None
    if w.pre_pos.shape[0]:
        pre_slots = pa.pa_slot_mapping(torch.from_numpy(w.pre_block_tables).to(dev),
                                       torch.from_numpy(w.pre_seq_idx).to(dev), torch.from_numpy(w.pre_pos).to(dev),
                                       bs)
    pre_k = w.pre_k.to(dev) if pre_slots is not None else None
    pre_v = w.pre_v.to(dev) if pre_slots is not None else None
    for c in range(copies):
        if fp8:
            kc = torch.full((w.num_blocks, bs, hkv, hd), 0x7F, dtype=torch.uint8, device=dev)  # NaN codes
            vc = torch.full_like(kc, 0x7F)
            ks = torch.full((w.num_blocks, hkv, bs), float("nan"), dtype=torch.float32, device=dev)
            vs = torch.full_like(ks, float("nan"))
            pool = (kc, vc, ks, vs)
        else:
            kc = torch.full((w.num_blocks, bs, hkv, hd), float("nan"), dtype=tdt, device=dev)
            vc = torch.full_like(kc, float("nan"))
            pool = (kc, vc)
        if pre_slots is not None:
            (pa.pa_write_kv_fp8 if fp8 else pa.pa_write_kv)(pre_k, pre_v, pre_slots, *pool)
        pools.append(pool)
    w.pre_k = w.pre_v = pre_k = pre_v = None
    bt = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.query_start_loc).to(dev)
    seq_idx = torch.from_numpy(w.new_seq_idx).to(dev)
    pos = torch.from_numpy(w.new_pos).to(dev)
    pairs = torch.from_numpy(w.cow_pairs).to(dev)
    q, new_k, new_v = w.q.to(dev).contiguous(), w.new_k.to(dev).contiguous(), w.new_v.to(dev).contiguous()
    out = torch.empty_like(q)
    slot_buf = torch.empty(N, dtype=torch.int64, device=dev)
    if not decode:
        ws_bytes = (pa.pa_varlen_fp8_workspace_size if fp8 else pa.pa_varlen_workspace_size)(
            S, N, max_q, hq, hkv, hd, bs, max_ctx, tdt)
    elif decode:
        ws_bytes = (pa.pa_decode_fp8_workspace_size if fp8 else pa.pa_decode_workspace_size)(S, hq, hkv, hd, bs,
                                                                                              max_ctx, tdt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def attend(pool, qq, tables, ll, cuq, st, o=None):
        o = out if o is None else o
        if fp8 and not decode:
            pa.pa_varlen_fp8(o, qq, *pool, tables, ll, cuq, max_q, max_ctx, w.scale, causal=w.causal,
                             workspace=ws, stream=st)
        elif fp8:
            pa.pa_decode_fp8(o, qq, *pool, tables, ll, max_ctx, w.scale, workspace=ws, stream=st)
        elif decode:
            pa.pa_decode(o, qq, *pool, tables, ll, max_ctx, w.scale, workspace=ws, stream=st)
        else:
            pa.pa_varlen(o, qq, *pool, tables, ll, cuq, max_q, max_ctx, w.scale, causal=w.causal,
                         workspace=ws, stream=st)

    fused = decode and not args.unfused

    def run_step_unfused(i, t_in, o=None):
        pool = pools[i % copies]
        st = torch.cuda.current_stream()
        d_q, d_k, d_v, d_bt, d_lens, d_cu, d_seq, d_pos, d_pairs = t_in
        if d_pairs.shape[0]:
            pa.pa_copy_blocks(pool[0], pool[1], d_pairs, stream=st)
            if fp8:  # the scale pools' blocks move with the codes
                pa.pa_copy_blocks(pool[2], pool[3], d_pairs, stream=st)
        pa.pa_slot_mapping(d_bt, d_seq, d_pos, bs, slot_out=slot_buf, stream=st)
        (pa.pa_write_kv_fp8 if fp8 else pa.pa_write_kv)(d_k, d_v, slot_buf, *pool, stream=st)
        attend(pool, d_q, d_bt, d_lens, d_cu, st, o)

    def run_step(i, t_in, o=None):
        """One pass of the path through the C ABI on the current stream (output to o, default out)."""
        if not fused:
            return run_step_unfused(i, t_in, o)
        d_q, d_k, d_v, d_bt, d_lens = t_in[:5]
        (pa.pa_decode_append_fp8 if fp8 else pa.pa_decode_append)(
            out if o is None else o, d_q, d_k, d_v, *pools[i % copies], d_bt, d_lens, max_ctx, w.scale,
            workspace=ws, stream=torch.cuda.current_stream())

    dev_in = (q, new_k, new_v, bt, lens, cu, seq_idx, pos, pairs)
    if fused:
        dev_in = dev_in[:5]  # a fused step reads q, the new rows, the tables and the lengths

    def step(i):
        run_step(i, dev_in)

    def kernel_only(i):
        attend(pools[i % copies], q, bt, lens, cu, torch.cuda.current_stream())

    tc_decode = (decode and w.dtype in ("bf16", "f16") and hd in ((128, 256) if fp8 else (64, 128, 256)) and
                 hq // hkv <= 16 and (not fp8 or bs == 8 or (bs % 16 == 0 and bs <= 256)))
    # the append happens inside the decode kernel (a code cache: head_dim 128 and
    # no more (sequence, KV head) units than the grid's warps, 3 CTAs x 4 warps per SM)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused_in_kernel = tc_decode and (not fp8 or (hd == 128 and S * hkv <= sms * 3 * 4))
    # the tensor-core decode is two launches: the decode and its split merge
    launches_per_step = ((1 if fused_in_kernel else 2) if fused else 3 + (1 if pairs.shape[0] else 0)) + \
        (1 if tc_decode else 0) + (1 if fp8 and pairs.shape[0] else 0)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()

    def capture(fn):
        gs = []
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn(c)
            gs.append(g)
        return gs

    step_graphs, kern_graphs = capture(step), capture(kernel_only)
    unfused_graphs = capture(lambda i: run_step_unfused(i, (q, new_k, new_v, bt, lens, cu, seq_idx, pos, pairs))) \
        if fused else None
    for i in range(max(args.warmup, 3)):
        step_graphs[i % copies].replay()
        kern_graphs[i % copies].replay()
    torch.cuda.synchronize()

    def timed(fn_i, steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        a.record()
        for i in range(steps):
            fn_i(i)
        b.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return a.elapsed_time(b)

    clocks = Clocks()
    if rank == 0 and not args.no_extras:
        clocks.start()
        time.sleep(0.5)
    ms = timed(lambda i: step_graphs[i % copies].replay(), args.steps)
    clk = clocks.stop() if rank == 0 and not args.no_extras else None
    kern_ms = timed(lambda i: kern_graphs[i % copies].replay(), args.steps) / args.steps
    # the median of 51 launches timed one by one (CUDA events around each replay)
    kern_med_us = None
    if not args.no_extras:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(51)]
        torch.cuda.synchronize()
        for j, (ea, eb) in enumerate(evs):
            ea.record()
            kern_graphs[j % copies].replay()
            eb.record()
        torch.cuda.synchronize()
        kern_med_us = statistics.median(ea.elapsed_time(eb) for ea, eb in evs) * 1e3
    # the varlen mix's two parts, each as a pa_varlen call of its own over the
    # same pools (prefill chunks: tensor-bound; decode rows: HBM-bound); in the
    # mixed call they share one launch, so these times do not add up to it
    parts = None
    if not decode and not fp8 and not args.no_extras:
        parts = {}
        peaks_p, _ = measured_peaks()
        for name, sel in (("prefill_chunks", np.where(w.query_lens > 1)[0]),
                          ("decode_rows", np.where(w.query_lens == 1)[0])):
            if len(sel) == 0:
                continue
            rows = np.concatenate([np.arange(w.query_start_loc[i], w.query_start_loc[i + 1]) for i in sel])
            qp = q[torch.from_numpy(rows).to(dev).long()].contiguous()
            op = torch.empty_like(qp)
            cup = torch.from_numpy(np.concatenate([[0], np.cumsum(w.query_lens[sel])]).astype(np.int32)).to(dev)
            selt = torch.from_numpy(sel).to(dev).long()
            btp, lp = bt[selt].contiguous(), lens[selt].contiguous()
            mqp = int(w.query_lens[sel].max())

            def part_call(i, qp=qp, op=op, cup=cup, btp=btp, lp=lp, mqp=mqp):
                pa.pa_varlen(op, qp, *pools[i % copies], btp, lp, cup, mqp, max_ctx, w.scale, causal=w.causal,
                             workspace=ws, stream=torch.cuda.current_stream())

            for i in range(3):
                part_call(i)
            pg = capture(part_call)
            for i in range(3):
                pg[i % copies].replay()
            torch.cuda.synchronize()
            p_ms = timed(lambda i: pg[i % copies].replay(), args.steps) / args.steps
            fl = varlen_flops(w, sel)
            kvb = int(sum(int(w.seq_lens[i]) for i in sel)) * hkv * hd * 2 * w.elt
            parts[name] = {"requests": int(len(sel)), "query_rows": int(len(rows)), "kernel_us": p_ms * 1e3,
                           "TFLOP/s": fl / (p_ms / 1e3) / 1e12,
                           "tensor_frac": fl / (p_ms / 1e3) / 1e12 / peaks_p["bf16_tflops"],
                           "kv_bytes": kvb, "kv_GB/s": kvb / (p_ms / 1e3) / 1e9,
                           "hbm_frac": kvb / (p_ms / 1e3) / 1e9 / peaks_p["hbm_gbs"]}
    unfused_ms = (timed(lambda i: unfused_graphs[i % copies].replay(), args.steps) / args.steps
                  if unfused_graphs else None)
    eager_steps = min(args.steps, 2000)
    eager_ms = timed(step, eager_steps) / eager_steps
    ms = max_over_ranks(ms, dev)
    ms_step = ms / args.steps
    job_kv_bytes, job_seqs = sum_over_ranks(kv_bytes, dev), sum_over_ranks(S, dev)
    value = whole_job_rate(job_kv_bytes, args.steps, ms) / 1e9
    seq_per_s = whole_job_rate(job_seqs, args.steps, ms)

    # e2e: each step's inputs from pinned host memory -> H2D, the step, the
    # output D2H to pinned memory
    e2e = None
    if not args.no_extras:
        # the step's inputs live in one pinned host buffer (each tensor at a
        # 256-byte aligned offset) and cross to the device in one copy, as a
        # serving loop would stage them
        offs, at = [], 0
        for t in dev_in:
            offs.append(at)
            at += (t.numel() * t.element_size() + 255) // 256 * 256
        host_buf = torch.empty(max(at, 256), dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty_like(host_buf, device=dev)

        def views(buf):
            return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, dev_in)]

        for hv, t in zip(views(host_buf), dev_in):
            hv.copy_(t.cpu())
        dev_copy = views(dev_buf)
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in dev_in)
        d2h = h_out.numel() * h_out.element_size()

        # A serving loop's pipeline: two sets of input/output buffers; step i's
        # inputs cross (copy-in stream) while step i-1 computes, and its output
        # comes back (copy-out stream) while step i+1 computes.  Every step's
        # H2D and D2H copies are inside the timed region.
        host_bufs = [host_buf, torch.empty_like(host_buf).pin_memory()]
        host_bufs[1].copy_(host_buf)
        dev_bufs = [dev_buf, torch.empty_like(dev_buf)]
        dev_views = [views(b) for b in dev_bufs]
        outs = [out, torch.empty_like(out)]
        h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def pipe_step(i, s_comp):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])  # step i-2 has finished reading dev_bufs[b]
                dev_bufs[b].copy_(host_bufs[b], non_blocking=True)
                ev_in[b].record(s_in)
            s_comp.wait_event(ev_in[b])
            if i >= 2:
                s_comp.wait_event(ev_out[b])  # step i-2's output has left outs[b]
            run_step(i, dev_views[b], outs[b])
            ev_comp[b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                h_outs[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(s_out)

        # one CUDA graph holds GS pipelined steps (every pool copy, both buffer
        # sets) with the streams' event edges, and is replayed
        GS = copies if copies % 2 == 0 else 2 * copies
        while GS < 8:
            GS *= 2

        def pipe_block():
            cs = torch.cuda.current_stream()
            s_in.wait_stream(cs)
            s_out.wait_stream(cs)
            for i in range(GS):
                pipe_step(i, cs)
            cs.wait_stream(s_in)
            cs.wait_stream(s_out)

        pipe_block()
        torch.cuda.synchronize()
        pg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg, capture_error_mode="thread_local"):
            pipe_block()
        for _ in range(2):
            pg.replay()
        torch.cuda.synchronize()
        reps = max(1, min(args.steps, 5000) // GS)
        e_steps = reps * GS
        e_ms = max_over_ranks(timed(lambda i: pg.replay(), reps), dev)
        e2e = {"value": whole_job_rate(job_kv_bytes, e_steps, e_ms) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / e_steps,
               "how": "pinned-host inputs (one packed buffer per step) -> one H2D copy on a copy stream -> "
                      "the step's C-ABI calls -> D2H output on a second copy stream; two buffer sets, so "
                      "step i's copies overlap its neighbours' kernels; %d steps per CUDA graph replay" % GS}

    peaks, kind = measured_peaks()
    # the committed DRAM counters hold for one GPU's whole batch only
    tkey = traffic_key(args.workload, fp8, bs) if world == 1 else None
    if decode:
        nblk = int(sum((L + bs - 1) // bs for L in w.seq_lens.tolist()))
        alg = kv_bytes + 2 * S * hq * hd * w.elt + nblk * 4 + S * 4
        achieved = alg / (kern_ms / 1e3) / 1e9
        call = "pa_decode_fp8" if fp8 else "pa_decode"
        roof = {"bound": "hbm", "kernel": ("decode_tc_kernel%s (%s, split merge included)" % (
                    "<FP8>" if fp8 else "", call) if tc_decode else "attn_simt_kernel (%s, CUDA-core path)" % call),
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_kind": kind + " hbm_gbs", "algorithmic_bytes": alg,
                "traffic": traffic_record(tkey, "pa_decode_tc.cu") if tc_decode else None,
                "kernel_us": kern_ms * 1e3, "kernel_us_median_of_51": kern_med_us}
    elif fp8 and w.dtype in ("bf16", "f16") and hd == 128 and (bs == 8 or (bs % 16 == 0 and bs <= 256)):
        # the mixed step over a code cache on the tensor cores (codes turned
        # into f16 in shared memory by the producer warps)
        fl = varlen_flops(w)
        achieved = fl / (kern_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]  # the f16 rate equals the bf16 rate
        roof = {"bound": "tensor", "kernel": "varlen_umma_kernel<FP8> (pa_varlen_fp8, tcgen05)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": kind + " bf16_tflops (burst; f16 runs at the same rate)", "algorithmic_flops": fl,
                "kv_bytes": kv_bytes, "kv_GBps_in_kernel": kv_bytes / (kern_ms / 1e3) / 1e9,
                "traffic": traffic_record(tkey, "pa_varlen_umma.cu"),
                "kernel_us": kern_ms * 1e3, "kernel_us_median_of_51": kern_med_us}
    elif fp8:
        # the mixed step over a code cache on the CUDA-core kernel: its
        # bound is issue, reported here against the copy peak in K/V bytes
        achieved = kv_bytes / (kern_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "attn_simt_kernel<FP8> (pa_varlen_fp8, CUDA-core path)",
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_kind": kind + " hbm_gbs", "algorithmic_bytes": kv_bytes,
                "algorithmic_flops": varlen_flops(w), "traffic": None, "kernel_us": kern_ms * 1e3,
                "kernel_us_median_of_51": kern_med_us}
    else:
        fl = varlen_flops(w)
        achieved = fl / (kern_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "kernel": "varlen_umma_kernel (pa_varlen, tcgen05)", "achieved": achieved,
                "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": kind + " bf16_tflops (burst)",
                "algorithmic_flops": fl, "kv_bytes": kv_bytes, "kv_GBps_in_kernel": kv_bytes / (kern_ms / 1e3) / 1e9,
                "unique_kv_bytes": unique_kv_bytes(w), "parts": parts,
                "traffic": traffic_record(tkey, "pa_varlen_umma.cu"), "kernel_us": kern_ms * 1e3,
                "kernel_us_median_of_51": kern_med_us}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("e4m3 cache, %s q/out" % w.dtype) if fp8 else w.dtype, "data": "synthetic",
            "config": {"workload": w.name + ("_fp8cache" if fp8 else ""), "num_seqs": S, "new_tokens": N, "num_heads": hq, "num_kv_heads": hkv,
                       "head_dim": hd, "block_size": bs, "num_blocks": w.num_blocks,
                       "total_context": int(w.seq_lens.sum()), "cow_pairs": int(w.cow_pairs.shape[0]),
                       "kv_bytes_per_step": kv_bytes,
                       "l2": l2_note,
                       "step": ("%s (slot translation + K/V %s + decode, one call)" % (
                                    "pa_decode_append_fp8" if fp8 else "pa_decode_append",
                                    "quantizing write" if fp8 else "write") if fused else
                                ("pa_copy_blocks + " if pairs.shape[0] else "") + "pa_slot_mapping + " +
                                (("pa_write_kv_fp8 + " + ("pa_decode_fp8" if decode else "pa_varlen_fp8")) if fp8 else
                                 "pa_write_kv + " + ("pa_decode" if decode else "pa_varlen"))) +
                               ", replayed as a CUDA graph",
                       "seed": 0,
                       "parallelism": ("one GPU" if world == 1 else
                                       "%d ranks, each with its shard (length-balanced cut by sequence, own block "
                                       "pool) of a batch %d times the configuration; no data-path collective"
                                       % (world, world)),
                       "global_num_seqs": int(job_seqs)},
            "seq_per_s": seq_per_s,
            "eager_ms_per_step": eager_ms,
            "unfused_ms_per_step": unfused_ms,
            "roofline": roof,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "e2e": e2e,
        }
        if not args.no_extras:
            line["cpu_baseline"] = cpu_sample(args.workload, fp8=fp8)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
