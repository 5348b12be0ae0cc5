"""Benchmark of the paged-KV hot path on the 64-sequence GQA decode batch.

One step = the generation step of the batch through the C ABI:
pa_slot_mapping (the new token of each sequence) -> pa_write_kv (its K/V
row) -> pa_decode (tensor-core kernel + split merge).  Inputs are resident
in HBM; two copies of the K/V pool (2 x 0.55 GB, each larger than the
129 MB L2) alternate between steps so no step reads a pool the previous one
left in L2.

Prints ONE JSON line (rank 0).  `value` is algorithmic K/V bytes read per
step over the device time of the step (GB/s); `roofline` is the decode
kernels' own time against the measured HBM copy bandwidth; `e2e` is the same
metric with each step's inputs copied from pinned host memory and the output
copied back inside the timed region; `cpu_baseline` is the CPU oracle on a
bounded sample.  `--impl reference` times that oracle alone as the
reference arm.

Multi-GPU (torchrun): every rank runs its own replica of the batch (the
sequences are independent, no data-path collective); `value` sums all ranks'
bytes over the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attention KV GB/s (fraction of HBM peak) and sequences/s, 1×GB300")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rotate", action="store_true", help="one pool copy (for profiling)")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, clocks and cpu_baseline")
    ap.add_argument("--num-seqs", type=int, default=64)
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def traffic_record(kernel_file):
    """DRAM bytes per launch of the decode kernel from a committed ncu
    summary, if it was taken on the current kernel source."""
    src = os.path.join(ROOT, "paged_kv_cache_116_gb300", "csrc", kernel_file)
    path = os.path.join(ROOT, "profiles", "decode_tc_gqa64_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("source_sha256") == sha:
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _oracle_batch(num_seqs):
    """The first num_seqs sequences of the batch (the same length stream),
    values drawn on the host, written into an oracle-side pool."""
    import numpy as np

    import oracle
    from paged_kv_cache_116_gb300 import workloads as W

    w = W.gqa_decode_batch(num_seqs=num_seqs)
    kc = np.full((w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), 0x7FC0, dtype=np.uint16)
    vc = kc.copy()
    s = oracle.slot_mapping(w.pre_block_tables, w.pre_seq_idx, w.pre_pos, w.block_size)
    oracle.write_kv(W.raw_numpy(w.pre_k), W.raw_numpy(w.pre_v), s, kc, vc)
    s = oracle.slot_mapping(w.block_tables, w.new_seq_idx, w.new_pos, w.block_size)
    oracle.write_kv(W.raw_numpy(w.new_k), W.raw_numpy(w.new_v), s, kc, vc)
    return w, kc, vc, W.raw_numpy(w.q)


def cpu_baseline(total_seqs, sample=8, budget_s=10.0):
    """The oracle (as it stands) on a bounded sample: the first `sample`
    sequences of the batch, repeated for about budget_s seconds."""
    import oracle

    w, kc, vc, q = _oracle_batch(sample)
    per_tok = w.num_kv_heads * w.head_dim * 2 * w.elt
    repeats, t = 0, time.perf_counter()
    while True:
        oracle.decode_attention(q, kc, vc, w.block_tables, w.seq_lens, w.scale, w.dtype)
        repeats += 1
        el = time.perf_counter() - t
        if el >= budget_s:
            break
    return {"value": int(w.seq_lens.sum()) * per_tok * repeats / el / 1e9, "unit": "GB/s",
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": "first %d of %d sequences (%d tokens) x %d, fp64 C oracle with OpenMP, %.1f s" % (
                sample, total_seqs, int(w.seq_lens.sum()), repeats, el),
            "seq_per_s": sample * repeats / el}


def run_reference(args, rank):
    """Reference arm: the CPU oracle on the first 8 sequences of the batch
    per step (rank 0 only)."""
    if rank != 0:
        return
    import oracle

    sample = 8
    w, kc, vc, q = _oracle_batch(sample)
    step_bytes = int(w.seq_lens.sum()) * w.num_kv_heads * w.head_dim * 2 * w.elt
    for _ in range(args.warmup):
        oracle.decode_attention(q, kc, vc, w.block_tables, w.seq_lens, w.scale, w.dtype)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_attention(q, kc, vc, w.block_tables, w.seq_lens, w.scale, w.dtype)
    dt = time.perf_counter() - t
    value = step_bytes * args.steps / dt / 1e9
    desc = "first %d of %d sequences per step, fp64 C oracle with OpenMP" % (sample, args.num_seqs)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gqa_decode_bf16_64seq", "num_seqs": args.num_seqs, "sample_seqs": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
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

    __graft_entry__.build() if rank == 0 or world == 1 else None
    if world > 1:
        dist.barrier()
    import paged_kv_cache_116_gb300 as pa
    from paged_kv_cache_116_gb300 import workloads as W

    w = W.gqa_decode_batch(num_seqs=args.num_seqs, device=dev)
    S, hq, hkv, hd, bs = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    max_ctx = int(w.seq_lens.max())
    kv_bytes = w.kv_bytes_read()
    # algorithmic bytes of the decode: K/V once per KV head + q + out + tables + lengths
    alg_bytes = kv_bytes + 2 * S * hq * hd * w.elt + int(sum((L + bs - 1) // bs for L in w.seq_lens)) * 4 + S * 4

    # resident pools (two copies, alternated), filled through the library
    copies = 1 if args.no_rotate else 2
    pools = []
    for c in range(copies):
        kc = torch.full((w.num_blocks, bs, hkv, hd), float("nan"), dtype=torch.bfloat16, device=dev)
        vc = torch.full_like(kc, float("nan"))
        slots = pa.pa_slot_mapping(torch.from_numpy(w.pre_block_tables).to(dev), torch.from_numpy(w.pre_seq_idx).to(dev),
                                   torch.from_numpy(w.pre_pos).to(dev), bs)
        pa.pa_write_kv(w.pre_k, w.pre_v, slots, kc, vc)
        pools.append((kc, vc))
    del w.pre_k, w.pre_v
    bt = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    seq_idx = torch.from_numpy(w.new_seq_idx).to(dev)
    pos = torch.from_numpy(w.new_pos).to(dev)
    q, new_k, new_v = w.q.contiguous(), w.new_k.contiguous(), w.new_v.contiguous()
    out = torch.empty_like(q)
    slot_buf = torch.empty(S, dtype=torch.int64, device=dev)
    ws_bytes = pa.pa_decode_workspace_size(S, hq, hkv, hd, bs, max_ctx, torch.bfloat16)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    def step(i):
        """One generation step through the C ABI on the current stream."""
        kc, vc = pools[i % copies]
        st = torch.cuda.current_stream()
        pa.pa_slot_mapping(bt, seq_idx, pos, bs, slot_out=slot_buf, stream=st)
        pa.pa_write_kv(new_k, new_v, slot_buf, kc, vc, stream=st)
        pa.pa_decode(out, q, kc, vc, bt, lens, max_ctx, w.scale, workspace=ws, stream=st)

    def decode_only(i):
        kc, vc = pools[i % copies]
        pa.pa_decode(out, q, kc, vc, bt, lens, max_ctx, w.scale, workspace=ws, stream=torch.cuda.current_stream())

    launches_per_step = 3  # slot mapping, write, decode

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()

    # The step is captured once per pool copy into CUDA graphs (what a serving
    # loop replays); the same C-ABI calls run eagerly give `eager`.
    def capture(fn):
        gs = []
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn(c)
            gs.append(g)
        return gs

    step_graphs = capture(step)
    dec_graphs = capture(decode_only)
    for i in range(max(args.warmup, 3)):
        step_graphs[i % copies].replay()
        dec_graphs[i % copies].replay()
    torch.cuda.synchronize()

    def timed(fn_i):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        a.record()
        for i in range(args.steps):
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
    ms = timed(lambda i: step_graphs[i % copies].replay())
    clk = clocks.stop() if rank == 0 and not args.no_extras else None
    dec_ms = timed(lambda i: dec_graphs[i % copies].replay()) / args.steps
    eager_ms = timed(step) / args.steps

    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / args.steps
    value = kv_bytes * world * args.steps / (ms / 1e3) / 1e9
    seq_per_s = S * world * args.steps / (ms / 1e3)

    # e2e: each step's inputs from pinned host memory, the step, the output
    # back to pinned host memory -- all inside the timed region (captured as
    # one graph per pool copy, like the device-only step)
    e2e = None
    if not args.no_extras:
        h_q = q.cpu().pin_memory()
        h_k, h_v = new_k.cpu().pin_memory(), new_v.cpu().pin_memory()
        h_bt, h_lens = bt.cpu().pin_memory(), lens.cpu().pin_memory()
        h_seq, h_pos = seq_idx.cpu().pin_memory(), pos.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(new_k), torch.empty_like(new_v)
        d_bt, d_lens, d_seq, d_pos = torch.empty_like(bt), torch.empty_like(lens), torch.empty_like(seq_idx), \
            torch.empty_like(pos)
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_bt, h_lens, h_seq, h_pos))
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step(i):
            kc, vc = pools[i % copies]
            st = torch.cuda.current_stream()
            for d, h in ((d_q, h_q), (d_k, h_k), (d_v, h_v), (d_bt, h_bt), (d_lens, h_lens), (d_seq, h_seq),
                         (d_pos, h_pos)):
                d.copy_(h, non_blocking=True)
            pa.pa_slot_mapping(d_bt, d_seq, d_pos, bs, slot_out=slot_buf, stream=st)
            pa.pa_write_kv(d_k, d_v, slot_buf, kc, vc, stream=st)
            pa.pa_decode(out, d_q, kc, vc, d_bt, d_lens, max_ctx, w.scale, workspace=ws, stream=st)
            h_out.copy_(out, non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_graphs = capture(e2e_step)
        for i in range(3):
            e2e_graphs[i % copies].replay()
        torch.cuda.synchronize()
        e_ms = timed(lambda i: e2e_graphs[i % copies].replay())
        if world > 1:
            t = torch.tensor([e_ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_ms = float(t.item())
        e2e = {"value": kv_bytes * world * args.steps / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "how": "pinned-host inputs -> H2D copies -> pa_slot_mapping/pa_write_kv/pa_decode -> D2H output, "
                      "replayed as a CUDA graph per step"}

    peaks, kind = measured_peaks()
    dec_avg = dec_ms
    achieved = alg_bytes / (dec_avg / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": "decode_tc_kernel (one pa_decode call, split merge included)",
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "peak_kind": kind, "traffic": traffic_record("pa_decode_tc.cu"), "algorithmic_bytes": alg_bytes,
            "decode_us": dec_avg * 1e3}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "num_seqs": S, "num_heads": hq, "num_kv_heads": hkv, "head_dim": hd,
                       "block_size": bs, "num_blocks": w.num_blocks, "total_context": int(w.seq_lens.sum()),
                       "kv_bytes_per_step": kv_bytes, "l2": "inputs larger than L2: %d pool copies of %.2f GB "
                       "alternate between steps" % (copies, 2 * pools[0][0].numel() * 2 / 1e9),
                       "step": "pa_slot_mapping + pa_write_kv + pa_decode, replayed as a CUDA graph",
                       "seed": 0},
            "seq_per_s": seq_per_s,
            "eager_ms_per_step": eager_ms,
            "roofline": roof,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "e2e": e2e,
        }
        if not args.no_extras:
            line["cpu_baseline"] = cpu_baseline(S)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
