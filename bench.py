#!/usr/bin/env python3
"""Benchmark: paged decode attention over a paged KV cache on GB300.

One step = one decode step of the whole hot path for the batch: host slot
assignment with copy-on-write (pkv_prepare_append), the step's table/slot
uploads, the block copy, and for every layer the append of the new token's K/V
followed by paged decode attention (split-KV, fused combine).

Default workload: 7B shape (32 layers, 32 heads x 128, fp16 KV), block size 16,
batch 32 with context lengths U[256, 2048], pool 1.3x the blocks needed with
shuffled block ids. Each layer's KV (~0.5 GB) is far larger than the 129 MB L2,
so no flush is needed between steps.

Prints ONE JSON line (rank 0). ``value`` is KV GB/s: algorithmic K+V bytes read by
the attention launches of the timed steps / device time of those steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--config 2|3|4|5] [--layout NHD|HND] [--block-size B]
"""
from __future__ import annotations

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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak); seq·steps/s at 7B shape"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILES = {"f16": os.path.join(ROOT, "profiles", "decode_attention_traffic.txt"),
                 "e4m3": os.path.join(ROOT, "profiles", "decode_attention_e4m3_traffic.txt")}
KERNEL_SRC = os.path.join(ROOT, "paged_kv_cache_88_gb300", "csrc", "decode_attention.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--layout", default="HND", choices=["NHD", "HND"])
    ap.add_argument("--block-size", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (profiling captures only)")
    ap.add_argument("--kv-dtype", default="f16", choices=["f16", "e4m3"])
    ap.add_argument("--swap", action="store_true", help="measure swap-out / swap-in of one sequence instead")
    ap.add_argument("--prefill", type=int, default=0, metavar="CHUNK",
                    help="measure causal prefill of CHUNK-token chunks over the workload's cache instead")
    ap.add_argument("--no-cascade", action="store_true",
                    help="attend shared prefixes per sequence (no prefix pass)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def device_code_hash() -> str:
    """Hash of the attention kernel's device code: its .cu up to the host-side section, plus the
    device headers it includes (ptx.cuh, quant.cuh)."""
    text = open(KERNEL_SRC).read()
    cut = text.find("// ------------------------------------------------------------------ host side")
    h = hashlib.sha256(text[:cut].encode())
    for hdr in ("ptx.cuh", "quant.cuh"):
        h.update(open(os.path.join(os.path.dirname(KERNEL_SRC), hdr)).read().encode())
    return h.hexdigest()[:16]


def kernel_traffic(bytes_per_launch: float, kv_dtype: str = "f16"):
    """DRAM bytes per launch from the committed ncu summary of the kernel variant for
    kv_dtype, scaled to this launch's KV bytes.

    The summary holds dram__bytes_read.sum + dram__bytes_write.sum of one captured
    launch and that launch's algorithmic KV bytes; traffic grows in proportion to
    the tokens read, so it is scaled by the ratio. None if the kernel source
    changed since the capture (the hash of its device code is recorded in the summary).
    """
    try:
        text = open(TRAFFIC_FILES[kv_dtype]).read()
        vals = {}
        for line in text.splitlines():
            if ":" in line and not line.lstrip().startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("device_code_sha256") != device_code_hash():
            return None
        return float(vals["dram_bytes_per_launch"]) * bytes_per_launch / float(vals["algorithmic_bytes_at_capture"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def aggregate_ranks(ms: float, kv_bytes: float, seq_steps: float, device=None):
    """Whole-job figures over the ranks: the slowest rank's time, the sum of the work.

    Ranks are independent replicas (each its own pool and batch): the only
    communication is this reduction of the measurements.
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, kv_bytes, seq_steps
    t = torch.tensor([ms, kv_bytes, seq_steps], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return mx[0].item(), sm[1].item(), sm[2].item()


def rank_seed(config: int, rank: int) -> int:
    """Seed of rank ``rank``'s batch (rank 0 runs the single-GPU workload)."""
    return 1000 + config + 7919 * rank


def bench_total_steps(args) -> int:
    """Decode steps the pool is sized for: warm-up (eager and graph), timed, end-to-end, spare."""
    e2e_steps = 0 if args.no_e2e else args.steps
    return 3 * args.warmup + args.steps + e2e_steps + 4


def make_bench_workload(args, extra_steps: int):
    import workloads as wl
    w = wl.make_workload(args.config, decode_steps=extra_steps, layout=args.layout, block_size=args.block_size,
                         num_layers=args.layers, kv_dtype=args.kv_dtype)
    return w


def cpu_baseline_oracle(w, k_layer, v_layer, tables, lens, seconds: float, k_scale=None, v_scale=None):
    """The oracle on one layer, repeated for ~``seconds``: the C float64 oracle (OpenMP over
    (sequence, head)) for an fp16 cache; the NumPy E4M3 oracle on one sequence for a quantised one."""
    import numpy as np
    from oracle import ref_attn_c as rc
    if w.kv_dtype == "e4m3":
        from oracle import fp8
        q = np.random.default_rng(0).standard_normal((1, w.num_heads, w.head_dim)).astype(np.float16)
        t0 = time.perf_counter()
        passes = 0
        while True:
            s = passes % w.num_seqs
            fp8.decode_attention(q, k_layer, v_layer, k_scale, v_scale, tables[s:s + 1], lens[s:s + 1], w.block_size,
                                 layout=w.layout)
            passes += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        nbytes = sum(int(lens[i % w.num_seqs]) for i in range(passes)) * w.kv_bytes_per_token_layer
        return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{passes} sequence(s) of one layer, NumPy E4M3 oracle (dequantise, float64), {el:.1f} s"}
    rng = np.random.default_rng(0)
    q = rng.standard_normal((w.num_seqs, w.num_heads, w.head_dim)).astype(np.float16)
    lens64 = np.asarray(lens, dtype=np.int64)
    bytes_per = int(lens64.sum()) * w.kv_bytes_per_token_layer
    cores = rc.max_threads()
    # one core first (the thread count a call sets stays for the next call), on the
    # batch's first eighth of sequences
    sub = max(1, w.num_seqs // 8)
    t0 = time.perf_counter()
    p1 = 0
    while True:
        rc.decode_attention(q[:sub], k_layer, v_layer, tables[:sub], lens[:sub], w.block_size, w.layout,
                            num_threads=1)
        p1 += 1
        el1 = time.perf_counter() - t0
        if el1 >= seconds / 4 or p1 >= 64:
            break
    one_core = int(lens64[:sub].sum()) * w.kv_bytes_per_token_layer * p1 / el1 / 1e9
    t0 = time.perf_counter()
    passes = 0
    while True:
        rc.decode_attention(q, k_layer, v_layer, tables, lens, w.block_size, w.layout, num_threads=cores)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds or passes >= 64:
            break
    return {"value": bytes_per * passes / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "one_core_value": one_core, "cpu_model": cpu_model(),
            "sample": f"{passes} pass(es) of one layer ({w.num_seqs} seqs x {w.num_heads} heads, "
                      f"{int(np.sum(lens))} tokens) of the same workload, fp64 C oracle, {el:.1f} s; one core: "
                      f"{p1} pass(es) of its first {sub} seqs, {el1:.1f} s"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    import platform
    import subprocess
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in outp.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def run_reference(args):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import workloads as wl
    from oracle import ref_alloc as ra
    from oracle import ref_attn_c as rc
    w = make_bench_workload(args, bench_total_steps(args))   # the GPU arm's workload, pool size included
    op = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    tables = np.asarray([ra.admit(op, int(t), w.block_size, w.max_blocks) for t in w.context_lens], dtype=np.int32)
    lens = np.asarray(w.context_lens, dtype=np.int32)
    shape = wl.pool_shape(w)[1:]
    k = wl.normal_fp16(w.seed, (100, 0), shape)
    v = wl.normal_fp16(w.seed, (101, 0), shape)
    q = wl.normal_fp16(w.seed, (200, 0), (w.num_seqs, w.num_heads, w.head_dim))
    bytes_per = int(lens.astype(np.int64).sum()) * w.kv_bytes_per_token_layer
    # every host core the process may use, whatever OMP_NUM_THREADS says (torchrun sets 1)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    for _ in range(args.warmup):
        rc.decode_attention(q, k, v, tables, lens, w.block_size, w.layout, num_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rc.decode_attention(q, k, v, tables, lens, w.block_size, w.layout, num_threads=cores)
    el = time.perf_counter() - t0
    val = bytes_per * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), step="one layer of the workload (bounded sample)"),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step = one layer of {w.num_seqs} seqs x {w.num_heads} heads, "
                                   f"{int(lens.sum())} tokens, fp64 C oracle"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_cow(eng, w, dev, peak):
    """The copy-on-write the workload's first write after the fork needed (pkv_copy_blocks over
    all layers), re-timed after the decode steps: the same source blocks copied into freshly
    allocated ones, so the cache the steps read is untouched. Also the blocks the pool holds
    against the blocks an unshared layout of the same sequences would need."""
    import numpy as np
    import torch
    pairs = np.concatenate(eng.cow_log)
    st = eng.pool.stats()
    unshared = int(sum(-(-int(t) // w.block_size) for t in eng.lens[:w.num_seqs]))
    n = min(len(pairs), int(st["free_blocks"]))
    res = {"pairs": int(len(pairs)), "layers": w.num_layers, "blocks_used": int(st["used_blocks"]),
           "blocks_unshared": unshared}
    if n == 0:
        return res
    fresh = eng.pool.alloc(n)
    pd = torch.tensor(np.stack([pairs[:n, 0], np.asarray(fresh, dtype=np.int32)], 1), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    times = []
    for it in range(13):
        ev[0].record(stream)
        eng.pool.copy_blocks(pd, status=eng.status, stream=stream)
        ev[1].record(stream)
        torch.cuda.synchronize()
        if it >= 3:
            times.append(ev[0].elapsed_time(ev[1]))
    eng.pool.free(fresh)
    ms = float(np.median(times))
    per_block = w.num_layers * w.block_size * w.kv_bytes_per_token_layer   # K and V of a block, all layers
    copied = n * per_block
    # distinct bytes: each source block read once (forked sequences share one source), every copy written
    distinct = (len(np.unique(pairs[:n, 0])) + n) * per_block
    res.update({"timed_pairs": n, "distinct_src_blocks": int(len(np.unique(pairs[:n, 0]))),
                "bytes_copied": int(copied), "ms": ms,
                "gbps_distinct": distinct / (ms / 1e3) / 1e9,
                "frac_distinct_of_hbm_peak": distinct / (ms / 1e3) / 1e9 / peak})
    return res


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)      # before the process group, so NCCL binds this rank's GPU
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from paged_kv_cache_88_gb300.engine import DecodeEngine
    import paged_kv_cache_88_gb300 as pkv

    e2e_steps = 0 if args.no_e2e else args.steps
    total_steps = bench_total_steps(args)
    w = make_bench_workload(args, total_steps)
    if world > 1:                         # weak scaling: each rank serves its own batch
        import workloads as wl
        w = wl.make_workload(args.config, decode_steps=total_steps, layout=args.layout,
                             block_size=args.block_size, num_layers=args.layers, seed=rank_seed(args.config, rank),
                             kv_dtype=args.kv_dtype)
    eng = DecodeEngine(w, device=str(dev), fill="torch", cascade=not args.no_cascade)
    eng.run_script(values="torch")
    torch.cuda.synchronize()
    L, S, H, D = w.num_layers, w.num_seqs, w.num_heads, w.head_dim
    q, kn, vn = eng.step_inputs(0, "torch")
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- warm-up (eager), then the step is captured once as a CUDA graph
    for _ in range(args.warmup):
        eng.step(q, kn, vn, out, stream)
    barrier()
    eng.capture(q, kn, vn, out)
    for _ in range(args.warmup):
        eng.step_graph(stream)
    barrier()
    if eng.device_status() != 0:
        raise RuntimeError(f"device status {eng.device_status():#x} after warm-up")

    # ---- timed region: K decode steps, inputs resident in HBM
    step_bytes = []
    step_unique = []
    launches = 0
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        barrier()
        t_start.record(stream)
        h0 = time.perf_counter()
        for _ in range(args.steps):
            n_slots, n_pairs = eng.step_graph(stream)
            step_bytes.append(eng.kv_bytes_per_layer())
            step_unique.append(eng.unique_kv_bytes_per_layer())
            launches += (L if eng.fused else 2 * L) + (L if eng.plan_groups else 0) + (1 if n_pairs else 0)
        host_ms = (time.perf_counter() - h0) * 1e3 / args.steps
        t_end.record(stream)
        barrier()
        # roofline pass: the dominant kernel alone, back to back over the
        # step's layers (same launches as in a step, without the appends), CUDA
        # events on the launching stream at both ends
        n_attn = max(2, args.steps // 2) * L
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(n_attn):
            eng.attention(i % L, q, out, stream, early=i > 0)
        a1.record(stream)
        barrier()
        # serialised pass: each launch alone, as when the kernel before it on the stream is not
        # one of ours (no early start, no programmatic overlap): a small torch kernel runs
        # between launches, outside each launch's pair of CUDA events
        n_ser = max(2, args.steps // 8) * L
        gap = torch.zeros(1024, dtype=torch.float32, device=dev)
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ser)]
        for i in range(n_ser):
            gap.add_(1.0)
            sev[i][0].record(stream)
            eng.attention(i % L, q, out, stream, early=False)
            sev[i][1].record(stream)
        barrier()
    clocks = clk.summary()
    ms = t_start.elapsed_time(t_end)
    attn_ms_total = a0.elapsed_time(a1)
    attn_launch_bytes = eng.kv_bytes_per_layer()
    cascading = bool(eng.plan_groups)
    if cascading:   # the layer's attention is the prefix pass + the private pass: count distinct bytes
        attn_launch_bytes = eng.unique_kv_bytes_per_layer()
    status = eng.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status:#x} in the timed region")

    kv_bytes = sum(step_bytes) * L
    ms_job, bytes_job, seqsteps_job = aggregate_ranks(ms, float(kv_bytes), float(S * args.steps), dev)
    value = bytes_job / (ms_job / 1e3) / 1e9
    seq_steps = seqsteps_job / (ms_job / 1e3)

    # roofline of the dominant kernel (decode attention): algorithmic bytes / average launch time
    extra = 2 * S * H * D * 2 + S * 4 + int(np.sum(-(-eng.lens // w.block_size))) * 4
    mean_launch_ms = attn_ms_total / n_attn
    achieved = (attn_launch_bytes + extra) / (mean_launch_ms / 1e3) / 1e9
    serial_ms = float(np.mean([a.elapsed_time(b) for a, b in sev]))
    serial_achieved = (attn_launch_bytes + extra) / (serial_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = None if cascading else kernel_traffic(attn_launch_bytes + extra, w.kv_dtype)

    # ---- end to end through the public API: inputs from pinned host memory, output read back.
    # A serving loop overlaps the transfers with the steps: a copy stream brings step n+1's
    # inputs into a device staging buffer while step n runs and takes step n's output back
    # from another; the compute stream only adds two device-to-device copies per step.
    e2e = None
    if e2e_steps:
        hq = q.cpu().pin_memory()
        hk = kn.cpu().pin_memory()
        hv = vn.cpu().pin_memory()
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        stage_in = [tuple(torch.empty_like(t) for t in (q, kn, vn)) for _ in range(2)]
        stage_out = [torch.empty_like(out) for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(2)]     # step's inputs staged
        ev_free = [torch.cuda.Event() for _ in range(2)]   # staging buffer read by the step
        ev_out = [torch.cuda.Event() for _ in range(2)]    # step's output staged
        copy = torch.cuda.Stream()

        def h2d(n):
            b = n % 2
            with torch.cuda.stream(copy):
                if n >= 2:
                    copy.wait_event(ev_free[b])
                for dst, src in zip(stage_in[b], (hq, hk, hv)):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(copy)

        e_bytes = 0
        barrier()
        copy.wait_stream(stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy.wait_event(e0)
        h2d(0)
        for n in range(e2e_steps):
            b = n % 2
            if n + 1 < e2e_steps:
                h2d(n + 1)
            stream.wait_event(ev_in[b])
            with torch.cuda.stream(stream):
                for dst, src in zip((q, kn, vn), stage_in[b]):
                    dst.copy_(src, non_blocking=True)
            ev_free[b].record(stream)
            eng.step_graph(stream)
            e_bytes += eng.kv_bytes_per_layer() * L
            with torch.cuda.stream(stream):
                stage_out[b].copy_(out, non_blocking=True)
            ev_out[b].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(ev_out[b])
                hout[b].copy_(stage_out[b], non_blocking=True)
        stream.wait_stream(copy)
        e1.record(stream)
        barrier()
        e_ms = e0.elapsed_time(e1)
        h2d = 3 * q.numel() * 2 + eng.tables.size * 4 + S * 4 + S * 8
        e2e = {"value": e_bytes / (e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(out.numel() * 2), "ms_per_step": e_ms / e2e_steps}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kl = eng.k_pool[0].cpu().numpy()
        vl = eng.v_pool[0].cpu().numpy()
        ks = eng.k_scale[0].cpu().numpy() if eng.k_scale is not None else None
        vs = eng.v_scale[0].cpu().numpy() if eng.v_scale is not None else None
        cpu = cpu_baseline_oracle(w, kl, vl, eng.tables.copy(), eng.lens.copy(), args.cpu_seconds, ks, vs)

    info = pkv.decode_launch_info(S, D, w.kv_dtype)
    kname = f"decode_attention_kernel<{D}{', E4M3' if w.kv_dtype == 'e4m3' else ''}>"
    cow = measure_cow(eng, w, dev, peak) if eng.cow_log else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_job / args.steps, "host_ms_per_step": host_ms,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if w.kv_dtype == "f16" else "e4m3",
            "accumulate": "f32", "data": "synthetic",
            "config": dict(w.describe(), l2="inputs larger than L2 (each layer's KV >> 129 MB), no flush",
                           parallelism="replicas" if world > 1 else "single",
                           mean_context_timed=float(np.mean(step_bytes)) / w.kv_bytes_per_token_layer / S,
                           step=("decode step as one CUDA graph: per layer the shared-prefix pass, then one "
                                 "fused append+attention launch over the private rest" if cascading else
                                 "decode step as one CUDA graph: per layer one fused append+attention launch"
                                 if eng.fused else
                                 "decode step as one CUDA graph: per layer one append launch (quantising for "
                                 "an E4M3 cache), then one attention launch")),
            "seq_steps_per_s": seq_steps,
            "frac_of_hbm_peak": value / peak,
            **({"unique_gbps": value * sum(step_unique) / sum(step_bytes),
                "frac_unique_of_hbm_peak": value * sum(step_unique) / sum(step_bytes) / peak,
                "cascade": {"groups": int(eng.plan_groups), "splits": int(eng.plan_splits),
                            "prefix_tokens": int(eng.plan_prefix)}} if cascading else {}),
            **({"cow": cow} if cow else {}),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "kernel": (f"prefix pass + {kname} (distinct KV bytes)" if cascading else kname),
                         "launches": n_attn,
                         "mean_launch_us": 1e3 * mean_launch_ms, "bytes_per_launch": attn_launch_bytes + extra,
                         "grid_ctas": info["grid_ctas"], "ctas_per_sm": info["ctas_per_sm"],
                         "timing": "back to back over the step's layers, each launch flagged to start early "
                                   "behind the previous one (CUDA events around the whole pass)",
                         "serial": {"achieved": serial_achieved, "frac": serial_achieved / peak,
                                    "mean_launch_us": 1e3 * serial_ms, "launches": n_ser,
                                    "timing": "each launch alone: no early start, a torch kernel between "
                                              "launches, CUDA events around each launch"}},
            "clocks": clocks,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_swap(args):
    """Swap-out / swap-in of the longest sequence of the workload (all layers) through pinned host memory."""
    import torch
    from paged_kv_cache_88_gb300.engine import DecodeEngine
    w = make_bench_workload(args, 8)
    eng = DecodeEngine(w, fill="torch")
    eng.run_script(values="torch")
    s = int(np.argmax(eng.lens))
    n = -(-int(eng.lens[s]) // w.block_size)
    bpb = eng.pool.swap_bytes_per_block()
    host = torch.empty(n * bpb, dtype=torch.uint8).pin_memory()
    staging = torch.empty(n * bpb, dtype=torch.uint8, device="cuda")
    blocks = torch.tensor(eng.tables[s, :n], dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    # staged: gather into device memory, one copy to pinned host (and back, then scatter);
    # direct: the kernels write / read the pinned host buffer themselves
    times = {"gather": [], "d2h": [], "h2d": [], "scatter": [], "gather_direct": [], "scatter_direct": []}
    for it in range(args.warmup + args.steps):
        ev[0].record(st)
        eng.pool.gather_blocks(blocks, staging, stream=st)
        ev[1].record(st)
        host.copy_(staging, non_blocking=True)
        ev[2].record(st)
        staging.copy_(host, non_blocking=True)
        ev[3].record(st)
        eng.pool.scatter_blocks(blocks, staging, stream=st)
        ev[4].record(st)
        eng.pool.gather_blocks(blocks, host, stream=st)
        ev[5].record(st)
        eng.pool.scatter_blocks(blocks, host, stream=st)
        ev[6].record(st)
        torch.cuda.synchronize()
        if it >= args.warmup:
            for i, k in enumerate(times):
                times[k].append(ev[i].elapsed_time(ev[i + 1]))
    nbytes = n * bpb
    med = {k: statistics.median(v) for k, v in times.items()}
    res = {k: nbytes / (v / 1e3) / 1e9 for k, v in med.items()}
    print(json.dumps({"metric": "swap GB/s (one sequence, all layers)", "unit": "GB/s", "bytes": nbytes,
                      "blocks": n, "config": w.describe(), **{f"{k}_gbps": v for k, v in res.items()},
                      "swap_out_ms": med["gather"] + med["d2h"], "swap_in_ms": med["h2d"] + med["scatter"],
                      "swap_out_direct_ms": med["gather_direct"], "swap_in_direct_ms": med["scatter_direct"]}))


def run_prefill(args):
    """Causal prefill of the last CHUNK tokens of every sequence over its cache (tensor cores)."""
    import torch
    from paged_kv_cache_88_gb300.engine import DecodeEngine
    w = make_bench_workload(args, 8)
    eng = DecodeEngine(w, fill="torch")
    eng.run_script(values="torch")
    L, S, H, D = w.num_layers, w.num_seqs, w.num_heads, w.head_dim
    chunks = np.minimum(eng.lens, args.prefill).astype(np.int64)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    total = int(q_start[-1])
    q = torch.randn((total, H, D), device="cuda", dtype=torch.float16)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qs = torch.from_numpy(q_start).cuda()
    st = torch.cuda.current_stream()
    # causal work: query i of a chunk of C over T tokens sees T - C + i + 1 keys; 4 D flops per (query, key, head)
    keys = sum(int(np.sum(np.arange(int(T) - int(C) + 1, int(T) + 1))) for T, C in zip(eng.lens, chunks))
    flops = 4.0 * D * H * keys
    def one(layer):
        eng.pool.prefill_attention(layer, q, qs, int(chunks.max()), eng.tables_d, eng.lens_d, out, status, stream=st)
    for i in range(args.warmup):
        one(i % L)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(args.steps):
        one(i % L)
    e1.record(st)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x}")
    ms = e0.elapsed_time(e1) / args.steps
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("bf16_tflops", 1957.5) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    tf = flops / (ms / 1e3) / 1e12
    print(json.dumps({"metric": "paged prefill attention TFLOP/s (causal, fp16, tensor cores)", "value": tf,
                      "unit": "TFLOP/s", "ms_per_layer": ms, "flops_per_layer": flops, "chunk": args.prefill,
                      "queries": total, "config": w.describe(),
                      "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                                   "frac": tf / peak, "peak_source": "measured bf16 (fp16 runs at the same rate)"}}))


def main():
    args = parse_args()
    if args.prefill:
        run_prefill(args)
        return
    if args.swap:
        run_swap(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
