#!/usr/bin/env python3
"""Throughput of C = ReLU(A . B) (fp16 in, fp32 accumulate, fp16 out) on GB300.

One step = one gemm_relu call over one input set of the workload (default:
M = N = K = 4096, A, B ~ N(0, 1) * 4096**-0.25, seed 2 -- the largest of the
five workloads and the square, tensor-core bound one).  Inputs rotate over enough seeded sets that
their total exceeds twice the 129 MB L2, so no step starts with its inputs
in L2.  Device timing uses CUDA events on the launching stream: K launches
back to back between one event pair (queued behind a short device-side
sleep, so the events measure the device and not Python); a second pass
with an event pair around each launch gives the per-launch min / median
reported beside it (the roofline block gives the fraction both ways: `frac`
from the back-to-back average, `frac_isolated` from the per-launch median,
which is what a serialised profile of one launch corroborates).  The other
workloads, a labelled hot-L2 figure for the skinny shape, and the CPU
oracle's rate on every workload (all cores; one core for the two small
ones) are reported in the same line.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (the slow reference arm).

Multi-GPU (torchrun): every rank runs an independent replica on its own GPU
(the product needs no exchange between GPUs); the timed region is bracketed
by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gemm_relu TFLOP/s at 1 GB300 and fraction of FP16 tensor / HBM roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure the skinny shape's target is stated against
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "schedule.h", "plan.cpp", "gemm_relu.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")


# ----------------------------------------------------------------- helpers

def code_without_comments(text: str) -> str:
    """C/C++ source with comments, blank lines and trailing blanks removed
    (string literals in these sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(read=None) -> str:
    """Hash of the kernel and launch sources, comments aside: traffic taken
    with ncu stays valid while only comments change."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, "tiled_dense_gemm_gb300", "csrc", f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(code_without_comments(text).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    cur = kernel_source_hash()
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == cur:
            return float(parts[2])
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.strip().split(", ") for r in self.out.read().splitlines() if r.strip()]
        self.out.close()
        os.unlink(self.out.name)
        return self.summarize(rows)

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        busy = []
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
                busy.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"], "samples": len(rows)}
        # "under load": samples drawing more than the median power
        thr = statistics.median(busy) if busy else 0.0
        loaded = [s for s, p in zip(sm, busy) if p >= thr] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(busy) if busy else None}


# ----------------------------------------------------------------- workloads

def workload_summary(w):
    return (f"{w.name}: gemm_relu M={w.M} N={w.N} K={w.K}, A {w.dist_a}*{w.scale_a:.4g}, "
            f"B {w.dist_b}*{w.scale_b:.4g}, seed {w.seed}, fp16 in, fp32 accumulate, ReLU, fp16 out")


def make_device_sets(w, device, min_bytes):
    import torch
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    per = 2 * (w.M * w.K + w.K * w.N)
    n = max(3, -(-min_bytes // per))
    sets = []
    for i in range(n):
        A, B = workload_inputs(w, seed_offset=i)
        sets.append((A.to(device), B.to(device),
                     torch.empty((w.M, w.N), dtype=torch.float16, device=device)))
    return sets


def time_device(w, device, steps, warmup, world):
    """Device-timed K steps; returns dict of timings (ms)."""
    import torch
    from tiled_dense_gemm_gb300 import binding
    sets = make_device_sets(w, device, 2 * L2_BYTES)
    stream = torch.cuda.current_stream(device)
    relu = True
    # warm-up (also grows any library workspace before graph capture)
    for i in range(max(warmup, 3)):
        a, b, c = sets[i % len(sets)]
        binding.gemm_relu(a, b, c, relu, stream)
    binding.check_device_error(stream)
    torch.cuda.synchronize(device)

    # The K launches run back to back between one pair of events on the
    # launching stream (an event pair around every launch would add its own
    # gaps); each launch reads the next of the rotating input sets, which
    # together exceed L2, so no launch finds its operands cached.
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    # keep the device busy while the launches are queued
    torch.cuda._sleep(int(max(4_000_000, steps * 1_000_000)))
    start.record(stream)
    for i in range(steps):
        a, b, c = sets[i % len(sets)]
        binding.gemm_relu(a, b, c, relu, stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    binding.check_device_error(stream)
    total = start.elapsed_time(end)
    # Second pass, reported beside the back-to-back figure: an event pair
    # around each launch (>= 100 launches), for the per-launch min / median.
    n_each = max(steps, 100)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_each)]
    torch.cuda.synchronize(device)
    torch.cuda._sleep(int(max(4_000_000, n_each * 1_000_000)))
    for i, (e0, e1) in enumerate(evs):
        a, b, c = sets[i % len(sets)]
        e0.record(stream)
        binding.gemm_relu(a, b, c, relu, stream)
        e1.record(stream)
    torch.cuda.synchronize(device)
    binding.check_device_error(stream)
    each = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
    # what an event pair with nothing between takes, queued the same way:
    # part of every per-launch figure above
    empty = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_each)]
    torch.cuda._sleep(int(max(4_000_000, n_each * 200_000)))
    for e0, e1 in empty:
        e0.record(stream)
        e1.record(stream)
    torch.cuda.synchronize(device)
    alone = sorted(e0.elapsed_time(e1) for e0, e1 in empty)
    return {"total_ms": total, "launch_ms": total / steps, "sets": len(sets),
            "set_bytes": 2 * (w.M * w.K + w.K * w.N),
            "per_launch_event_us": {"launches": n_each, "min": each[0] * 1e3,
                                    "median": each[len(each) // 2] * 1e3,
                                    "event_pair_alone_median": alone[len(alone) // 2] * 1e3}}


def host_call_us(w, device, calls=400):
    """Host time of one gemm_relu call (CPU timer around a run of calls
    queued behind a device-side sleep, so no call waits for the GPU):
    with the plan and tensor maps cached (the normal path), and with both
    rebuilt on every call (the same plan forced through
    GEMM_RELU_FORCE_PATH, which bypasses both caches)."""
    import torch
    from tiled_dense_gemm_gb300 import binding
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    A, B = workload_inputs(w)
    a, b = A.to(device), B.to(device)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=device)
    stream = torch.cuda.current_stream(device)
    pl = binding.plan(w.M, w.N, w.K, torch.cuda.get_device_properties(device).multi_processor_count)
    force = {(2, 64): "tiled64", (2, 128): "tiled128", (2, 256): "tiled256", (4, 256): "pair"}.get(
        (pl.path, pl.mma_n), "swap")
    out = {}
    for label, env in (("cached", None), ("rebuilt", force)):
        if env:
            os.environ["GEMM_RELU_FORCE_PATH"] = env
        try:
            for _ in range(5):
                binding.gemm_relu(a, b, c, True, stream)
            torch.cuda.synchronize(device)
            torch.cuda._sleep(int(calls * 40_000))  # keeps the device busy while the calls queue
            t0 = time.perf_counter()
            for _ in range(calls):
                binding.gemm_relu(a, b, c, True, stream)
            out[label] = (time.perf_counter() - t0) / calls * 1e6
            torch.cuda.synchronize(device)
        finally:
            os.environ.pop("GEMM_RELU_FORCE_PATH", None)
    binding.check_device_error(stream)
    out["forced_plan"] = force
    return out


def time_hot_l2(w, device, steps):
    """The same input set every launch (operands may stay in L2): a labelled
    hot-L2 figure, not the headline."""
    import torch
    from tiled_dense_gemm_gb300 import binding
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    A, B = workload_inputs(w)
    a, b = A.to(device), B.to(device)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        binding.gemm_relu(a, b, c, True, stream)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    torch.cuda._sleep(int(max(4_000_000, steps * 1_000_000)))
    start.record(stream)
    for _ in range(steps):
        binding.gemm_relu(a, b, c, True, stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    binding.check_device_error(stream)
    return start.elapsed_time(end) / steps


def soak(w, device, seconds):
    """Run the same kernel back to back (CUDA graph) for ~`seconds` so the
    clock sampler sees the GPU under this load."""
    import torch
    from tiled_dense_gemm_gb300 import binding
    sets = make_device_sets(w, device, 2 * L2_BYTES)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for a, b, c in sets[:2]:
            binding.gemm_relu(a, b, c, True, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    reps = 64
    with torch.cuda.graph(g, stream=stream):
        for i in range(reps):
            a, b, c = sets[i % len(sets)]
            binding.gemm_relu(a, b, c, True, torch.cuda.current_stream(device))
    t0 = time.time()
    n = 0
    while time.time() - t0 < seconds:
        g.replay()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize(device)
    torch.cuda.synchronize(device)
    del g, sets


def time_e2e(w, steps, warmup, device):
    """Host buffers through the C ABI: H2D copies, kernel, D2H copy, per step."""
    import torch
    from tiled_dense_gemm_gb300 import binding
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    hsets = []
    for i in range(2):
        A, B = workload_inputs(w, seed_offset=i)
        hsets.append((A.pin_memory(), B.pin_memory()))
    C = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    stream = torch.cuda.current_stream(device)
    for i in range(max(warmup, 3)):
        a, b = hsets[i % 2]
        binding.gemm_relu_host(a, b, C, True, stream, device)
    t0 = time.perf_counter()
    for i in range(steps):
        a, b = hsets[i % 2]
        binding.gemm_relu_host(a, b, C, True, stream, device)
    dt = time.perf_counter() - t0
    return dt / steps * 1e3


def cpu_oracle_rate(w, target_seconds, threads):
    """The oracle as it stands, on a row sample of the workload, repeated for
    about `target_seconds`; returns (TFLOP/s, description)."""
    import oracle
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    A, B = workload_inputs(w)
    rows = w.M
    # bound one call to ~2 GFLOP
    while rows > 16 and 2.0 * rows * w.N * w.K > 2.2e9:
        rows //= 2
    a = A[:rows].contiguous()
    oracle.gemm_relu(a[: min(rows, 8)], B, True, threads=threads)  # load + warm
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.gemm_relu(a, B, True, threads=threads)
        n += 1
        if time.perf_counter() - t0 >= target_seconds:
            break
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * n
    desc = (f"{n} x oracle on rows 0..{rows - 1} of {w.name} ({rows}x{w.N}x{w.K}), "
            f"{dt:.1f} s, {threads} threads")
    return flops / dt / 1e12, desc, dt


# ----------------------------------------------------------------- arms

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    from tiled_dense_gemm_gb300.workloads import workload_inputs
    A, B = workload_inputs(w)
    rows = w.M
    while rows > 16 and 2.0 * rows * w.N * w.K > 1.1e9:
        rows //= 2
    a = A[:rows].contiguous()
    for _ in range(args.warmup):
        oracle.gemm_relu(a, B, True, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_relu(a, B, True, threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = f"each step: the oracle on rows 0..{rows - 1} of {w.name} ({rows}x{w.N}x{w.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_summary(w), "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    from tiled_dense_gemm_gb300 import binding
    from tiled_dense_gemm_gb300.workloads import WORKLOADS

    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (
        str(uuid) if uuid is not None else str(local))
    sampler = ClockSampler(gpu_id)
    sampler.start()
    soak(w, device, args.soak)
    res = time_device(w, device, args.steps, args.warmup, world)
    clocks = sampler.stop()

    total_ms = reduce_max_over_ranks(res["total_ms"], world, device)
    avg_launch_ms = res["launch_ms"]
    flops = w.flops
    value = world * args.steps * flops / (total_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    plan = binding.plan(w.M, w.N, w.K, props.multi_processor_count).as_dict()

    def roofline_for(wl, launch_ms, pl, isolated_ms):
        """Roofline of one workload's kernel.  `frac` uses the back-to-back
        average launch time (consecutive launches overlap their set-up);
        `frac_isolated` the median of launches timed one by one, the figure
        a serialised ncu capture of one launch corroborates."""
        if wl.M <= 128 and pl["path"] == 3:
            achieved = wl.algorithmic_bytes / (launch_ms * 1e-3) / 1e9
            iso = wl.algorithmic_bytes / (isolated_ms * 1e-3) / 1e9
            peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
            return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_source": f"hbm_gbs ({peak_src})",
                    "achieved_isolated": iso, "frac_isolated": iso / peak,
                    "frac_vs_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                    "frac_isolated_vs_nominal_8tbs": iso / NOMINAL_HBM_GBS,
                    "traffic": measured_traffic(wl.name),
                    "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
                    "profile_corroborates": "frac_isolated"}
        achieved = wl.flops / (launch_ms * 1e-3) / 1e12
        iso = wl.flops / (isolated_ms * 1e-3) / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])  # fp16 dense rate == bf16
        sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_source": f"bf16_tflops burst ({peak_src}); fp16 dense rate = bf16 rate",
                "achieved_isolated": iso, "frac_isolated": iso / peak,
                "frac_vs_sustained_peak": achieved / sustained,
                "traffic": measured_traffic(wl.name), "algorithmic_flops_per_launch": wl.flops,
                "profile_corroborates": "frac_isolated"}

    roof = roofline_for(w, avg_launch_ms, plan, res["per_launch_event_us"]["median"] * 1e-3)

    others = {}
    if not args.no_extra and rank == 0:
        for name in ("c1_256", "c2_1024", "c3_4096", "c4_skinny", "c5_ragged"):
            if name == w.name:
                continue
            wo = WORKLOADS[name]
            r2 = time_device(wo, device, max(args.steps, 20), args.warmup, 1)
            ms = r2["launch_ms"]
            p2 = binding.plan(wo.M, wo.N, wo.K, props.multi_processor_count).as_dict()
            ro = roofline_for(wo, ms, p2, r2["per_launch_event_us"]["median"] * 1e-3)
            others[name] = {"workload": workload_summary(wo), "tflops": wo.flops / (ms * 1e-3) / 1e12,
                            "avg_launch_us": ms * 1e3, "roofline": ro,
                            "per_launch_event_us": r2["per_launch_event_us"],
                            "plan": {k: p2[k] for k in ("path", "mma_n", "grid", "cluster", "splits",
                                                        "sk_tiles")},
                            "steps": max(args.steps, 20)}
            if name == "c1_256":
                others[name]["host_us_per_call"] = host_call_us(wo, device)
            if name == "c4_skinny":
                hot = time_hot_l2(wo, device, max(args.steps, 20))
                others[name]["hot_l2"] = {
                    "avg_launch_us": hot * 1e3,
                    "gbs": wo.algorithmic_bytes / (hot * 1e-3) / 1e9,
                    "note": "one input set reused every launch: B may be partly L2-resident; "
                            "not the headline"}
            torch.cuda.empty_cache()

    e2e_ms = time_e2e(w, args.steps, args.warmup, device)
    e2e_ms = reduce_max_over_ranks(e2e_ms, world, device)

    cpu = None
    cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        threads = len(os.sched_getaffinity(0))
        rate, desc, _ = cpu_oracle_rate(w, args.cpu_seconds, threads)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}
        if not args.no_extra:
            # every workload on all cores, and c1 / c2 on one core (bounded
            # samples of ~2 s each; compiled with -O2, no fast-math)
            cpu_all = {"flags": "gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp"}
            for name in ("c1_256", "c2_1024", "c3_4096", "c4_skinny", "c5_ragged"):
                wo = WORKLOADS[name]
                r_all, d_all, _ = cpu_oracle_rate(wo, 2.0, threads)
                entry = {"all_cores": {"tflops": r_all, "cores": threads, "sample": d_all}}
                if name in ("c1_256", "c2_1024"):
                    r_one, d_one, _ = cpu_oracle_rate(wo, 2.0, 1)
                    entry["one_core"] = {"tflops": r_one, "cores": 1, "sample": d_one}
                cpu_all[name] = entry

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": workload_summary(w), "M": w.M, "N": w.N, "K": w.K,
                       "accumulate": "f32", "relu": True,
                       "l2": f"inputs rotate over {res['sets']} seeded sets of "
                             f"{res['set_bytes'] / 2**20:.1f} MiB (> 2x the 129 MB L2)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "plan": {k: plan[k] for k in ("path", "mma_n", "grid", "dp_tiles",
                                                     "sk_tiles", "num_stages")}},
            "roofline": roof,
            "avg_launch_us": avg_launch_ms * 1e3,
            "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 2 * (w.M * w.K + w.K * w.N),
                    "d2h_bytes_per_step": 2 * w.M * w.N,
                    "path": "gemm_relu_host (pinned host buffers, copies inside the timed region)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "cpu_oracle_by_workload": cpu_all,
            "per_launch_event_us": res["per_launch_event_us"],
            "other_workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile_launches(args, w):
    """A few launches on one input set, for an ncu capture (no timing).
    --b-layout / --dtype select a gemm_relu_ex variant (B stored (N, K),
    bfloat16 elements) on the same shape and value distribution."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from tiled_dense_gemm_gb300 import binding
    from tiled_dense_gemm_gb300.workloads import make_inputs
    device = torch.device("cuda", 0)
    dt = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    A, B = make_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.scale_a, w.dist_b, w.scale_b,
                       dtype=dt, b_layout=args.b_layout)
    a, b = A.to(device), B.to(device)
    c = torch.empty((w.M, w.N), dtype=dt, device=device)
    plain = args.b_layout == "kn" and args.dtype == "f16"
    for _ in range(args.ncu_launches):
        if plain:
            binding.gemm_relu(a, b, c, True)
        else:
            binding.gemm_relu_ex(a, b, c, True, b_layout=args.b_layout)
    binding.check_device_error()
    torch.cuda.synchronize(device)
    print(f"profile launches done: {args.ncu_launches} x {w.name} (B {args.b_layout}, {args.dtype})")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3_4096")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load for clock sampling")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads' side measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--ncu-launches", type=int, default=0,
                    help="profiling mode: run only this many launches of the workload and exit")
    ap.add_argument("--b-layout", choices=["kn", "nk"], default="kn",
                    help="profiling mode: B stored (K, N) or (N, K) (gemm_relu_ex)")
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="f16",
                    help="profiling mode: element type (gemm_relu_ex)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from tiled_dense_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.ncu_launches:
        return run_profile_launches(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
