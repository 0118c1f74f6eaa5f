"""Benchmark of the clipped-AdamW optimizer step with resumable checkpoints.

One step = one pass of the optimizer path over one batch of synthetic input:
the global-norm reduction, the host bias-correction scalars and the fused
clip+AdamW kernel, launched as the library launches them (the fused kernel a
programmatic dependent of the norm).  `value` is params/s over K such steps
with the inputs (w, g, m, v: 1.77 GB for the 110M list, larger than L2)
resident in HBM.  The checkpoint (device pack, side-stream copy into pinned
host memory, atomic tmp-then-rename write of step_NNNNNN.bin) runs every 100
steps in the pages' cadence: one checkpoint is measured after the timed
steps and 1/100 of it is charged per step in `whole_path`.  Also reported:
per-kernel times from a second region with an event between the kernels,
the dominant kernel's roofline, `e2e` (the gradient copied from pinned host
memory and the norm read back every step), per-config objects for the flat
2^30 (1B), 12.8M and 65,536 states, and the CPU oracle beside each.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead; --sweep prints per-size kernel
rates (flat 2^20 .. 2^30) instead of the bench line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--ckpt-every C] [--impl ours|reference] [--sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "clip+AdamW params/sec and achieved HBM GB/s vs ~8 TB/s peak, 1 GB300"
UNIT = "params/s"
STEP_BYTES = 28      # fused kernel: read w, g, m, v; write w, m, v (float32)
NORM_BYTES = 4       # norm kernel: read g
PACK_BYTES = 24      # pack kernel: read w, m, v; write the staging image
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s HBM3e figure the metric is quoted against
# the source files each kernel is compiled from (its traffic record is tied
# to their contents)
KERNEL_SOURCES = {"k_clip_adamw": ("step.cu", "adamw_dev.cuh", "common.cuh", "internal.h"),
                  "k_grad_norm": ("norm.cu", "norm_dev.cuh", "common.cuh", "internal.h"),
                  "k_ckpt_pack": ("pack.cu", "common.cuh", "internal.h")}
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="gpt-110M-list",
                   help="gpt-110M-list | flat-12.8M | flat-65536 | flat-2^K")
    p.add_argument("--ckpt-every", type=int, default=100)
    p.add_argument("--ckpt-dir", default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-config objects (flat 2^30, 12.8M, 65,536)")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--sweep", action="store_true",
                   help="per-size kernel measurements (flat 2^20..2^30, latency at 65,536); "
                        "prints one JSON object per size instead of the bench line")
    p.add_argument("--sweep-parts", default="sizes,mixed,latency",
                   help="with --sweep: which parts to run (comma list of sizes, mixed, latency; "
                        "latency includes the one-launch crossover at 2^16 .. 2^20)")
    return p.parse_args(argv)


def workload(name):
    from synthetic import workloads as W
    if name.startswith("flat-2^"):
        return W.flat_pow2(int(name.split("^")[1]))
    return W.WORKLOADS[name]()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel):
    """sha256 prefix over the kernel's source files, in order."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "optimizer_step_resumable_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel, workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        digest = source_digest(kernel)
        for line in open(path):
            f = line.split()
            if len(f) >= 4 and f[0] == kernel and f[1] == workload_name and f[3] == digest:
                return float(f[2])
    except OSError:
        pass
    return None


def copy_overlap(step_iv, copy_iv):
    """Which timed steps ran beside each checkpoint's staging copy, and the
    step time they lost.  step_iv: (start, end) of each step's fused kernel,
    copy_iv: (start, end) of each copy, all in ms from one reference event.
    A step overlaps a copy when the intervals intersect; the loss is the
    overlapped steps' time above the median of the steps that overlap none."""
    hit = [any(a < hi and b > lo for lo, hi in copy_iv) for a, b in step_iv]
    clean = [b - a for (a, b), h in zip(step_iv, hit) if not h]
    base = statistics.median(clean) if clean else None
    out = []
    for lo, hi in copy_iv:
        durs = [b - a for a, b in step_iv if a < hi and b > lo]
        out.append({"copy_ms": hi - lo, "steps_overlapped": len(durs),
                    "step_ms_lost": (sum(durs) - len(durs) * base) if base is not None else None})
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self, index, enabled=True):
        self.proc = None
        self.path = None
        if not enabled or shutil.which("nvidia-smi") is None:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={index}", f"--query-gpu={CLOCK_FIELDS}", "--format=csv",
             "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f.read().splitlines()[1:]:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    rows.append((float(c[1].split()[0]), float(c[2].split()[0]),
                                 float(c[3].split()[0]) if c[3][0].isdigit() else 0.0, c[5:9]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, flag in zip(names, r[3]) if flag == "Active"})
        busy = [r[0] for r in rows if r[2] > 300.0] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(r[2] for r in rows)}


_HOST_GROUP = None  # gloo group for host-side collectives (barrier, max)


def dist_setup(device_collectives=False):
    """Process group from torchrun's environment.  With device_collectives
    (the GPU arm), the default group is NCCL -- the step's exchange runs on
    the device -- and a gloo group carries the host-side barrier and max."""
    global _HOST_GROUP
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if device_collectives:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", rank=rank, world_size=world,
                                    device_id=torch.device("cuda", local))
            _HOST_GROUP = dist.new_group(backend="gloo")
        else:
            dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier(group=_HOST_GROUP)


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=_HOST_GROUP)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)
# ---------------------------------------------------------------------------
class OracleTimer:
    """The oracle's full step (norm, clip, AdamW) on the first S parameters
    of the workload, inputs prepared once.  With threads > 1 the sample is
    cut into one contiguous slice per thread: each thread sums its slice's
    squares (the oracle's sumsq), the sums are added in slice order, the
    oracle's clip factor of the total is taken, and each thread updates its
    slice with it (the oracle's update over a range).  The oracle's C calls
    release the GIL, so the threads run on separate cores."""

    def __init__(self, wl, sample=1 << 21, threads=1):
        import numpy as np

        import oracle
        import synthetic
        self.o = oracle.load()
        self.wl = wl
        self.S = S = min(wl.n, sample)
        self.threads = max(1, min(threads, S))
        self.bounds = [S * i // self.threads for i in range(self.threads + 1)]
        self.pool = None
        if self.threads > 1:
            from concurrent.futures import ThreadPoolExecutor
            self.pool = ThreadPoolExecutor(self.threads)
        self.w = synthetic.weights(wl.seed, n=S)
        self.g = synthetic.grads(wl.seed, 1, wl.grad_sigma, n=S, outlier_frac=wl.outlier_frac,
                                 outlier_mult=wl.outlier_mult)
        self.m = np.zeros(S, np.float32)
        self.v = np.zeros(S, np.float32)
        self.t = 1
        self.total_steps = 0
        self.total_s = 0.0

    def step(self):
        wl = self.wl
        if self.pool is None:
            self.o.adamw_clip_step(self.w, self.g, self.m, self.v, self.t, wl.lr, wl.wd, wl.clip)
            return
        b, T = self.bounds, self.threads
        parts = list(self.pool.map(lambda i: self.o.sumsq(self.g[b[i]:b[i + 1]]), range(T)))
        total = 0.0
        for p in parts:  # slice order
            total += p
        s = self.o.clip_scale(math.sqrt(total), wl.clip)
        list(self.pool.map(lambda i: self.o.adamw_update_range(
            self.w, self.g, self.m, self.v, b[i], b[i + 1], s, self.t, wl.lr, wl.wd), range(T)))

    def run(self, seconds):
        """params/s over repeated steps lasting at least `seconds`."""
        reps = 0
        t0 = time.perf_counter()
        while True:
            self.step()
            reps += 1
            self.t += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        self.total_steps += reps
        self.total_s += el
        return self.S * reps / el

    def describe(self, value):
        how = ("single thread" if self.threads == 1 else
               f"{self.threads} threads, one contiguous slice each, slice sums of squares "
               f"added in slice order")
        return {"value": value, "unit": UNIT, "cores": self.threads, "kind": "oracle",
                "sample": f"oracle clip+AdamW step (norm, clip, update; double intermediates) "
                          f"on the first {self.S} parameters of {self.wl.name}, "
                          f"{self.total_steps} steps in {self.total_s:.1f} s, {how}"}

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def time_oracle(wl, seconds):
    """All host cores (the reported baseline) and, for context, one core."""
    cores = host_cores()
    timer = OracleTimer(wl, sample=1 << 24, threads=cores)
    timer.run(min(1.0, seconds / 10))  # warm-up: first touch of the arrays
    timer.total_steps, timer.total_s = 0, 0.0
    out = timer.describe(timer.run(seconds * 2 / 3))
    timer.close()
    single = OracleTimer(wl)
    out["single_thread"] = single.describe(single.run(seconds / 3))
    return out


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = workload(args.workload)
    per_step = max(0.25, min(args.cpu_seconds, 90.0 / max(1, args.steps + args.warmup)))
    timer = OracleTimer(wl, sample=1 << 24, threads=host_cores())
    for _ in range(args.warmup):
        timer.run(per_step / 4)
    timer.total_steps, timer.total_s = 0, 0.0
    runs = [timer.run(per_step) for _ in range(args.steps)]
    value = statistics.median(runs)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wl.n / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "n_params": wl.n, "sample_params": timer.S},
        "cpu_baseline": timer.describe(value),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    timer.close()
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def _state(dev, wl):
    """w, g, m, v of the workload on the device: the input generator's
    weights and step-1 gradient, zero moments."""
    import torch

    from synthetic import device as synth_dev
    n = wl.n
    w = torch.empty(n, device=dev)
    g = torch.empty(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    synth_dev.fill_grads(g, wl.seed, 1, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
    return w, g, m, v


def _timing_events(k):
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k)]
    return evs


def time_region(step, t0, K, main, split=False):
    """K steps back to back on `main` (t = t0, t0 + 1, ...), bracketed by
    one event before the first and one after the last step.  Returns
    (elapsed ms, [(norm ms, fused ms)] per step if split).  With split the
    library records an event between each step's two kernels (that turns
    off the programmatic launch of the fused kernel for those steps)."""
    import torch
    evs = _timing_events(K) if split else []
    for trio in evs:  # record once, so that the events exist
        for e in trio:
            e.record(main)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(main)
    for k in range(K):
        step(t0 + k, evs[k] if split else None)
    end.record(main)
    torch.cuda.synchronize()
    parts = [(a.elapsed_time(b), b.elapsed_time(c)) for a, b, c in evs]
    return start.elapsed_time(end), parts


def kernel_stats(parts, n, peak):
    norm = [p[0] for p in parts]
    fused = [p[1] for p in parts]
    out = {}
    for name, ms_list, per in (("k_grad_norm", norm, NORM_BYTES), ("k_clip_adamw", fused, STEP_BYTES)):
        avg = statistics.mean(ms_list)
        gbs = per * n / avg / 1e6
        out[name] = {"avg_ms": avg, "min_ms": min(ms_list), "GB/s": gbs, "frac": gbs / peak,
                     "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS}
    return out


def pack_stats(osr, ctx, w, m, v, main, side, reps, n, peak):
    """The pack kernel alone (events on the main stream; the staging copy to
    the pinned image goes to the side stream and is waited for between
    reps) and the copy (events from the end of the pack to the end of the
    copy)."""
    import torch
    pk, cp = [], []
    for _ in range(reps):
        torch.cuda.synchronize()
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(main)
        osr.ckpt_pack(ctx, 1, w, m, v, main_stream=main, side_stream=side)
        b.record(main)
        c.record(side)
        torch.cuda.synchronize()
        pk.append(a.elapsed_time(b))
        cp.append(b.elapsed_time(c))
    pm = statistics.median(pk)
    return {"k_ckpt_pack": {"ms": pm, "GB/s": PACK_BYTES * n / pm / 1e6,
                            "frac": PACK_BYTES * n / pm / 1e6 / peak,
                            "frac_of_nominal_8tbs": PACK_BYTES * n / pm / 1e6 / NOMINAL_HBM_GBS},
            "staging_to_pinned": {"ms": statistics.median(cp),
                                  "GB/s": (8 + 12 * n) / statistics.median(cp) / 1e6}}


def oracle_rates(wl, seconds):
    """The oracle on this workload (a bounded sample of its first
    parameters): every host core and one core."""
    cores = host_cores()
    timer = OracleTimer(wl, sample=min(wl.n, 1 << 24), threads=cores)
    timer.run(min(0.5, seconds / 10))  # first touch of the arrays
    timer.total_steps, timer.total_s = 0, 0.0
    out = {"all_cores": timer.describe(timer.run(seconds * 2 / 3))}
    timer.close()
    single = OracleTimer(wl, sample=min(wl.n, 1 << 21))
    out["one_core"] = single.describe(single.run(seconds / 3))
    return out


def _guarded(fn, *args):
    """fn(*args), or {"error": ...} if it raises (for example when a state of
    2^30 parameters, or its pinned checkpoint image, does not fit), so that
    one configuration cannot cost the bench line."""
    import torch
    try:
        return fn(*args)
    except Exception as e:  # noqa: BLE001 -- reported in the line instead
        try:
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        except Exception:  # noqa: BLE001 -- the error above is the one reported
            pass
        return {"error": f"{type(e).__name__}: {e}"[:300]}


def config_throughput(name, K, W, dev, main, side, peak, cpu_seconds):
    """params/s of the library's default step on one flat workload (inputs
    resident; above L2 for 12.8M and up), each kernel's rate from a second
    region with events between the kernels, the checkpoint pack's rate,
    and the oracle's rate beside it."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    wl = workload(name)
    n = wl.n
    w, g, m, v = _state(dev, wl)
    ctx = osr.adamw_create(n)

    def step(t, ev):
        if ev is not None:
            osr.adamw_record_events(ctx, *ev)
        osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)

    for t in range(1, W + 1):
        step(t, None)
    ms, _ = time_region(step, W + 1, K, main)
    _, parts = time_region(step, W + 1 + K, K, main, split=True)
    out = {"workload": wl.name, "n_params": n, "steps": K,
           "ms_per_step": ms / K, "params/s": n * K / (ms / 1e3),
           "step_GB/s": (STEP_BYTES + NORM_BYTES) * n * K / ms / 1e6,
           "frac": (STEP_BYTES + NORM_BYTES) * n * K / ms / 1e6 / peak,
           "frac_of_nominal_8tbs": (STEP_BYTES + NORM_BYTES) * n * K / ms / 1e6 / NOMINAL_HBM_GBS,
           "l2": f"w, g, m, v = {16 * n / 1e9:.3g} GB, {'above' if 16 * n > 126e6 else 'within'} L2"}
    out.update(kernel_stats(parts, n, peak))
    out.update(pack_stats(osr, ctx, w, m, v, main, side, 3, n, peak))
    ctx.close()
    del w, g, m, v
    torch.cuda.empty_cache()
    out["oracle"] = oracle_rates(wl, cpu_seconds)
    return out


def config_latency(dev, main, cpu_seconds):
    """The 65,536-parameter state (L2-resident): microseconds per step,
    host-driven through the library's default step and its step graph, and
    the GPU time of steps captured back to back into one CUDA graph."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    wl = workload("flat-65536")
    n = wl.n
    w, g, m, v = _state(dev, wl)
    steps = 2000
    out = {"workload": wl.name, "n_params": n}
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_graph_create(ctx, w, g, m, v)
        for mode in ("host_loop", "step_graph"):
            graph = mode == "step_graph"
            for t in range(1, 50):
                (osr.adamw_graph_step(ctx, t, wl.lr, wl.wd, wl.clip) if graph
                 else osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip))
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for t in range(50, 50 + steps):
                if graph:
                    osr.adamw_graph_step(ctx, t, wl.lr, wl.wd, wl.clip)
                else:
                    osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            b.record(main)
            b.synchronize()
            out[mode] = {"us_per_step": 1e3 * a.elapsed_time(b) / steps,
                         "params/s": n * steps / (a.elapsed_time(b) / 1e3)}
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gr, stream=cap):
                for _ in range(50):
                    osr.adamw_clip_step(ctx, w, g, m, v, 100, wl.lr, wl.wd, wl.clip, stream=cap)
        gr.replay()
        torch.cuda.synchronize()
        ms, _, _ = median_ms(gr.replay, 20, main)
        out["gpu_time_captured"] = {"us_per_step": 1e3 * ms / 50,
                                    "params/s": n * 50 / (ms / 1e3)}
        del gr
    out["oracle"] = oracle_rates(wl, cpu_seconds)
    return out


def run_ours(args):
    import torch

    import optimizer_step_resumable_gb300 as osr
    from optimizer_step_resumable_gb300 import build as lib_build
    from optimizer_step_resumable_gb300 import sharded

    lib_build.build()  # no-op when the library is up to date
    world, rank, local = dist_setup(device_collectives=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload(args.workload)
    n = wl.n
    off, num = wl.table()
    K, W, C = args.steps, max(args.warmup, 0), max(args.ckpt_every, 1)
    peak, peak_kind = measured_peaks()

    w, g, m, v = _state(dev, wl)
    ctx = osr.adamw_create(n, off, num)
    exchange = sharded.DeviceExchange(world, dev) if world > 1 else None
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ckdir = tempfile.mkdtemp(prefix="ckpt_", dir=args.ckpt_dir)
    torch.cuda.synchronize()

    def step(t, ev=None, grad=None):
        """One optimizer step (single GPU: norm + fused kernel; N ranks: each
        rank owns one shard of an N x n state, the shards' sums of squares
        are exchanged and added in rank order, then the fused update)."""
        gr = g if grad is None else grad
        if world == 1:
            if ev is not None:
                osr.adamw_record_events(ctx, *ev)
            osr.adamw_clip_step(ctx, w, gr, m, v, t, wl.lr, wl.wd, wl.clip)
            return
        # N ranks: the shard's sum of squares, an NCCL all-gather and the
        # rank-order sum all on the device (no host round trip)
        if ev is not None:
            ev[0].record(main)
        osr.grad_sumsq_to(ctx, gr, exchange.send)
        torch.distributed.all_gather_into_tensor(exchange.recv, exchange.send)
        if ev is not None:
            ev[1].record(main)
        osr.adamw_clip_step_gathered(ctx, w, gr, m, v, t, wl.lr, wl.wd, wl.clip, exchange.recv)
        if ev is not None:
            ev[2].record(main)

    # (1) the timed region of `value`: K steps as the library runs them, right
    # after the W warm-up steps (no idle gap between them, so the first timed
    # steps do not start on a GPU that has been idle)
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.3 if sampler.proc else 0)
    barrier(world)
    t = 1
    for _ in range(W):
        step(t)
        t += 1
    elapsed_ms, _ = time_region(step, t, K, main)
    t += K
    barrier(world)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    # (2) the same K steps with an event between the two kernels of each:
    # per-kernel times (the dominant kernel's roofline)
    barrier(world)
    split_ms, parts = time_region(step, t, K, main, split=True)
    t += K
    barrier(world)
    clocks = sampler.stop()
    norm_val, scale = osr.adamw_last_norm(ctx) if world == 1 else (None, None)

    # (3) one checkpoint of the state (pack, staging copy to the pinned image
    # on the side stream, O_DIRECT write + fsync + rename, all waited for),
    # twice; then the copy beside the next steps
    ck = []
    for _ in range(2):
        osr.ckpt_wait(ctx)
        torch.cuda.synchronize()
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        h0 = time.perf_counter()
        a.record(main)
        osr.ckpt_pack(ctx, t - 1, w, m, v, main_stream=main, side_stream=side)
        b.record(main)
        c.record(side)
        osr.ckpt_write(ctx, ckdir)
        ck.append({"total_s": time.perf_counter() - h0, "pack_ms": a.elapsed_time(b),
                   "copy_ms": b.elapsed_time(c)})
    ck_s = ck[-1]["total_s"]
    # a checkpoint written in the background while 40 steps run: which steps
    # ran beside the staging copy and what they lost
    ov = _timing_events(40)
    for trio in ov:
        for e in trio:
            e.record(main)
    ref, pack_end, copy_end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    ref.record(main)
    osr.ckpt_pack(ctx, t - 1, w, m, v, main_stream=main, side_stream=side)
    pack_end.record(main)
    copy_end.record(side)
    osr.ckpt_write_async(ctx, ckdir)
    for k in range(40):
        step(t, ov[k])
        t += 1
    osr.ckpt_wait(ctx)
    torch.cuda.synchronize()
    beside = copy_overlap([(ref.elapsed_time(b), ref.elapsed_time(c)) for _, b, c in ov],
                          [(ref.elapsed_time(pack_end), ref.elapsed_time(copy_end))])

    # end to end through the public API: every step's gradient copied from
    # pinned host memory (on an upload stream, into one of two device
    # buffers, so the copy for step k + 1 runs while step k computes, as a
    # data loader would feed it) and every step's norm read back on the host
    e2e = None
    if not args.no_e2e:
        g_host = g.cpu().pin_memory()
        bufs = [g, torch.empty_like(g)]
        up = torch.cuda.Stream()
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e_start.record(main)
        up.wait_event(e_start)
        with torch.cuda.stream(up):
            bufs[0].copy_(g_host, non_blocking=True)
        ready[0].record(up)
        for k in range(K):
            cur, nxt = k % 2, 1 - k % 2
            if k + 1 < K:
                if k >= 1:  # buffer nxt was read by step k - 1
                    up.wait_event(used[nxt])
                with torch.cuda.stream(up):
                    bufs[nxt].copy_(g_host, non_blocking=True)
                ready[nxt].record(up)
            main.wait_event(ready[cur])
            step(t, grad=bufs[cur])
            used[cur].record(main)
            if world == 1:
                osr.adamw_last_norm(ctx)
            else:
                exchange.recv.cpu()
            t += 1
        e_end.record(main)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(e_start.elapsed_time(e_end), world)
        e2e = {"value": world * n * K / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 8 * (1 if world == 1 else world),
               "ms_per_step": e_ms / K,
               "how": "gradient uploaded from pinned host memory every step into one of two "
                      "device buffers on an upload stream (step k + 1's copy overlaps step k), "
                      "the norm read back on the host after every step"}
        del bufs

    ctx.close()
    del w, g, m, v
    torch.cuda.empty_cache()
    shutil.rmtree(ckdir, ignore_errors=True)
    if rank != 0:
        return 0

    ks = kernel_stats(parts, n, peak)
    fused_ms = ks["k_clip_adamw"]["avg_ms"]
    achieved = STEP_BYTES * n / fused_ms / 1e6
    traffic = traffic_record("k_clip_adamw", wl.name)
    step_ms = elapsed_ms / K
    value = world * n * K / (elapsed_ms / 1e3)
    whole_ms = step_ms + 1e3 * ck_s / C
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": wl.name, "n_params": n, "tensors": len(off),
            "parallelism": (f"zero1 x{world}: one {wl.name} shard per rank, sums of squares "
                            f"all-gathered (NCCL, on the device) and added in rank order "
                            f"each step")
                           if world > 1 else "single GPU",
            "value_is": "one optimizer step per step (norm kernel + fused clip+AdamW kernel as "
                        "the library launches them: the fused kernel a programmatic dependent "
                        "of the norm); the checkpoint, every 100 steps, is in whole_path",
            "l2": f"inputs larger than L2: w, g, m, v = {16 * n / 1e9:.2f} GB",
            "lr": wl.lr, "wd": wl.wd, "clip": wl.clip, "grad_norm": norm_val,
            "clip_scale": scale,
        },
        "roofline": {
            "bound": "hbm", "kernel": "k_clip_adamw", "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "bytes_per_launch": STEP_BYTES * n, "traffic": traffic,
            "timed": f"average of the {K} fused-kernel launches of the split region",
        },
        "step_pdl": {"ms": step_ms, "GB/s": (STEP_BYTES + NORM_BYTES) * n / step_ms / 1e6,
                     "frac": (STEP_BYTES + NORM_BYTES) * n / step_ms / 1e6 / peak,
                     "note": "the timed region of value: K steps, events only around it"},
        "step_only": {"ms": split_ms / K,
                      "kernels_ms": statistics.mean(a + b for a, b in parts),
                      "GB/s": (STEP_BYTES + NORM_BYTES) * n / (split_ms / K) / 1e6,
                      "note": "K more steps with an event between the two kernels of each "
                              "(plain stream order, no programmatic launch): kernels_ms is "
                              "the mean of the norm's and the fused kernel's event times"},
        "kernels_ms": ks,
        "whole_path": {
            "ms_per_step": whole_ms, "params/s": world * n / (whole_ms / 1e3),
            "ckpt_every": C, "checkpoint_s": ck_s,
            "how": f"step_pdl plus 1/{C} of one checkpoint measured after the timed steps "
                   f"(pack kernel, staging copy to the pinned image, O_DIRECT write, fsync, "
                   f"rename, directory fsync, all waited for): the pages' cadence of one "
                   f"checkpoint every {C} steps",
        },
        "checkpoint": {
            "bytes": 8 + 12 * n, "runs": ck,
            "pack_GB/s": PACK_BYTES * n / ck[-1]["pack_ms"] / 1e6,
            "copy_GB/s": (8 + 12 * n) / ck[-1]["copy_ms"] / 1e6,
            "write_GB/s": (8 + 12 * n) / (ck_s - 1e-3 * (ck[-1]["pack_ms"] + ck[-1]["copy_ms"]))
            / 1e9,
            "dir": "temp dir under " + (args.ckpt_dir or tempfile.gettempdir()),
            "copy_beside_steps": beside,
        },
        # value region: norm + fused per step (N ranks: norm, rank-order
        # total, fused)
        "gpu_launches": (2 if world == 1 else 3) * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_configs:
        cs = max(1.0, args.cpu_seconds / 4)
        line["per_config"] = {
            "flat-2^30": _guarded(config_throughput, "flat-2^30", K, W, dev, main, side, peak, cs),
            "flat-12.8M": _guarded(config_throughput, "flat-12.8M", K, W, dev, main, side, peak,
                                   cs),
            "flat-65536": _guarded(config_latency, dev, main, cs),
        }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def median_ms(fn, reps, stream):
    """Median duration of fn() over reps, CUDA events on `stream`."""
    import torch
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        out.append(a.elapsed_time(b))
    return statistics.median(out), min(out), max(out)


def run_sweep(args):
    """Kernel rates per state size (flat vectors, g ~ 1e-3 with 0.1% outliers
    x1000) and the launch-latency case at 65,536 parameters, plain vs graph.
    Each kernel is timed alone (median of reps, CUDA events); between reps
    the L2 is emptied by reading a 512 MB buffer (a read leaves no dirty
    lines whose write-back would land in the measured kernels).  The GPU
    time of a whole step without host launch overhead comes from replaying
    a CUDA graph of 50 captured steps."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    from optimizer_step_resumable_gb300 import build as lib_build
    from synthetic import device as synth_dev
    from synthetic import workloads as W

    lib_build.build()
    dev = torch.device("cuda", 0)
    main = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    flush = torch.ones(128 << 20, device=dev)
    rows = []
    parts = set(args.sweep_parts.split(","))
    for log2n in range(20, 31) if "sizes" in parts else ():
        wl = W.flat_pow2(log2n)
        n = wl.n
        w = torch.empty(n, device=dev)
        g = torch.empty(n, device=dev)
        m = torch.zeros(n, device=dev)
        v = torch.zeros(n, device=dev)
        synth_dev.fill_weights(w, wl.seed)
        synth_dev.fill_grads(g, wl.seed, 1, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
        ctx = osr.adamw_create(n)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in evs:
            e.record(main)
        reps = 20 if n <= (1 << 27) else 8
        norm_ms, step_ms, whole = [], [], {"pdl": [], "no_pdl": []}
        t = 1
        for mode in ("split", "pdl", "no_pdl"):
            osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_PDL if mode == "no_pdl" else 0)
            for r in range(reps + 3):
                flush.sum()
                if mode == "split":  # an event between the kernels: plain order
                    osr.adamw_record_events(ctx, *evs)
                else:
                    osr.adamw_record_events(ctx, evs[0], None, evs[2])
                osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
                t += 1
                evs[2].synchronize()
                if r < 3:
                    continue
                if mode == "split":
                    norm_ms.append(evs[0].elapsed_time(evs[1]))
                    step_ms.append(evs[1].elapsed_time(evs[2]))
                else:
                    whole[mode].append(evs[0].elapsed_time(evs[2]))
        osr.adamw_set_launch_options(ctx, 0)

        def pack():
            osr.ckpt_pack(ctx, 1, w, m, v, main_stream=main, side_stream=main)

        pack_ms, _, _ = median_ms(pack, max(3, reps // 2), main)
        osr.ckpt_wait(ctx)
        # the pack kernel alone: the copy goes to another stream, so the
        # events on the main stream bracket the kernel only
        side = torch.cuda.Stream()

        def pack_only():
            osr.ckpt_pack(ctx, 1, w, m, v, main_stream=main, side_stream=side)

        pack_only()
        torch.cuda.synchronize()
        pack_k = []
        for _ in range(max(3, reps // 2)):
            flush.sum()
            torch.cuda.synchronize()
            pack_k.append(median_ms(pack_only, 1, main)[0])
            torch.cuda.synchronize()
        pack_kernel_ms = statistics.median(pack_k)
        # GPU time per step without launch overhead: 50 steps in one graph
        # (t fixed inside the graph; the kernels' work does not depend on t)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gr, stream=cap):
                for _ in range(50):
                    osr.adamw_clip_step(ctx, w, g, m, v, 100, wl.lr, wl.wd, wl.clip, stream=cap)
        gr.replay()
        torch.cuda.synchronize()
        graph_ms, _, _ = median_ms(gr.replay, 5, main)
        graph_step_ms = graph_ms / 50
        ctx.close()
        nm, sm = statistics.median(norm_ms), statistics.median(step_ms)
        row = {"workload": wl.name, "n": n,
               "k_grad_norm": {"ms": nm, "GB/s": 4 * n / nm / 1e6, "frac": 4 * n / nm / 1e6 / peak},
               "k_clip_adamw": {"ms": sm, "GB/s": 28 * n / sm / 1e6,
                                "frac": 28 * n / sm / 1e6 / peak},
               "step": {"ms": nm + sm, "params/s": n / ((nm + sm) / 1e3),
                        "GB/s": 32 * n / (nm + sm) / 1e6},
               "step_whole": {m: {"ms": statistics.median(x),
                                  "GB/s": 32 * n / statistics.median(x) / 1e6}
                              for m, x in whole.items()},
               "step_graph": {"ms": graph_step_ms, "params/s": n / (graph_step_ms / 1e3),
                              "GB/s": 32 * n / graph_step_ms / 1e6},
               "pack+d2h": {"ms": pack_ms, "GB/s(device 24n)": 24 * n / pack_ms / 1e6},
               "k_ckpt_pack": {"ms": pack_kernel_ms, "GB/s": 24 * n / pack_kernel_ms / 1e6,
                               "frac": 24 * n / pack_kernel_ms / 1e6 / peak},
               "peak_GB/s": peak, "peak_kind": peak_kind}
        rows.append(row)
        print(json.dumps(row), flush=True)
        del w, g, m, v
        torch.cuda.empty_cache()

    if "mixed" in parts:
        sweep_mixed(dev, main, flush, peak)
    if "latency" in parts:
        sweep_latency(dev, main)
    return 0


def sweep_mixed(dev, main, flush, peak):
    """Mixed precision on the 110M tensor list: bfloat16 gradient, bfloat16
    copy of the new weights (2 + 28 bytes per parameter)."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    from synthetic import device as synth_dev
    from synthetic import workloads as W
    wl = W.gpt_110m()
    n = wl.n
    off, num = wl.table()
    w = torch.empty(n, device=dev)
    g32 = torch.empty(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    synth_dev.fill_grads(g32, wl.seed, 1, wl.grad_sigma)
    g16 = g32.to(torch.bfloat16)
    del g32
    w_lp = torch.empty(n, dtype=torch.bfloat16, device=dev)
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        times, norm_ms, fused_ms = [], [], []
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in evs:
            e.record(main)
        for t in range(1, 44):
            flush.sum()
            split = t % 2 == 0  # every other step: an event between the kernels
            osr.adamw_record_events(ctx, evs[0], evs[1] if split else None, evs[2])
            osr.adamw_clip_step_mixed(ctx, w, g16, m, v, t, wl.lr, wl.wd, wl.clip, w_lp=w_lp)
            evs[2].synchronize()
            if t > 3:
                if split:
                    norm_ms.append(evs[0].elapsed_time(evs[1]))
                    fused_ms.append(evs[1].elapsed_time(evs[2]))
                else:
                    times.append(evs[0].elapsed_time(evs[2]))
        ms = statistics.median(times)
        nm, fm = statistics.median(norm_ms), statistics.median(fused_ms)
    row = {"workload": wl.name + " mixed (bf16 g, bf16 weight copy)", "n": n,
           "step": {"ms": ms, "params/s": n / (ms / 1e3), "GB/s": 30 * n / ms / 1e6,
                    "frac": 30 * n / ms / 1e6 / peak},
           "k_grad_norm": {"ms": nm, "GB/s": 2 * n / nm / 1e6, "frac": 2 * n / nm / 1e6 / peak},
           "k_clip_adamw": {"ms": fm, "GB/s": 28 * n / fm / 1e6,
                            "frac": 28 * n / fm / 1e6 / peak}}
    print(json.dumps(row), flush=True)
    del w, m, v, g16, w_lp
    torch.cuda.empty_cache()


def sweep_latency(dev, main):
    """Latency case: 65,536 parameters (L2-resident): host-driven steps and
    the GPU time of captured steps, one-launch vs two-launch."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    from synthetic import device as synth_dev
    from synthetic import workloads as W
    wl = W.flat_65k()
    n = wl.n
    w = torch.empty(n, device=dev)
    g = torch.empty(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    synth_dev.fill_weights(w, wl.seed)
    synth_dev.fill_grads(g, wl.seed, 1, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
    steps = 1000
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        osr.adamw_graph_create(ctx, w, g, m, v)
        out = {}
        # host-driven loops: the default step (one launch of thread-block
        # clusters at this size), the two-launch step, the library's step
        # graph (one cluster-kernel node at this size, or the two-node graph)
        for mode in ("plain", "plain_two_launch", "graph", "graph_two_node"):
            osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS
                                         if mode.endswith("two_launch") or
                                         mode.endswith("two_node") else 0)
            graph = mode.startswith("graph")
            for t in range(1, 50):
                (osr.adamw_graph_step(ctx, t, wl.lr, wl.wd, wl.clip) if graph
                 else osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip))
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for t in range(50, 50 + steps):
                if graph:
                    osr.adamw_graph_step(ctx, t, wl.lr, wl.wd, wl.clip)
                else:
                    osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
            b.record(main)
            b.synchronize()
            out[mode] = {"us_per_step": 1e3 * a.elapsed_time(b) / steps,
                         "params/s": n * steps / (a.elapsed_time(b) / 1e3)}
        # GPU time per step: 50 steps captured into one graph and replayed
        for mode in ("captured", "captured_two_launch"):
            osr.adamw_set_launch_options(ctx, osr.LAUNCH_NO_ONEPASS
                                         if mode == "captured_two_launch" else 0)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(gr, stream=cap):
                    for _ in range(50):
                        osr.adamw_clip_step(ctx, w, g, m, v, 100, wl.lr, wl.wd, wl.clip,
                                            stream=cap)
            gr.replay()
            torch.cuda.synchronize()
            ms, _, _ = median_ms(gr.replay, 20, main)
            out[mode] = {"us_per_step": 1e3 * ms / 50, "params/s": n * 50 / (ms / 1e3)}
            del gr
        osr.adamw_set_launch_options(ctx, 0)
    row = {"workload": wl.name, "n": n, "latency": out}
    print(json.dumps(row), flush=True)
    del w, g, m, v
    sweep_one_launch_crossover(dev, main)
    return 0


def sweep_one_launch_crossover(dev, main):
    """The library's default step against two launches at 2^16 .. 2^20
    parameters: microseconds per host-driven step (2000 steps) and GPU time
    per step of 50 steps captured in one graph (replayed 20 times)."""
    import torch

    import optimizer_step_resumable_gb300 as osr
    from synthetic import device as synth_dev
    from synthetic import workloads as W
    for log2n in range(16, 21):
        wl = W.flat_pow2(log2n)
        n = wl.n
        w = torch.empty(n, device=dev)
        g = torch.empty(n, device=dev)
        m = torch.zeros(n, device=dev)
        v = torch.zeros(n, device=dev)
        synth_dev.fill_weights(w, wl.seed)
        synth_dev.fill_grads(g, wl.seed, 1, wl.grad_sigma, wl.outlier_frac, wl.outlier_mult)
        row = {"workload": wl.name, "n": n}
        with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
            for mode, flags in (("default", 0), ("two_launch", osr.LAUNCH_NO_ONEPASS)):
                osr.adamw_set_launch_options(ctx, flags)
                for t in range(1, 20):
                    osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(main)
                for t in range(20, 2020):
                    osr.adamw_clip_step(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip)
                b.record(main)
                b.synchronize()
                host_us = 1e3 * a.elapsed_time(b) / 2000
                gr = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream()
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(gr, stream=cap):
                        for _ in range(50):
                            osr.adamw_clip_step(ctx, w, g, m, v, 100, wl.lr, wl.wd, wl.clip,
                                                stream=cap)
                gr.replay()
                torch.cuda.synchronize()
                ms, _, _ = median_ms(gr.replay, 20, main)
                row[mode] = {"host_us_per_step": host_us, "gpu_us_per_step_captured": 1e3 * ms / 50}
                del gr
            osr.adamw_set_launch_options(ctx, 0)
        print(json.dumps(row), flush=True)
        del w, g, m, v
        torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
