#!/usr/bin/env python3
"""Benchmark of the GB300 GEMM library: one JSON line on stdout (rank 0).

A step is one pass of the measured workload: the bf16 8192^3 tensor-core GEMM followed
by the fp32 4096^3 FFMA GEMM (the two products the headline metric is quoted on), on
seeded synthetic inputs resident in HBM.  value = 2MNK summed over the step's GEMMs /
device time, in TFLOP/s, summed over ranks (replicas; the GEMM does not shard here).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workloads bf16_8192,f32_4096] [--no-extras]

--impl reference times the CPU oracle (fp64 triple loop) on a bounded row sample of the
same workload and prints the same kind of line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/device time) & % of GB300 peak, bf16 8192³ and fp32 4096³"
DEFAULT_WORKLOADS = ["bf16_8192", "f32_4096"]
EXTRA_WORKLOADS = ["f32_skinny", "conv4d"]
FP32_LANES_PER_SM = 128
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
L2_FLUSH_BYTES = 512 << 20
CLOCK_WINDOW_S = 1.5  # back-to-back run per workload with the clock sampler on (warm-L2 context numbers)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workloads", default=",".join(DEFAULT_WORKLOADS))
    ap.add_argument("--no-extras", action="store_true", help="skip the skinny / conv side measurements")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="--impl reference: target wall time of warm-up plus timed steps")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    a.steps = max(a.steps, 1)
    return a


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def fp32_simt_peak_tflops(sm_mhz: float, sms: int) -> float:
    """FP32 FFMA peak: SMs (queried from the device) x 128 lanes x 2 flop x clock."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


# ------------------------------------------------------------------ clock sampling

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + CLOCK_FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = None
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            self.rows = []
            with open(self.path) as fh:
                for r in csv.reader(fh):
                    if len(r) >= 9:
                        self.rows.append([c.strip() for c in r])
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)

    def summary(self):
        return summarize_clocks(self.rows)


def summarize_clocks(rows):
    """Median SM clock and throttle reasons over the samples taken under load (power
    draw above 250 W), from nvidia-smi rows; rows None = no sampler."""
    if rows is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

    def num(v):
        try:
            return float(v)
        except ValueError:
            return None
    smax = max((num(r[2]) or 0) for r in rows)
    busy = [r for r in rows if (num(r[3]) or 0) > 250.0] or rows  # power draw marks load
    clocks = [num(r[1]) for r in busy if num(r[1]) is not None]
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in busy:
        for name, v in zip(names, r[5:9]):
            if v.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(clocks) if clocks else None, "sm_max_mhz": smax,
            "reasons": sorted(reasons), "samples": len(busy),
            "power_w_max": max((num(r[3]) or 0) for r in rows)}


def reduce_max(value: float, dist_mod, device) -> float:
    """Max of a per-rank scalar over the process group (identity without one)."""
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def aggregate(flops_per_step: float, ms_local: float, world: int, dist_mod, device):
    """Whole-job throughput of `world` replicas: every rank does `flops_per_step` per step
    and the step time is the slowest rank's.  Returns (TFLOP/s, ms per step)."""
    ms = reduce_max(ms_local, dist_mod, device)
    return world * flops_per_step / (ms * 1e-3) / 1e12, ms


def clocks_rejected(c) -> bool:
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and c["sm_mhz"] < 0.5 * c["sm_max_mhz"] and not c["reasons"]:
        return True
    return False


# ------------------------------------------------------------------ traffic record

def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "programming_tiled_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# the translation units whose device code a capture measured (a change there makes the
# recorded DRAM traffic stale)
KERNEL_SOURCES = {"tc_gemm": ["tc_gemm.cu", "ptx.h"], "ffma_persistent": ["ffma_tma.cu", "ptx.h"],
                  "ffma_tiled": ["ffma.cu"], "skinny": ["skinny_tma.cu", "ptx.h"],
                  "im2col4d": ["im2col.cu"], "conv_implicit": ["conv_implicit.cu", "ffma.cu"]}


def recorded_traffic(kernel: str, units: float):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(kernel)
    if not rec or rec.get("source_hash") != kernel_source_hash(KERNEL_SOURCES[kernel]):
        return None
    # scale a capture on a smaller case to the benchmarked launch, by units processed
    return rec["dram_bytes_per_launch"] * units / rec["units"]


# ------------------------------------------------------------------ our implementation

def run_ours(args, rank, world, local_rank):
    import torch

    import programming_tiled_gemm_gb300 as g
    import seeded_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    lib = g.Gemm(local_rank)
    stream = torch.cuda.current_stream(dev)
    names = [n for n in args.workloads.split(",") if n]

    ops = []
    shas = {}
    for n in names:
        w = si.WORKLOADS[n]
        A, B = si.workload_operands(w)  # for the convolution: (x, weights)
        shas[n] = si.sha256(A, B)[:16]
        Ad, Bd = A.to(dev), B.to(dev)
        Cd = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
        ops.append((w, Ad, Bd, Cd))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def run_op(op):
        w, Ad, Bd, Cd = op
        torch.cuda.nvtx.range_push(w.name)  # lets a profiler's range filter pick one product
        if w.kind == "conv4d":
            lib.conv4d_implicit(Ad, Bd, out=Cd)  # implicit GEMM: y = W . col(x), no column matrix
        else:
            lib.matmul(Ad, Bd, out=Cd)
        torch.cuda.nvtx.range_pop()

    for _ in range(args.warmup):
        for op in ops:
            run_op(op)
    torch.cuda.synchronize()
    if lib.device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    def timed_region():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(args.steps)]
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        launches0 = lib.launch_count()
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush.zero_()  # L2 flush, outside the events
            evs[s][0].record(stream)
            for i, op in enumerate(ops):
                run_op(op)
                evs[s][i + 1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        launches = lib.launch_count() - launches0
        if pg:
            pg.barrier()
        per_op = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps)] for i in range(len(ops))]
        step_ms = [evs[s][0].elapsed_time(evs[s][-1]) for s in range(args.steps)]
        return step_ms, per_op, wall, launches

    def clock_windows():
        """Each workload back to back (no flush) for about CLOCK_WINDOW_S with the clock
        sampler on: its warm-L2 time and the SM clock the GPU holds under that load
        (the timed region itself is too short for a 100 ms sampler to see)."""
        res = []
        for op in ops:
            run_op(op)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run_op(op)
            e1.record(stream)
            torch.cuda.synchronize()
            reps = max(10, int(CLOCK_WINDOW_S * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
            with ClockSampler(local_rank) as cw:
                e0.record(stream)
                for _ in range(reps):
                    run_op(op)
                e1.record(stream)
                torch.cuda.synchronize()
            res.append((e0.elapsed_time(e1) / reps, reps, cw.rows))
        return res

    with ClockSampler(local_rank) as cs:
        step_ms, per_op, wall, launches = timed_region()
    windows = clock_windows()
    remeasured = False

    def all_clocks(timed_rows, wins):
        rows = None if timed_rows is None else list(timed_rows) + [r for *_, rw in wins for r in (rw or [])]
        return summarize_clocks(rows)
    clocks = all_clocks(cs.rows, windows)
    if clocks_rejected(clocks):
        with ClockSampler(local_rank) as cs:
            step_ms, per_op, wall, launches = timed_region()
        windows = clock_windows()
        clocks = all_clocks(cs.rows, windows)
        remeasured = True
    clocks["timed_region"] = summarize_clocks(cs.rows)
    if lib.device_status() != 0:
        raise RuntimeError("device status error in the timed region")

    flops_step = sum(op[0].flops for op in ops)
    value, ms_step = aggregate(flops_step, statistics.mean(step_ms), world, pg, dev)

    peaks, peak_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = fp32_simt_peak_tflops(peaks.get("sm_max_mhz", 2070.0), sms)
    per = {}
    kernels = []
    for (w, *_), times, (wms, wreps, wrows) in zip(ops, per_op, windows):
        ms = statistics.mean(times)
        wclk = summarize_clocks(wrows)
        tflops = w.flops / (ms * 1e-3) / 1e12
        if w.dtype == "bf16":
            peak, bound, kname = peaks["bf16_tflops"], "tensor", "tc_gemm"
        elif w.kind == "conv4d":
            peak, bound, kname = fp32_peak, "alu", "conv_implicit"
        elif w.M <= 32:
            peak, bound, kname = fp32_peak, "alu", "skinny"
        else:
            peak, bound, kname = fp32_peak, "alu", "ffma_persistent"
        entry = {"ms": round(ms, 4), "tflops": round(tflops, 2), "peak_tflops": round(peak, 1),
                 "frac": round(tflops / peak, 4), "flops": w.flops, "input_sha256": shas[w.name],
                 "warm_ms": round(wms, 4), "warm_tflops": round(w.flops / (wms * 1e-3) / 1e12, 2),
                 "clock_window": {"reps": wreps, "seconds": round(wms * wreps * 1e-3, 2),
                                  "sm_mhz": wclk.get("sm_mhz"), "samples": wclk.get("samples"),
                                  "reasons": wclk.get("reasons")}}
        wmhz = wclk.get("sm_mhz")
        if wmhz:
            # the kernel time scaled to cycles: time x the SM clock held under this load
            entry["ms_x_sm_ghz"] = round(ms * wmhz / 1e3, 4)
        if w.dtype != "bf16":
            if wmhz:
                entry["frac_at_median_clock"] = round(tflops / fp32_simt_peak_tflops(wmhz, sms), 4)
        else:
            entry["frac_of_sustained"] = round(tflops / peaks.get("bf16_tflops_sustained", peak), 4)
        per[w.name] = entry
        kernels.append((ms, w, kname, bound, peak, tflops))
    # dominant kernel = the one taking the largest share of the step
    ms_dom, w_dom, kname, bound, peak, tflops = max(kernels, key=lambda k: k[0])
    roofline = {"kernel": kname, "workload": w_dom.name, "bound": bound, "achieved": round(tflops, 2),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                "peak_source": ("of measured" if (bound == "tensor" and peak_src == "measured") else
                                "derived: %d SMs (queried from the device) x 128 FP32 lanes x 2 flop x %.0f MHz "
                                "(max SM clock)" % (sms, peaks.get("sm_max_mhz", 2070.0)) if bound == "alu"
                                else "of fallback"),
                "traffic": recorded_traffic(kname, w_dom.flops)}
    rooflines = [{"kernel": k[2], "workload": k[1].name, "bound": k[3], "achieved": round(k[5], 2),
                  "peak": round(k[4], 1), "unit": "TFLOP/s", "frac": round(k[5] / k[4], 4),
                  "traffic": recorded_traffic(k[2], k[1].flops)} for k in kernels]

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "+".join(sorted({op[0].dtype for op in ops})), "data": "synthetic",
        "config": {"workload": "+".join(names), "shapes": {w.name: [w.M, w.N, w.K] for w, *_ in ops},
                   "inputs": "seeded synthetic: bf16 = normal(0,1) rounded to bf16 (seed 2), "
                             "fp32 = uniform[-1,1] (seed 1); row-major, ld = cols",
                   "l2": "flushed between steps (%d MiB write, outside the events)" % (L2_FLUSH_BYTES >> 20),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "per_workload": per, "roofline": roofline, "rooflines": rooflines,
        "peaks_source": peak_src, "clocks": clocks, "clocks_remeasured": remeasured,
        "gpu_launches": int(launches), "wall_s_timed_region": round(wall, 3),
    }

    if not args.no_extras and rank == 0:
        out["also_measured"] = measure_extras(lib, dev, stream, peaks, fp32_peak)
    if not args.no_e2e:
        out["e2e"] = measure_e2e(lib, ops, args, dev, world, pg)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(ops, args.cpu_seconds)
    lib.close()
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_extras(lib, dev, stream, peaks, fp32_peak, reps=20):
    """Side measurements of the other two fp32 configurations (not part of `value`)."""
    import torch

    import seeded_inputs as si
    res = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def time_fn(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    w = si.WORKLOADS["f32_skinny"]
    A, B = si.workload_operands(w)
    Ad, Bd = A.to(dev), B.to(dev)
    C = torch.empty((w.M, w.N), device=dev)
    ms = time_fn(lambda: lib.matmul(Ad, Bd, out=C))
    bytes_min = 4 * (w.M * w.K + w.K * w.N + w.M * w.N)
    res["f32_skinny"] = {"ms": round(ms, 4), "tflops": round(w.flops / ms / 1e9, 2),
                         "gbs": round(bytes_min / ms / 1e6, 1), "hbm_frac": round(bytes_min / ms / 1e6 / peaks["hbm_gbs"], 4),
                         "bound": "hbm", "bytes_algorithmic": bytes_min}
    del Ad, Bd, C

    w = si.WORKLOADS["conv4d"]
    c = w.conv
    x, wt = si.workload_operands(w)
    xd, wd = x.to(dev), wt.to(dev).reshape(c["cout"], -1)
    col = torch.empty((w.K, w.N), device=dev)
    y = torch.empty((w.M, w.N), device=dev)
    ms_col = time_fn(lambda: lib.im2col4d(xd, list(c["ks"]), col=col))
    ms = time_fn(lambda: lib.matmul(wd, col, out=y))
    bytes_gemm = 4 * (w.M * w.K + w.K * w.N + w.M * w.N)
    res["conv4d"] = {"gemm_ms": round(ms, 4), "tflops": round(w.flops / ms / 1e9, 2),
                     "fp32_frac": round(w.flops / ms / 1e9 / fp32_peak, 4),
                     "hbm_frac": round(bytes_gemm / ms / 1e6 / peaks["hbm_gbs"], 4),
                     "im2col_ms": round(ms_col, 4),
                     "im2col_hbm_frac": round(4 * w.K * w.N / ms_col / 1e6 / peaks["hbm_gbs"], 4)}
    del col
    w6 = wt.to(dev)
    ms_imp = time_fn(lambda: lib.conv4d_implicit(xd, w6, out=y))
    res["conv4d_implicit"] = {"ms": round(ms_imp, 4), "tflops": round(w.flops / ms_imp / 1e9, 2),
                              "fp32_frac": round(w.flops / ms_imp / 1e9 / fp32_peak, 4), "bound": "alu",
                              "vs_im2col_plus_gemm": round((ms_col + ms) / ms_imp, 2)}
    # the same convolution on the tensor cores: the same values rounded to bf16, channel-last
    # (one tcgen05 kernel reading the caller's tensors)
    xc, wc = si.channel_last(x, wt, "bf16")
    xcd, wcd = xc.to(dev), wc.to(dev)
    outs = [i - k + 1 for i, k in zip(c["ins"], c["ks"])]
    ycl = torch.empty(outs + [c["cout"]], device=dev)
    ms_tc = time_fn(lambda: lib.conv4d_cl(xcd, wcd, out=ycl))
    res["conv4d_tc_bf16"] = {"ms": round(ms_tc, 4), "tflops": round(w.flops / ms_tc / 1e9, 2),
                             "tensor_frac": round(w.flops / ms_tc / 1e9 / peaks["bf16_tflops"], 4), "bound": "tensor",
                             "layout": "channel-last bf16 in, fp32 out", "vs_fp32_implicit": round(ms_imp / ms_tc, 2)}
    # and from channel-first bf16 operands: one re-layout launch, then the same kernel
    # storing y channel-first
    xb, wb = x.to(torch.bfloat16).to(dev), wt.to(torch.bfloat16).to(dev)
    ycf = torch.empty([c["cout"]] + outs, device=dev)
    ms_cf = time_fn(lambda: lib.conv4d_tc(xb, wb, out=ycf))
    res["conv4d_tc_bf16_channel_first"] = {"ms": round(ms_cf, 4), "tflops": round(w.flops / ms_cf / 1e9, 2),
                                           "tensor_frac": round(w.flops / ms_cf / 1e9 / peaks["bf16_tflops"], 4),
                                           "bound": "tensor", "layout": "channel-first bf16 in, fp32 out",
                                           "launches": 2}
    return res


def measure_e2e(lib, ops, args, dev, world, pg, reps=None):
    """Same metric through the host-buffer C entry point: H2D + GEMM + D2H every step."""
    import torch
    host = []
    h2d = d2h = 0
    for w, Ad, Bd, Cd in ops:
        if w.kind != "gemm":
            continue
        A = Ad.cpu().pin_memory()
        B = Bd.cpu().pin_memory()
        C = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
        host.append((w, A, B, C))
        h2d += A.numel() * A.element_size() + B.numel() * B.element_size()
        d2h += C.numel() * 4
    if not host:
        return None
    n = reps or max(3, min(args.steps, 20))
    pairs = [(A, B) for w, A, B, C in host]
    outs = [C for w, A, B, C in host]
    # one step = the step's products as one host pipeline: a later product's inputs travel
    # while earlier ones compute and their results travel back
    lib.matmul_host_batch(pairs, outs=outs)
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    for _ in range(n):
        lib.matmul_host_batch(pairs, outs=outs)
    dt = reduce_max((time.perf_counter() - t0) / n, pg, dev)
    # the same products one gemm_run_host call at a time, for comparison
    t1 = time.perf_counter()
    for _ in range(max(3, n // 4)):
        for w, A, B, C in host:
            lib.matmul_host(A, B, out=C)
    dt_single = (time.perf_counter() - t1) / max(3, n // 4)
    flops = sum(w.flops for w, *_ in host)
    return {"value": round(world * flops / dt / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(dt * 1e3, 3), "steps": n,
            "api": "gemm_run_host_batch (pinned host buffers)",
            "one_call_per_product_ms": round(dt_single * 1e3, 3)}


def oracle_sample(ops_cpu, rows_per_op):
    """Run the oracle on the first rows of each GEMM; returns (flops, seconds)."""
    import oracle
    flops = 0
    t0 = time.perf_counter()
    for (w, A, B), r in zip(ops_cpu, rows_per_op):
        oracle.gemm(A[:r], B)
        flops += 2 * r * w.N * w.K
    return flops, time.perf_counter() - t0


def cpu_baseline(ops, seconds):
    import numpy as np
    ops_cpu = [(w, Ad.float().cpu().numpy(), Bd.float().cpu().numpy()) for w, Ad, Bd, _ in ops if w.kind == "gemm"]
    if not ops_cpu:
        return None
    # calibrate on a small block, then size the sample to about `seconds`
    f0, t0 = oracle_sample(ops_cpu, [8] * len(ops_cpu))
    rate = f0 / max(t0, 1e-6)
    per_row = sum(2 * w.N * w.K for w, *_ in ops_cpu)
    rows = int(max(8, min(min(w.M for w, *_ in ops_cpu), seconds * rate / per_row)))
    f, t = oracle_sample(ops_cpu, [rows] * len(ops_cpu))
    import oracle
    del np
    return {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": round(t, 2),
            "sample": "first %d rows of each GEMM (%s), full K and N, fp64 accumulation" %
                      (rows, ", ".join(w.name for w, *_ in ops_cpu))}


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    import seeded_inputs as si
    names = [n for n in args.workloads.split(",") if n]
    ops_cpu = []
    for n in names:
        w = si.WORKLOADS[n]
        A, B = si.workload_operands(w)
        ops_cpu.append((w, A.float().numpy(), B.float().numpy()))
    # size one step to a few seconds so warm-up + steps end within a few minutes
    f0, t0 = oracle_sample(ops_cpu, [4] * len(ops_cpu))
    rate = f0 / max(t0, 1e-6)
    per_row = sum(2 * w.N * w.K for w, *_ in ops_cpu)
    budget = args.ref_budget_s / (args.steps + args.warmup)
    rows = int(max(1, min(min(w.M for w, *_ in ops_cpu), budget * rate / per_row)))
    for _ in range(args.warmup):
        oracle_sample(ops_cpu, [rows] * len(ops_cpu))
    times = []
    flops = 0
    for _ in range(args.steps):
        flops, t = oracle_sample(ops_cpu, [rows] * len(ops_cpu))
        times.append(t)
    dt = statistics.mean(times)
    value = flops / dt / 1e12
    sample = "first %d rows of each GEMM (%s) per step, full K and N" % (rows, ", ".join(names))
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "+".join(names), "shapes": {w.name: [w.M, w.N, w.K] for w, *_ in ops_cpu},
                   "parallelism": "CPU oracle, host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.default_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
