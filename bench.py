#!/usr/bin/env python3
"""Benchmark of the tensor-core matrix multiply-accumulate D = A*B + C.

One step runs every part of the path once, at the full workload sizes:

  dense_i8_4096        mma_gemm        i8 4096^3 -> i32
  dense_bf16_8192      mma_gemm        bf16 8192^3 -> f32
  dense_bf16_skinny    mma_gemm        bf16 1024 x 1024 x 65536 (K split)
  sparse_f16_keep02    compress + sparse42_gemm, f16 8192^3, keep-{0,2} pattern
  sparse_f16_random    compress + sparse42_gemm, f16 8192^3, random 2-of-4
  sparse_e4m3_e5m2     compress + sparse42_gemm, E4M3 x E5M2 16384^3
  dense_e4m3_16384     mma_gemm        E4M3 x E4M3 16384^3

The headline value is the suite's throughput in TFLOP/s (2*M*N*K per GEMM with
the uncompressed K, the ops convention of the pages, over the step time);
``per_workload`` gives each GEMM's TFLOP/s and its fraction of the tensor peak
of its type.  Inputs are seeded synthetic matrices resident in HBM; a step
streams several GB, far more than the 126 MB L2, so no explicit flush is used.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the deliberately slow reference
definition) on a bounded row sample of the same workloads.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

from tensor_core_matrix_02_gb300 import workloads as W

SUITE = ["dense_i8_4096", "dense_bf16_8192", "dense_bf16_skinny", "sparse_f16_keep02",
         "sparse_f16_random", "sparse_e4m3_e5m2", "dense_e4m3_16384"]
# nominal dense tensor rate of each input type relative to bf16, and 2x for 4:2-sparse
RATE_VS_BF16 = {"bf16": 1.0, "f16": 1.0, "e4m3": 2.0, "e5m2": 2.0, "i8": 1.0, "u8": 1.0}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(p: W.Problem, pk: dict, sustained: bool = False) -> float:
    """Peak TFLOP/s of the GEMM's input type: measured bf16 x the nominal ratio
    (i8 runs on the bf16 tensor path here, so it takes the bf16 peak).  Each
    kernel is timed as one launch of a few milliseconds, not inside a seconds-long
    step, so the burst figure is the default; the sustained one (a back-to-back
    loop under the power cap) is also reported."""
    base = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return base * RATE_VS_BF16[p.ta] * (2.0 if p.sparse else 1.0)


# ------------------------------------------------------------------ our arm

class Entry:
    """One workload of the step: for 4:2-sparse ones, compression then the GEMM."""

    def __init__(self, name: str, p: W.Problem):
        self.name, self.p = name, p
        self.D = torch.empty_like(p.C)

    def run(self, mm, events=None):
        p = self.p
        if p.sparse:
            if p.sparse == "prune":
                vals, idx = mm.sparse42_prune(p.A)
            else:
                vals, idx = mm.sparse42_compress(p.A)
            if events is not None:
                events.record()
            mm.sparse42_gemm(vals, idx, p.B, p.C, self.D)
        else:
            if events is not None:
                events.record()
            mm.mma_gemm(p.A, p.B, p.C, self.D)

    @property
    def compress_bytes(self):
        """Algorithmic bytes of the compression: read A, write vals and idx."""
        p = self.p
        a = p.A.numel() * p.A.element_size()
        return a + a // 2 + p.M * p.K // 8 if p.sparse else 0

    @property
    def h2d_bytes(self):
        p = self.p
        return sum(t.numel() * t.element_size() for t in (p.A, p.B, p.C))

    @property
    def d2h_bytes(self):
        return self.D.numel() * self.D.element_size()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms; only the
    samples taken inside the timed window (host wall clock) are summarised."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)                      # let the sampler start before the timed work
        except OSError:
            self.proc = None
        return self

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        import datetime
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({nm for r in use for nm, v in zip(self.NAMES, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "sm_mhz_min": min(r[1] for r in use), "reasons": reasons, "samples": len(use),
                "in_window": bool(inside)}


# The source files each GEMM kernel is built from (its template, the shared PTX
# wrappers, and the host code that picks its launch configuration).  A recorded DRAM
# traffic figure stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "gemm_pair_kernel": ["gemm_pair_kernel.cuh", "gemm_pair.cu", "gemm_kernel.cuh"],
    "gemm_sparse_pair_kernel": ["gemm_sparse_pair_kernel.cuh", "gemm_sparse_launch.cuh",
                                "gemm_sparse_f16.cu", "gemm_sparse_f8.cu", "gemm_kernel.cuh"],
}
COMMON_SOURCES = ["ptx.cuh", "gemm_args.h", "launch.h", "api.cu"]


def source_digest(kernel: str) -> str:
    family = kernel.split("<")[0]
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_core_matrix_02_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[family] + COMMON_SOURCES):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (None otherwise)."""
    try:
        with open(TRAFFIC_PATH) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get(f"{kernel}:{workload}")
    if not rec or rec.get("source_digest") != source_digest(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def kernel_of(p: W.Problem) -> tuple[str, str]:
    """(name used in the JSON line, regex matching the demangled ncu kernel name)."""
    kind = "f8f6f4" if p.ta in ("e4m3", "e5m2") else "f16"
    if p.sparse:
        return f"gemm_sparse_pair_kernel<{kind}>", "gemm_sparse_pair_kernel"
    return f"gemm_pair_kernel<{kind}>", "gemm_pair_kernel"


def algorithmic_bytes(p: W.Problem) -> int:
    """Bytes the GEMM kernel must move at least: read its operands and C once, write D."""
    a = p.M * p.K * (1 if p.ta in ("e4m3", "e5m2", "i8", "u8") else 2)
    if p.sparse:
        a = a // 2 + p.M * p.K // 8           # compressed values and the 2-bit index
    b = p.K * p.N * (1 if p.tb in ("e4m3", "e5m2", "i8", "u8") else 2)
    return a + b + 2 * p.M * p.N * (2 if p.tacc in ("f16", "bf16") else 4)


def graph_per_call(fn, calls: int = 200, reps: int = 5):
    """Device time per call of `calls` back-to-back calls captured in one CUDA graph
    (warm inputs; the host's per-call cost is out of the picture), median of `reps`
    replays; (None, reason) if the calls cannot be captured."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn(); fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                fn()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); g.replay(); b.record(); torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / calls)
        ts.sort()
        return round(ts[len(ts) // 2], 3), f"{calls} calls in one CUDA graph, median of {reps} replays"
    except Exception as e:   # a capture the driver refuses: report it, keep the run
        torch.cuda.synchronize()
        return None, f"not captured: {str(e).splitlines()[0][:120]}"


def small_case(mm, dev, hbm_gbs: float, reps: int = 21) -> dict:
    """The smallest configuration (dense f16 128 x 128 x 256, one tile: launch- and
    latency-bound) timed per call on the device, warm (inputs in L2) and cold (L2
    flushed by writing a buffer twice its size first).  A device-side sleep ahead of
    each timed call keeps the host's launch latency out of the measurement."""
    p = W.make("dense_f16_128", device=dev)
    D = torch.empty_like(p.C)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for mode in ("warm", "cold"):
        ts = []
        for _ in range(reps):
            mm.mma_gemm(p.A, p.B, p.C, D)
            if mode == "cold":
                flush.fill_(1)
            torch.cuda._sleep(200000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            mm.mma_gemm(p.A, p.B, p.C, D)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        ts.sort()
        out[f"us_{mode}"] = round(ts[len(ts) // 2], 2)
    out["us_per_call_in_graph"], out["graph_note"] = graph_per_call(lambda: mm.mma_gemm(p.A, p.B, p.C, D))
    byts = algorithmic_bytes(p)
    gbs = {m: byts / (out[f"us_{m}"] * 1e-6) / 1e9 for m in ("warm", "cold")}
    return {"workload": "dense_f16_128", "M": p.M, "N": p.N, "K": p.K, **out,
            "algorithmic_bytes": byts, "gbs_warm": round(gbs["warm"], 1), "gbs_cold": round(gbs["cold"], 1),
            "frac_of_hbm_warm": round(gbs["warm"] / hbm_gbs, 5), "frac_of_hbm_cold": round(gbs["cold"] / hbm_gbs, 5),
            "tflops_warm": round(p.flops / (out["us_warm"] * 1e-6) / 1e12, 3),
            "what": "us_warm / us_cold: median of 21 single calls, each queued behind a device-side sleep "
                    "(event times here move in steps of about 2 us); us_per_call_in_graph: back-to-back calls"}


def record_traffic(args):
    """Read an ncu CSV (--metrics dram__bytes_read.sum,dram__bytes_write.sum,
    gpu__time_duration.sum) of one workload's GEMM launches and store the DRAM
    bytes per launch, with the digest of the kernel's sources, in traffic.json."""
    if not args.workloads or len(args.workloads) != 1:
        raise SystemExit("--record-traffic needs exactly one --workloads entry")
    name = args.workloads[0]
    r = W.RECIPES[name]
    prob = W.Problem(name, r.M, r.N, r.K, r.ta, r.tb, r.tacc, None, None, None, r.sparse, None)
    kernel, pattern = kernel_of(prob)
    need = ("dram__bytes_read.sum", "dram__bytes_write.sum")
    got = [m for m in _ncu_launches(args.record_traffic, pattern) if all(k in m for k in need)]
    if not got:
        raise SystemExit(f"no {pattern} launch with DRAM counters in {args.record_traffic}")
    rd = sum(m["dram__bytes_read.sum"] for m in got) / len(got)
    wr = sum(m["dram__bytes_write.sum"] for m in got) / len(got)
    dur = [m["gpu__time_duration.sum"] * 1e-9 for m in got if "gpu__time_duration.sum" in m]
    try:
        with open(TRAFFIC_PATH) as f:
            d = json.load(f)
    except (OSError, ValueError):
        d = {}
    d[f"{kernel}:{name}"] = {
        "dram_bytes_per_launch": int(rd + wr), "dram_read": int(rd), "dram_write": int(wr),
        "algorithmic_bytes": algorithmic_bytes(prob), "launches": len(got),
        "ncu_duration_s": (sum(dur) / len(dur)) if dur else None,
        "source_digest": source_digest(kernel), "csv": os.path.basename(args.record_traffic)}
    with open(TRAFFIC_PATH, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    print(json.dumps(d[f"{kernel}:{name}"]))


NCU_PATH = os.path.join(ROOT, "profiles", "ncu.json")
# the counters kept per GEMM kernel and workload (one ncu pass group, a few passes)
NCU_METRICS = ("gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
               "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
               "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "sm__cycles_elapsed.avg.per_second")


# ncu prints a metric in the unit its "Metric Unit" column names, scaled by magnitude
# in some outputs (SI prefixes): values are brought to bytes, nanoseconds and hertz
NCU_UNIT_SCALE = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
                  "ns": 1.0, "nsecond": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6,
                  "s": 1e9, "second": 1e9,
                  "hz": 1.0, "khz": 1e3, "mhz": 1e6, "ghz": 1e9,
                  "%": 1.0, "": 1.0}


def _ncu_launches(csv_path: str, pattern: str) -> list[dict]:
    """Per-launch metric dictionaries of the kernels matching ``pattern`` in an ncu
    CSV (``--csv`` output of ``--metrics``), in base units (an unknown unit is an
    error, not a silent misreading)."""
    import csv
    with open(csv_path) as f:
        rows = [ln for ln in f if ln.startswith('"')]
    launches = {}
    for row in csv.DictReader(rows):
        if pattern not in row["Kernel Name"]:
            continue
        m = launches.setdefault(row["ID"], {})
        try:
            v = float(row["Metric Value"].replace(",", ""))
        except ValueError:
            continue
        unit = row.get("Metric Unit", "").strip().lower()
        if unit not in NCU_UNIT_SCALE:
            raise SystemExit(f"{csv_path}: {row['Metric Name']} in unknown unit {unit!r}")
        m[row["Metric Name"]] = v * NCU_UNIT_SCALE[unit]
    return list(launches.values())


def record_ncu(args):
    """Read an ncu CSV of one workload's GEMM launches (the NCU_METRICS counters)
    and store their per-launch means, with the kernel's source digest and the
    captured shape, in profiles/ncu.json."""
    if not args.workloads or len(args.workloads) != 1:
        raise SystemExit("--record-ncu needs exactly one --workloads entry")
    name = args.workloads[0]
    r = W.RECIPES[name]
    M, N, K = args.shape if args.shape else (r.M, r.N, r.K)
    prob = W.Problem(name, M, N, K, r.ta, r.tb, r.tacc, None, None, None, r.sparse, None)
    kernel, pattern = kernel_of(prob)
    got = [m for m in _ncu_launches(args.record_ncu, pattern) if all(k in m for k in NCU_METRICS)]
    if not got:
        raise SystemExit(f"no {pattern} launch with the ncu counters in {args.record_ncu}")
    mean = {k: sum(m[k] for m in got) / len(got) for k in NCU_METRICS}
    dur = mean["gpu__time_duration.sum"] * 1e-9
    rd, wr = mean["dram__bytes_read.sum"], mean["dram__bytes_write.sum"]
    try:
        with open(NCU_PATH) as f:
            d = json.load(f)
    except (OSError, ValueError):
        d = {}
    pk, _ = peaks()
    d[f"{kernel}:{name}"] = {
        "shape": [M, N, K], "launches": len(got), "ncu_duration_us": round(dur * 1e6, 2),
        "sm_mhz": round(mean["sm__cycles_elapsed.avg.per_second"] / 1e6, 1),
        "tensor_pipe_active_pct": round(mean["sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed"], 2),
        "dram_read": int(rd), "dram_write": int(wr), "dram_gbs": round((rd + wr) / dur / 1e9, 1),
        "dram_frac_of_hbm": round((rd + wr) / dur / 1e9 / pk["hbm_gbs"], 4),
        "dram_throughput_pct": round(mean["gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed"], 2),
        "algorithmic_bytes": algorithmic_bytes(prob),
        "tflops_under_ncu": round(prob.flops / dur / 1e12, 1),
        "source_digest": source_digest(kernel), "csv": os.path.basename(args.record_ncu)}
    with open(NCU_PATH, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    print(json.dumps(d[f"{kernel}:{name}"]))


def recorded_ncu(kernel: str, workload: str):
    """The committed ncu counters of this kernel on this workload, if they were
    taken on the current kernel sources (None otherwise)."""
    try:
        with open(NCU_PATH) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get(f"{kernel}:{workload}")
    if not rec or rec.get("source_digest") != source_digest(kernel):
        return None
    return {k: v for k, v in rec.items() if k not in ("source_digest", "csv")}


def cpu_sample(problems, frac_rows: int, oracle_mod):
    """Time the oracle on every frac_rows-th row of each workload; returns
    (flops of the sample, seconds, threads, description)."""
    flops, secs = 0, 0.0
    for name, p in problems:
        rows = list(range(0, p.M, frac_rows))
        A = p.A[rows].cpu()
        B = W.bits(p.B.cpu())
        C = p.C[rows].cpu().numpy()
        t0 = time.perf_counter()
        if p.sparse:
            step = oracle_mod.prune if p.sparse == "prune" else oracle_mod.compress
            vals, idx, _ = step(W.bits(A), p.ta)
            oracle_mod.sparse_gemm(vals, idx, p.ta, B, p.tb, C, p.K)
        else:
            oracle_mod.gemm(W.bits(A), p.ta, B, p.tb, C)
        secs += time.perf_counter() - t0
        flops += 2 * len(rows) * p.N * p.K
    desc = f"every {frac_rows}th row of each suite workload (all columns, full K)"
    return flops, secs, oracle_mod.num_threads(), desc


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
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
    import platform
    return platform.machine()


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def run_ours(args):
    from tensor_core_matrix_02_gb300 import build, mma42
    dist, rank, world, local = dist_setup(args.gpus)
    build.build()
    mm = mma42
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    names = args.workloads or SUITE
    shape = dict(zip("MNK", args.shape)) if args.shape else {}
    entries = [Entry(n, W.make(n, device=dev, **shape)) for n in names]
    pk, pk_src = peaks()

    for _ in range(args.warmup):
        for e in entries:
            e.run(mm)
    if mm.mma_sync_status() != 0:
        raise RuntimeError("device error during warm-up")

    starts = [[torch.cuda.Event(enable_timing=True) for _ in entries] for _ in range(args.steps)]
    mids = [[torch.cuda.Event(enable_timing=True) for _ in entries] for _ in range(args.steps)]
    ends = [[torch.cuda.Event(enable_timing=True) for _ in entries] for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = mm.mma_launch_count()
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        w0 = time.time()
        t_begin.record()
        for s in range(args.steps):
            for i, e in enumerate(entries):
                starts[s][i].record()
                e.run(mm, mids[s][i])      # mid: after compression, before the GEMM
                ends[s][i].record()
        t_end.record()
        torch.cuda.synchronize()
        clocks.mark(w0, time.time())
    barrier(dist)
    launches = mm.mma_launch_count() - launches0
    if mm.mma_sync_status() != 0:
        raise RuntimeError("device error during the timed steps")
    total_ms = max_over_ranks(dist, t_begin.elapsed_time(t_end), dev)
    step_flops = sum(e.p.flops for e in entries)
    value = world * step_flops * args.steps / (total_ms * 1e-3) / 1e12

    # the warp-level (mma.sync / mma.sp) tensor path's ceilings on this GPU, measured
    # after the timed region: the i8 GEMM runs on bf16 tcgen05 because this path is
    # the only one with an 8-bit integer multiply here
    legacy = {k: mm.mma_legacy_mma_peak(k) / 1e12 for k in mm.LEGACY_KINDS}
    # tcgen05.mma's own ceilings, also measured after the timed region: ops per SM clock
    # of each kind on operands resident in shared memory.  The nominal peak of a type is
    # SMs x that rate x the maximum SM clock; the kernels' fractions of it show how
    # well their pipelines feed the tensor cores, whatever the clock.
    tc = {k: mm.mma_tcgen05_peak(k) for k in mm.TCGEN05_KINDS}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = float(pk.get("sm_max_mhz", 2070.0))
    nominal = {k: sms * clk * max_mhz * 1e6 / 1e12 for k, (_, clk) in tc.items()}

    def tc_kind(p):
        # the 8-bit integer GEMMs run on bf16 operands
        return ("e4m3" if p.ta in ("e4m3", "e5m2") else "bf16") + ("_sparse" if p.sparse else "")
    small = small_case(mm, dev, pk["hbm_gbs"]) if not args.shape else None

    def legacy_kind(p):
        if p.ta in ("i8", "u8"):
            return "s8_sparse" if p.sparse else "s8"
        if p.sparse:
            return None
        return "bf16" if p.ta in ("f16", "bf16") else "e4m3"

    per = []
    for i, e in enumerate(entries):
        ms = sum(starts[s][i].elapsed_time(ends[s][i]) for s in range(args.steps)) / args.steps
        gemm_ms = sum(mids[s][i].elapsed_time(ends[s][i]) for s in range(args.steps)) / args.steps
        tf = e.p.flops / (gemm_ms * 1e-3) / 1e12
        peak = tensor_peak(e.p, pk)
        rec = {"workload": e.name, "M": e.p.M, "N": e.p.N, "K": e.p.K,
               "types": f"{e.p.ta}x{e.p.tb}->{e.p.tacc}", "sparse": e.p.sparse,
               "ms": round(ms, 4), "gemm_ms": round(gemm_ms, 4), "tflops": round(tf, 1),
               "peak_tflops": round(peak, 1), "frac_of_peak": round(tf / peak, 4),
               "frac_of_sustained_peak": round(tf / tensor_peak(e.p, pk, sustained=True), 4)}
        rec["frac_of_nominal_peak"] = round(tf / nominal[tc_kind(e.p)], 4)
        # ncu counters of this GEMM's kernel (one launch, cold, serialised; taken on
        # the shape named in the record), when captured on the current sources
        rec["ncu"] = recorded_ncu(kernel_of(e.p)[0], e.name) if not args.shape else None
        lk = legacy_kind(e.p)
        if lk:
            rec["vs_legacy_mma_peak"] = round(tf / legacy[lk], 3)
        if e.p.sparse:
            cms = ms - gemm_ms
            gbs = e.compress_bytes / (cms * 1e-3) / 1e9
            rec.update({"compress_ms": round(cms, 4), "compress_gbs": round(gbs, 1),
                        "compress_frac_of_hbm": round(gbs / pk["hbm_gbs"], 4)})
        per.append(rec)
    dom = max(range(len(entries)), key=lambda i: per[i]["gemm_ms"])
    dp = entries[dom].p
    kernel, _ = kernel_of(dp)
    achieved = per[dom]["tflops"]
    peak = tensor_peak(dp, pk)
    roofline = {"bound": "tensor", "kernel": kernel, "workload": entries[dom].name,
                "achieved": achieved, "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "frac_of_sustained_peak": round(achieved / tensor_peak(dp, pk, sustained=True), 4),
                "frac_of_nominal_peak": round(achieved / nominal[tc_kind(dp)], 4),
                "peak_source": f"{pk_src} bf16 burst x {RATE_VS_BF16[dp.ta] * (2 if dp.sparse else 1):g} (nominal type ratio); "
                               "frac_of_nominal_peak: SMs x measured tcgen05 ops per clock x the maximum SM clock",
                "traffic": recorded_traffic(kernel, entries[dom].name) if not args.shape else None,
                "algorithmic_bytes": algorithmic_bytes(dp)}

    # end to end through the public API: pinned host inputs -> device -> call -> host result
    e2e = None
    if not args.no_e2e:
        host_in = [(e.p.A.cpu().pin_memory(), e.p.B.cpu().pin_memory(), e.p.C.cpu().pin_memory()) for e in entries]
        host_out = [torch.empty(e.D.shape, dtype=e.D.dtype).pin_memory() for e in entries]
        # two sets of device buffers, used by alternate steps, so that one step's
        # uploads can run while the step before computes and downloads
        dev_in = [[(torch.empty_like(e.p.A), torch.empty_like(e.p.B), torch.empty_like(e.p.C)) for e in entries]
                  for _ in range(2)]
        dev_res = [[e.D for e in entries], [torch.empty_like(e.D) for e in entries]]

        # Uploads, compute and downloads on three streams: workload w+1's inputs go up
        # and workload w-1's result comes down while workload w computes, and the next
        # step's uploads start while this step still computes.  The host link carries
        # ~200 GB/s each way and is the bound, so the workloads go in order of
        # decreasing result size: the large downloads overlap later uploads and the
        # step ends on a small one.
        comp = torch.cuda.current_stream()
        upload, download = torch.cuda.Stream(), torch.cuda.Stream()
        order = sorted(range(len(entries)), key=lambda w: -entries[w].d2h_bytes)
        computed = [dict(), dict()]    # set -> workload -> event: its last compute finished
        fetched = [dict(), dict()]     # set -> workload -> event: its last result download finished

        def e2e_step(step):
            k = step % 2
            up = {w: torch.cuda.Event() for w in order}
            with torch.cuda.stream(upload):
                for w in order:
                    if w in computed[k]:                  # the step two back has read these inputs
                        upload.wait_event(computed[k][w])
                    for src, dst in zip(host_in[w], dev_in[k][w]):
                        dst.copy_(src, non_blocking=True)
                    up[w].record(upload)
            for w in order:
                e = entries[w]
                da, db, dc = dev_in[k][w]
                comp.wait_event(up[w])
                if w in fetched[k]:                       # the step two back's result has left
                    comp.wait_event(fetched[k][w])
                if e.p.sparse:
                    vals, idx = mm.sparse42_prune(da) if e.p.sparse == "prune" else mm.sparse42_compress(da)
                    mm.sparse42_gemm(vals, idx, db, dc, dev_res[k][w])
                else:
                    mm.mma_gemm(da, db, dc, dev_res[k][w])
                done = torch.cuda.Event()
                done.record(comp)
                computed[k][w] = done
                download.wait_event(done)
                with torch.cuda.stream(download):
                    host_out[w].copy_(dev_res[k][w], non_blocking=True)
                    got = torch.cuda.Event()
                    got.record(download)
                fetched[k][w] = got

        for i in range(max(2, min(args.warmup, 2))):
            e2e_step(i)
        comp.wait_stream(download)
        # the first step's uploads and the last step's downloads overlap nothing: 16
        # steps keep that fill and drain to a small part of the run (~0.5 s)
        e2e_steps = max(1, min(args.steps, 16))
        barrier(dist)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(e2e_steps):
            e2e_step(i)
        comp.wait_stream(download)                 # the run ends when every result is on the host
        b.record()
        torch.cuda.synchronize()
        barrier(dist)
        e2e_ms = max_over_ranks(dist, a.elapsed_time(b), dev)
        # the host link on these buffers, alone: the largest input up, the largest result down
        big_in = max((t for trio in host_in for t in trio), key=lambda t: t.numel() * t.element_size())
        dev_big = max((t for trio in dev_in[0] for t in trio), key=lambda t: t.numel() * t.element_size())
        big_out = max(host_out, key=lambda t: t.numel() * t.element_size())
        dev_out = max((e.D for e in entries), key=lambda t: t.numel() * t.element_size())

        def link_gbs(dst, src):
            n = min(dst.numel() * dst.element_size(), src.numel() * src.element_size())
            d8, s8 = dst.view(-1).view(torch.uint8)[:n], src.view(-1).view(torch.uint8)[:n]
            d8.copy_(s8, non_blocking=True)
            la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            la.record()
            d8.copy_(s8, non_blocking=True)
            lb.record()
            torch.cuda.synchronize()
            return n / (la.elapsed_time(lb) * 1e-3) / 1e9

        def both_gbs():
            """Both directions at once (the largest input up on one stream, the largest
            result down on another): their summed bytes over the time both take."""
            n_up = min(dev_big.numel() * dev_big.element_size(), big_in.numel() * big_in.element_size())
            n_dn = min(big_out.numel() * big_out.element_size(), dev_out.numel() * dev_out.element_size())
            up8 = (dev_big.view(-1).view(torch.uint8)[:n_up], big_in.view(-1).view(torch.uint8)[:n_up])
            dn8 = (big_out.view(-1).view(torch.uint8)[:n_dn], dev_out.view(-1).view(torch.uint8)[:n_dn])
            t = None
            for _ in range(2):                      # the first pass warms up
                la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                la.record(comp)
                for st, (dst, src) in ((upload, up8), (download, dn8)):
                    st.wait_event(la)
                    with torch.cuda.stream(st):
                        dst.copy_(src, non_blocking=True)
                comp.wait_stream(upload)
                comp.wait_stream(download)
                lb.record(comp)
                torch.cuda.synchronize()
                t = la.elapsed_time(lb) * 1e-3
            return (n_up + n_dn) / t / 1e9

        h2d_gbs = link_gbs(dev_big, big_in)
        d2h_gbs = link_gbs(big_out, dev_out)
        bidir_gbs = both_gbs()
        h2d_total = sum(e.h2d_bytes for e in entries)
        d2h_total = sum(e.d2h_bytes for e in entries)
        # the step cannot beat the host link: each direction at its own rate, and
        # both together at their measured combined rate
        link_floor_s = max(h2d_total / (h2d_gbs * 1e9), d2h_total / (d2h_gbs * 1e9),
                           (h2d_total + d2h_total) / (bidir_gbs * 1e9))
        e2e = {"value": round(world * step_flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
               "link_gbs": {"h2d": round(h2d_gbs, 1), "d2h": round(d2h_gbs, 1), "both": round(bidir_gbs, 1)},
               "upload_floor_ms": round(h2d_total / (h2d_gbs * 1e9) * 1e3, 3),
               "link_floor_ms": round(link_floor_s * 1e3, 3),
               "h2d_bytes_per_step": sum(e.h2d_bytes for e in entries),
               "d2h_bytes_per_step": sum(e.d2h_bytes for e in entries), "steps": e2e_steps,
               "ms_per_step": round(e2e_ms / e2e_steps, 3),
               "schedule": "pinned host buffers; uploads, compute and downloads overlapped on three streams, "
                           "largest result first; two sets of device buffers let a step's uploads overlap "
                           "the step before"}
        del host_in, host_out, dev_in, dev_res

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:   # the CPU baseline is an N = 1 figure
        import oracle
        f, s, thr, desc = cpu_sample([(e.name, e.p) for e in entries], args.cpu_rows, oracle)
        cpu = {"value": round(f / s / 1e12, 6), "unit": "TFLOP/s", "cores": thr, "cpu_model": cpu_model(),
               "kind": "oracle", "sample": desc, "seconds": round(s, 2)}

    if rank == 0:
        line = {"metric": "GEMM TFLOP/s per dtype, dense and 4:2-sparse, as % of GB300 tensor peak",
                "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "mixed: i8(bf16 path)->i32, bf16->f32, f16->f32, e4m3/e5m2->f32",
                "data": "synthetic, seeded",
                "config": {"workload": "suite: " + ",".join(names) + (f" at {args.shape}" if args.shape else ""),
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                           "l2": "inputs of one step stream several GB (> 126 MB L2); no flush"},
                "per_workload": per, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches), "clocks": clocks.summary(),
                "small_case": small,
                "legacy_mma_peaks": {"unit": "TOPS", **{k: round(v, 1) for k, v in legacy.items()},
                                     "what": "warp-level mma.sync / mma.sp ceilings measured in this run "
                                             "(every SM, operands in registers); per_workload.vs_legacy_mma_peak "
                                             "sets each GEMM against the one of its type"},
                "tcgen05_peaks": {"unit": "TFLOP/s",
                                  "ops_per_clk_sm": {k: round(c, 1) for k, (_, c) in tc.items()},
                                  "nominal_tflops": {k: round(v, 1) for k, v in nominal.items()},
                                  "burst_tflops": {k: round(o / 1e12, 1) for k, (o, _) in tc.items()},
                                  "what": "tcgen05.mma ceilings measured in this run (every SM pair, the pair "
                                          "kernels' instruction shapes, operands resident in shared memory); "
                                          "nominal = SMs x ops per SM clock x the maximum SM clock; "
                                          "per_workload.frac_of_nominal_peak sets each GEMM against its kind's"},
                "impl": "ours"}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_aux(args):
    """Bandwidth of the steps around the GEMMs, at the full sizes: 4:2 compression,
    pruning and quantisation, against the measured HBM copy bandwidth."""
    from tensor_core_matrix_02_gb300 import build, mma42 as mm
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_src = peaks()
    cases = []
    for wl in ("sparse_f16_random", "sparse_e4m3_e5m2"):
        A = W.make(wl, device=dev).A
        nb = A.numel() * A.element_size()
        cases.append((f"compress {wl}", lambda A=A: mm.sparse42_compress(A), nb + nb // 2 + A.numel() // 8))
    for wl in ("dense_bf16_8192", "dense_e4m3_16384"):
        A = W.make(wl, device=dev).A
        nb = A.numel() * A.element_size()
        cases.append((f"prune {wl}", lambda A=A: mm.sparse42_prune(A), nb + nb // 2 + A.numel() // 8))
    g = torch.Generator(device=dev).manual_seed(7)
    for n_side, dt in ((16384, torch.float8_e4m3fn), (8192, torch.bfloat16)):
        x = torch.randn((n_side, n_side), generator=g, device=dev)
        y = torch.empty(x.shape, dtype=dt, device=dev)
        cases.append((f"quantize f32 -> {str(dt).split('.')[-1]} {n_side}^2",
                      lambda x=x, y=y, dt=dt: mm.mma_quantize(x, dt, y), x.numel() * (4 + y.element_size())))
    for n_side, dt in ((16384, torch.float8_e4m3fn), (8192, torch.float16)):
        x = torch.randn((n_side, n_side), generator=g, device=dev)
        esz = torch.empty(0, dtype=dt).element_size()
        cases.append((f"quantize+prune f32 -> {str(dt).split('.')[-1]} {n_side}^2",
                      lambda x=x, dt=dt: mm.sparse42_quantize_prune(x, dt),
                      x.numel() * 4 + x.numel() // 2 * esz + x.numel() // 8))
    out = []
    for name, fn, nbytes in cases:
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.append({"step": name, "ms": round(ms, 4), "bytes": int(nbytes), "gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4)})
    if mm.mma_sync_status() != 0:
        raise RuntimeError("device error in the bandwidth steps")
    print(json.dumps({"aux": out, "hbm_gbs": pk["hbm_gbs"], "peak_source": pk_src,
                      "note": "inputs larger than L2 (>= 128 MB each); algorithmic bytes: read input, write output"}))


# Stage shapes for the TMA feed probe: (label, [(rows, row bytes) per box], stages)
FEED_STAGES = [
    ("4:2 f16, 64-byte compressed-A rows, index box, two B chunks", [(128, 64), (8, 256), (64, 128), (64, 128)], 7),
    ("4:2 FP8, 64-byte compressed-A rows, index box, one B chunk", [(128, 64), (16, 256), (128, 128)], 6),
    ("dense bf16 (A, two B chunks)", [(128, 128), (64, 128), (64, 128)], 6),
    ("dense FP8 (A, one B chunk)", [(128, 128), (128, 128)], 6),
    ("4:2 f16, 128-byte rows, index box, two B chunks", [(128, 128), (16, 256), (128, 128), (128, 128)], 4),
    ("4:2 FP8, 128-byte rows, index box, one B chunk", [(128, 128), (32, 256), (256, 128)], 3),
    ("4:2 f16, 128-byte rows, B chunks in one box (index in registers)", [(128, 128), (256, 128)], 4),
    ("4:2 FP8, 128-byte rows (index in registers)", [(128, 128), (256, 128)], 4),
]


def run_feed_probe(args):
    """The TMA fill rate of a CTA pair's ring for the kernels' stage shapes and for
    1-4 boxes of 64/128/256-byte rows: one JSON line per case."""
    from tensor_core_matrix_02_gb300 import build, mma42 as mm
    build.build()
    torch.cuda.set_device(0)
    cases = []
    for src in (64 << 20, 1 << 30):
        for label, boxes, st in FEED_STAGES:
            for cl in (0, 19):
                cases.append((label, boxes, st, cl, src))
    for rows, rb in ((128, 64), (128, 128), (64, 128), (16, 256)):
        for n in (1, 2, 3, 4):
            boxes = [(rows, rb)] * n
            sb = rows * rb * n
            for kb in (96, 196):
                cases.append((f"{n} x ({rows} rows x {rb} B)", boxes, max(2, min(16, kb * 1024 // sb)), 0, 64 << 20))
    for label, boxes, st, cl, src in cases:
        b, r = mm.mma_tma_feed_probe(boxes, st, clusters=cl, src_bytes=src)
        sb = sum(x * y for x, y in boxes)
        print(json.dumps({"stage": label, "boxes": boxes, "stages": st, "pairs": cl or "all", "source_mb": src >> 20,
                          "stage_bytes": sb, "bytes_per_clk_sm": round(b, 2), "rows_per_clk_sm": round(r, 4),
                          "clocks_per_stage": round(sb / b, 1)}), flush=True)
    if mm.mma_sync_status() != 0:
        raise RuntimeError("device error in the feed probe")


def run_reference(args):
    """The oracle, as it stands, on the host cores; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    names = args.workloads or SUITE
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"   # input drawing only; the oracle runs on the host
    problems = [(n, W.make(n, device=gen_dev)) for n in names]
    for _ in range(args.warmup):
        cpu_sample(problems, args.ref_rows, oracle)
    flops, secs = 0, 0.0
    for _ in range(args.steps):
        f, s, thr, desc = cpu_sample(problems, args.ref_rows, oracle)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {"metric": "GEMM TFLOP/s per dtype, dense and 4:2-sparse, as % of GB300 tensor peak",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/i64 (oracle)",
            "data": "synthetic, seeded", "config": {"workload": "suite: " + ",".join(names)},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workloads", nargs="*", default=None, help="subset of the suite")
    ap.add_argument("--shape", type=lambda t: [int(x) for x in t.split(",")], default=None,
                    help="M,N,K override for every selected workload (small profiling cases)")
    ap.add_argument("--cpu-rows", type=int, default=24, help="oracle sample: every n-th row")
    ap.add_argument("--ref-rows", type=int, default=512, help="reference arm sample: every n-th row")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--feed-probe", action="store_true",
                    help="TMA fill rate of the pair kernels' ring for their stage shapes (measurement helper)")
    ap.add_argument("--aux", action="store_true",
                    help="time only the bandwidth-bound steps (compression, pruning, quantisation)")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="store the DRAM bytes per launch of one workload's GEMM from an ncu CSV; no GPU")
    ap.add_argument("--record-ncu", metavar="CSV", default=None,
                    help="store one workload's GEMM counters (tensor pipe, DRAM) from an ncu CSV; no GPU")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args)
        return
    if args.record_ncu:
        record_ncu(args)
        return
    if args.aux:
        run_aux(args)
        return
    if args.feed_probe:
        run_feed_probe(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
