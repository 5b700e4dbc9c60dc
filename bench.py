"""Benchmark: tridiagonal eigenproblems per second on one GB300 (or N, one
process per GPU, each solving its own batch: weak scaling), with the achieved
fraction of the ALU roofline.

A step is one solve of the headline workload (float32, n = 16, jobz = V,
batch 32,768, d and e i.i.d. N(0,1) from seed 0): load, scale, settle, chase,
Q accumulation, sort and store, all in one kernel launch.  The companion
workloads of the same family (float32 n = 8 / 16, jobz V / N, and float64
n = 12 V / N) are timed the same way and reported under "workloads".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Inputs are generated on the host, copied to the device before the timed
region, restored before every step (the solve overwrites d) and L2 is
flushed by writing a 256 MiB buffer between steps.  Each step is timed with
CUDA events on the solve's stream.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from symmetric_tridiagonal_eigensolver_gb300 import inputs  # noqa: E402

METRIC = "tridiagonal eigenproblems/sec (n<=32, f32/f64, jobz V/N) and % of roofline"
UNIT = "problems/s"
HEADLINE = dict(dtype="float32", n=16, batch=32768, jobz=True)
COMPANIONS = [dict(dtype="float32", n=8, batch=65536, jobz=True),
              dict(dtype="float32", n=8, batch=65536, jobz=False),
              dict(dtype="float32", n=16, batch=32768, jobz=False),
              dict(dtype="float64", n=12, batch=32768, jobz=True),
              dict(dtype="float64", n=12, batch=32768, jobz=False)]
# The small case (float32 n = 4, batch 1,024, V) and the mixed hard-case
# batch at n = 32 in both precisions and both jobz.
SMALL_CASE = dict(dtype="float32", n=4, batch=1024, jobz=True)
MIXED = [dict(dtype=dt, n=32, batch=32768, jobz=jz, kind="mixed")
         for dt in ("float32", "float64") for jz in (True, False)]
# Context only: steqr_cta float n=16 V, batch 32,768, flat solver, RTX 4090
# (BatchLAS perf_steqr, "What ships" table: 450.9 us per call).
PAGES_BASELINE = 32768 / 450.9e-6
# DRAM bytes (read + write) per launch measured by ncu for a kernel variant,
# keyed by bstq_describe()'s text and the digest of the kernel's sources
# (kernel_digest()); a changed kernel no longer matches and reports null
# (profiles/split_f32_n16_V_batch32768.md).
NCU_TRAFFIC = {
    ("lane<f32,16,V,split,flat> tpb=512 grid=152 smem=207984 regs=128 work=131072", "ff1529af89771e95"):
        4.302848e6 + 0.148224e6,
}


# Translation unit of the headline kernel (split roles, float, n <= 16, V).
HEADLINE_UNIT = "bstq_kern_split_f32_v16.cu"


def _source_dirs():
    """Hand-written CUDA sources and the generated instantiation units (the
    build writes those; they are regenerated here if missing)."""
    from symmetric_tridiagonal_eigensolver_gb300 import build as _b
    if not os.path.exists(os.path.join(_b.GEN, "bstq_registry_list.inc")):
        _b.generate()
    return [_b.CSRC, _b.GEN]


def _find_source(f):
    for d in _source_dirs():
        if os.path.exists(os.path.join(d, f)):
            return os.path.join(d, f)
    return None


def kernel_sources(unit: str = HEADLINE_UNIT) -> list:
    """The CUDA sources a kernel's translation unit compiles: the unit and
    every header it includes with quotes, followed recursively; names in
    order."""
    import re
    seen, todo = set(), [unit]
    while todo:
        f = todo.pop()
        path = _find_source(f)
        if f in seen or path is None:
            continue
        seen.add(f)
        with open(path) as fh:
            todo.extend(re.findall(r'^\s*#\s*include\s+"([^"]+)"', fh.read(), flags=re.M))
    return sorted(seen)


def kernel_digest(unit: str = HEADLINE_UNIT) -> str:
    """Short SHA-256 over kernel_sources(unit), names and contents.  Launch
    shape, registers and shared memory are in bstq_describe()'s text, the
    other half of the traffic key."""
    import hashlib
    h = hashlib.sha256()
    for f in kernel_sources(unit):
        h.update(f.encode())
        with open(_find_source(f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


SM_FP32_LANES = 128     # FP32 FMA lanes per SM (Blackwell SM)
SM_FP64_LANES = 2       # FP64 FMA lanes per SM on GB300 (1.25 TFLOP/s nominal)


def aggregate(local_ms, local_problems, world, dist=None, device="cpu"):
    """Whole-job numbers over ranks: the slowest rank's time (max) and the
    problems all ranks solved (sum).  world == 1 needs no process group."""
    if world == 1:
        return float(local_ms), int(local_problems)
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    c = torch.tensor([float(local_problems)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return float(t.item()), int(round(c.item()))


def rank_seed(rank):
    """Each rank solves its own batch (weak scaling): seed = rank."""
    return int(rank)


def wl_name(w):
    kind = "mixed hard cases" if w.get("kind", "normal") == "mixed" else "N(0,1)"
    return f"{w['dtype']} n={w['n']} jobz={'V' if w['jobz'] else 'N'} batch={w['batch']} {kind} seed 0"


def algorithmic(w, counts):
    """Algorithmic flops and bytes of one solve of workload w.
    flops = R (40 + 6n [V]) + S 12 + D2 (25 + 6n [V]) with R rotations, S
    implicit steps and D2 2x2 solves counted by the oracle on the same input;
    bytes = batch ((3n - 1 (+ n^2 for V)) s + 4)."""
    n = w["n"]
    v = 6 * n if w["jobz"] else 0
    s = 4 if w["dtype"] == "float32" else 8
    flops = counts["R"] * (40 + v) + counts["S"] * 12 + counts["D2"] * (25 + v)
    per = (3 * n - 1 + (n * n if w["jobz"] else 0)) * s + 4
    return float(flops), float(per * w["batch"])


def oracle_counts(w, d, e):
    """Rotations, implicit steps and 2x2 solves of the oracle on the same
    input.  The eigenvector update does not change them, so the oracle runs
    without it."""
    import oracle
    r = oracle.steqr(d, e, jobz=False, nthreads=os.cpu_count() or 1)
    return {"R": r.rotations, "S": r.sweeps, "D2": r.solves2x2}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons over
    the headline's load window (untimed load right before the timed steps,
    then the timed steps)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def time_workload(w, steps, warmup, dist_barrier, flush, stream, seed=0, min_warm_s=0.0, **params):
    """Device-side timing of `steps` solves after `warmup` untimed ones (and,
    with min_warm_s, more untimed solves until that many seconds of load have
    passed, so that clock samples right before and during the short timed
    region are taken under load); returns (ms list, d, e, kernel)."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dt = np.float32 if w["dtype"] == "float32" else np.float64
    d, e = inputs.problems(w.get("kind", "normal"), w["n"], w["batch"], dt, seed=seed)
    dev = torch.device("cuda")
    d0 = torch.from_numpy(d).to(dev)
    eg = torch.from_numpy(e).to(dev)
    dg = torch.empty_like(d0)
    Q = torch.empty((w["batch"], w["n"], w["n"]), dtype=d0.dtype, device=dev) if w["jobz"] else None
    work = torch.empty(bstq.work_size(dt, w["jobz"], w["n"], w["batch"], **params), dtype=torch.uint8,
                       device=dev)
    desc = bstq.describe(dt, w["jobz"], w["n"], w["batch"], **params)
    times = []
    with torch.cuda.stream(stream):
        t_end = time.time() + min_warm_s
        while time.time() < t_end:
            for _ in range(20):
                dg.copy_(d0)
                bstq.solve(dg, eg, jobz=w["jobz"], Q=Q, work=work, stream=stream, **params)
            torch.cuda.synchronize()
        for it in range(warmup + steps):
            dg.copy_(d0)
            flush.zero_()
            if it == warmup:
                dist_barrier()
                torch.cuda.synchronize()
            s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            bstq.solve(dg, eg, jobz=w["jobz"], Q=Q, work=work, stream=stream, **params)
            t.record(stream)
            if it >= warmup:
                times.append((s, t))
        torch.cuda.synchronize()
        dist_barrier()
    ms = [s.elapsed_time(t) for s, t in times]
    info = work[: 4 * w["batch"]].view(torch.int32)
    assert int((info != 0).sum()) == 0, "unconverged problems in the benchmark batch"
    return ms, d, e, desc


def time_syev(n, batch, dtype, jobz, steps, warmup, flush, stream):
    """Device-side timing of the fused small-n syev (dense symmetric A, N(0,1)
    entries on and below the diagonal, seed 0): ms per call."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dt = np.float32 if dtype == "float32" else np.float64
    A = torch.from_numpy(inputs.dense_symmetric(n, batch, dt, seed=0)).cuda()
    work = torch.empty(bstq.syev_work_size(dt, jobz, n, batch), dtype=torch.uint8, device="cuda")
    times = []
    with torch.cuda.stream(stream):
        for it in range(warmup + steps):
            flush.zero_()
            s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            W, V, info = bstq.syev(A, jobz=jobz, work=work, stream=stream)
            t.record(stream)
            if it >= warmup:
                times.append((s, t))
        torch.cuda.synchronize()
    assert int((info != 0).sum()) == 0, "unconverged problems in the syev batch"
    return statistics.mean(s.elapsed_time(t) for s, t in times)


def time_leaves(n, leaf, batch, dtype, jobz, steps, warmup, flush, stream):
    """Device-side timing of the stedc leaf solve (tear, the batched leaf
    solves and the gather, all in the call) on N(0,1) d and e, seed 0:
    ms per call."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dt = np.float32 if dtype == "float32" else np.float64
    d, e = inputs.normal_problems(n, batch, dt, seed=0)
    d0 = torch.from_numpy(d).cuda()
    dg = torch.empty_like(d0)
    eg = torch.from_numpy(e).cuda()
    work = torch.empty(bstq.stedc_leaves_work_size(dt, jobz, n, leaf, batch), dtype=torch.uint8, device="cuda")
    times = []
    with torch.cuda.stream(stream):
        for it in range(warmup + steps):
            dg.copy_(d0)
            flush.zero_()
            s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            _, _, _, info = bstq.stedc_leaves(dg, eg, leaf, jobz=jobz, work=work, stream=stream)
            t.record(stream)
            if it >= warmup:
                times.append((s, t))
        torch.cuda.synchronize()
    assert int((info != 0).sum()) == 0, "unconverged leaves in the benchmark batch"
    return statistics.mean(s.elapsed_time(t) for s, t in times)


def time_e2e(w, steps, warmup, stream):
    """End to end through the C ABI on pinned host buffers: H2D of d and e,
    the solve, D2H of lambda, Q and info, per step."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dt = np.float32 if w["dtype"] == "float32" else np.float64
    d, e = inputs.normal_problems(w["n"], w["batch"], dt, seed=0)
    n, B = w["n"], w["batch"]
    hd0 = torch.from_numpy(d)
    hd = hd0.clone().pin_memory()
    he = torch.from_numpy(e).pin_memory()
    hq = torch.empty((B, n, n), dtype=hd.dtype).pin_memory() if w["jobz"] else None
    hi = torch.empty(B, dtype=torch.int32).pin_memory()
    devbuf = torch.empty(bstq.host_work_size(dt, w["jobz"], n, B), dtype=torch.uint8, device="cuda")
    ms = []
    for it in range(warmup + steps):
        hd.copy_(hd0)
        torch.cuda.synchronize()
        s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        bstq.solve_host(hd, he, hq, hi, devbuf, stream=stream, jobz=w["jobz"])
        t.record(stream)
        t.synchronize()
        if it >= warmup:
            ms.append(s.elapsed_time(t))
    s_ = 4 if dt == np.float32 else 8
    h2d = B * (2 * n - 1) * s_
    d2h = B * n * s_ + (B * n * n * s_ if w["jobz"] else 0) + 4 * B
    return statistics.mean(ms), h2d, d2h


def cpu_baseline(w, seconds=12.0):
    """The oracle as it stands on this host's cores, on a bounded sample of
    the same workload; problems/s."""
    import oracle
    dt = np.float32 if w["dtype"] == "float32" else np.float64
    d, e = inputs.normal_problems(w["n"], w["batch"], dt, seed=0)
    cores = os.cpu_count() or 1
    sample = min(w["batch"], 2048)
    t0 = time.perf_counter()
    oracle.steqr(d[:sample], e[:sample], jobz=w["jobz"], nthreads=cores)
    t1 = time.perf_counter()
    rate = sample / (t1 - t0)
    # grow the sample to ~`seconds` of work, capped at the whole batch
    sample2 = int(min(w["batch"], max(sample, rate * seconds)))
    reps = max(1, int(rate * seconds / sample2))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.steqr(d[:sample2], e[:sample2], jobz=w["jobz"], nthreads=cores)
    t1 = time.perf_counter()
    rate = sample2 * reps / (t1 - t0)
    # one thread, on a sample sized for about a quarter of `seconds`
    one = int(min(w["batch"], max(256, rate / cores * seconds / 4)))
    t0 = time.perf_counter()
    oracle.steqr(d[:one], e[:one], jobz=w["jobz"], nthreads=1)
    t1 = time.perf_counter()
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {sample2} problems of the batch x {reps}, {cores} threads",
            "one_thread": {"value": one / (t1 - t0), "unit": UNIT, "cores": 1,
                           "sample": f"first {one} problems of the batch, 1 thread"},
            "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    platform string)."""
    import platform
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
    return platform.processor() or platform.machine()


def run_reference(args, rank, world):
    """--impl reference: the oracle, as it stands, timed on the host cores."""
    if rank != 0:
        return 0
    import oracle
    w = HEADLINE
    dt = np.float32
    d, e = inputs.normal_problems(w["n"], w["batch"], dt, seed=0)
    cores = os.cpu_count() or 1
    sample = 4096
    ms = []
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.steqr(d[:sample], e[:sample], jobz=True, nthreads=cores)
        t1 = time.perf_counter()
        if it >= args.warmup:
            ms.append((t1 - t0) * 1e3)
    mean_ms = statistics.mean(ms)
    value = sample / (mean_ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl_name(w), "step": f"oracle on the first {sample} problems"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"first {sample} problems of the batch per step, {cores} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_alu_peaks():
    """Compile alu_peaks.cu for sm_103a in a temporary directory, run it on
    the current GPU and print its JSON line (context for the derived
    FP32 / FP64 peaks of the roofline)."""
    import shutil
    import tempfile
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "alu_peaks")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        os.path.join(ROOT, "alu_peaks.cu")], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.strip()
    print(out)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-companions", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the n = 1..32 sweep of the companions")
    ap.add_argument("--alu-peaks", action="store_true",
                    help="build and run alu_peaks.cu (FP32 / FP64 FMA throughput) and print its line")
    ap.add_argument("--sched", type=int, default=0, help="0 auto, 1 flat, 2 nested (with --only)")
    ap.add_argument("--qstore", type=int, default=0, help="Q storage policy (with --only)")
    ap.add_argument("--kernel", type=int, default=0, help="kernel family 1 static, 2 dynamic (with --only)")
    ap.add_argument("--only", default=None,
                    help="time one workload 'dtype:n:V|N[:batch]' or 'leaves:dtype:n:leaf[:batch]' "
                         "and print its line (profiling aid)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.alu_peaks:
        return run_alu_peaks()

    import torch
    import torch.distributed as tdist
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    bstq.load()  # fails loudly without the CUDA library
    torch.cuda.set_device(local)
    if world > 1:
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            tdist.barrier()

    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    peaks = read_peaks()
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    sm_max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    fp32_peak = sms * SM_FP32_LANES * 2 * sm_max_mhz * 1e6
    fp64_peak = sms * SM_FP64_LANES * 2 * sm_max_mhz * 1e6
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0)) * 1e9

    if args.only and args.only.startswith("leaves:"):
        # leaves:dtype:n:leaf[:batch], the stedc leaf solve alone
        parts = args.only.split(":")
        dtype = {"f32": "float32", "f64": "float64"}.get(parts[1], parts[1])
        n, leaf = int(parts[2]), int(parts[3])
        batch = int(parts[4]) if len(parts) > 4 else 8192
        ms_l = time_leaves(n, leaf, batch, dtype, True, args.steps, args.warmup, flush, stream)
        print(json.dumps({"workload": f"stedc leaves {dtype} n={n} leaf={leaf} jobz=V batch={batch}",
                          "ms": ms_l, "problems_per_s": batch / (ms_l / 1e3)}))
        return 0
    if args.only:
        parts = args.only.split(":")
        w = dict(dtype={"f32": "float32", "f64": "float64"}.get(parts[0], parts[0]), n=int(parts[1]),
                 jobz=parts[2].upper() == "V", batch=int(parts[3]) if len(parts) > 3 else 32768)
        wm, wd, we, wdesc = time_workload(w, args.steps, args.warmup, barrier, flush, stream,
                                          scheduler=args.sched, qstore=args.qstore, kernel=args.kernel)
        t = statistics.mean(wm) / 1e3
        print(json.dumps({"workload": wl_name(w), "ms": t * 1e3, "problems_per_s": w["batch"] / t,
                          "kernel": wdesc}))
        return 0

    with ClockSampler(local) as clk:
        ms, d, e, desc = time_workload(HEADLINE, args.steps, args.warmup, barrier, flush, stream,
                                       seed=rank_seed(rank), min_warm_s=0.8)
    clocks = clk.summary()
    mean_ms, total_problems = aggregate(statistics.mean(ms), HEADLINE["batch"], world, tdist, "cuda")

    e2e_ms, h2d, d2h = time_e2e(HEADLINE, max(3, args.steps // 4), 2, stream)

    workloads = {}
    counts_cache = {}

    def measure(w, steps, **params):
        """Time workload w (with solver parameters) and price it against the
        roofline from the oracle's counts on the same input."""
        wm, wd, we, wdesc = time_workload(w, steps, 3, lambda: None, flush, stream, **params)
        key = wl_name(w)
        if key not in counts_cache:
            counts_cache[key] = oracle_counts(w, wd, we)
        fl, by = algorithmic(w, counts_cache[key])
        peak = fp32_peak if w["dtype"] == "float32" else fp64_peak
        t = statistics.mean(wm) / 1e3
        roof_t = max(fl / peak, by / hbm_peak)
        return {"problems_per_s": w["batch"] / t, "ms": t * 1e3, "roofline_fraction": roof_t / t,
                "kernel": wdesc, "gflop": fl / 1e9, "mb": by / 1e6}

    if rank == 0 and not args.no_companions:
        csteps = max(5, args.steps // 2)
        for w in [SMALL_CASE] + COMPANIONS + MIXED:
            workloads[wl_name(w)] = measure(w, csteps)
        # flat lockstep against the nested loop, each forced, for the float
        # n = 8 / 16 and double n = 12 workloads
        for w in COMPANIONS:
            for sched, nm in ((1, "flat"), (2, "nested")):
                workloads[f"scheduler {nm}: {wl_name(w)}"] = measure(w, csteps, scheduler=sched)
        # n = 1 .. 32 in both precisions and both jobz (batch 65,536 for
        # n <= 8, else 32,768)
        if not args.no_sweep:
            sweep = {}
            for dtype in ("float32", "float64"):
                for jobz in (True, False):
                    rows = []
                    for n in range(1, 33):
                        w = dict(dtype=dtype, n=n, batch=65536 if n <= 8 else 32768, jobz=jobz)
                        r = measure(w, 3)
                        rows.append([n, round(r["problems_per_s"]), round(r["roofline_fraction"], 4),
                                     round(r["ms"], 4)])
                    sweep[f"{dtype} jobz={'V' if jobz else 'N'}"] = rows
            workloads["sweep n=1..32 (n, problems/s, roofline fraction, ms)"] = sweep
        for dtype, n in (("float32", 16), ("float64", 12)):
            ms_s = time_syev(n, 32768, dtype, True, max(5, args.steps // 2), 3, flush, stream)
            workloads[f"fused syev {dtype} n={n} jobz=V batch=32768 dense N(0,1) seed 0"] = {
                "problems_per_s": 32768 / (ms_s / 1e3), "ms": ms_s,
                "kernel": "syev_kernel (Householder reduction + dynamic-position solve, one launch)"}
        # saturation knee: per-problem time at 4x the batch against the batch
        for w in (HEADLINE, COMPANIONS[3]):
            w4 = dict(w, batch=4 * w["batch"])
            m4, _, _, desc4 = time_workload(w4, max(5, args.steps // 2), 3, lambda: None, flush, stream)
            t1 = statistics.mean(ms) / 1e3 if w is HEADLINE else workloads[wl_name(w)]["ms"] / 1e3
            t4 = statistics.mean(m4) / 1e3
            workloads[f"saturation: {wl_name(w4)}"] = {
                "problems_per_s": w4["batch"] / t4, "ms": t4 * 1e3, "kernel": desc4,
                "per_problem_time_vs_batch": (t4 / w4["batch"]) / (t1 / w["batch"])}
        for dtype, n, leaf, batch in (("float32", 64, 32, 8192), ("float64", 64, 32, 8192)):
            ms_l = time_leaves(n, leaf, batch, dtype, True, max(5, args.steps // 2), 3, flush, stream)
            workloads[f"stedc leaves {dtype} n={n} leaf={leaf} jobz=V batch={batch} N(0,1) seed 0"] = {
                "problems_per_s": batch / (ms_l / 1e3), "leaves_per_s": batch * (n // leaf) / (ms_l / 1e3),
                "ms": ms_l, "kernel": "tear + batched leaf solve + gather (bstq_stedc_leaves)"}
        # sizes beyond the sub-group width (dynamic family), with eigenvectors
        for w in (dict(dtype="float32", n=64, batch=32768, jobz=True), dict(dtype="float64", n=64, batch=32768, jobz=True),
                  dict(dtype="float32", n=128, batch=8192, jobz=True), dict(dtype="float64", n=128, batch=8192, jobz=True)):
            workloads[wl_name(w)] = measure(w, 3)

    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return 0
    counts = oracle_counts(HEADLINE, d, e)
    digest = kernel_digest()
    flops, bytes_ = algorithmic(HEADLINE, counts)
    t = mean_ms / 1e3
    value = total_problems / t
    achieved = flops / t
    roof_t = max(flops / fp32_peak, bytes_ / hbm_peak)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_BASELINE, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl_name(HEADLINE), "per_gpu_batch": HEADLINE["batch"],
                   "parallelism": f"replicas x{world} (independent problems, no collective)",
                   "l2": "flushed between steps (256 MiB write)", "kernel": desc,
                   "kernel_digest": digest,
                   "sweep_budget": "30 per eigenvalue"},
        "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": fp32_peak / 1e12,
                     "unit": "TFLOP/s", "frac": achieved / fp32_peak, "traffic": NCU_TRAFFIC.get((desc, digest)),
                     "roofline_fraction": roof_t / t,
                     "peak_source": f"derived: {sms} SMs x {SM_FP32_LANES} FP32 lanes x 2 x {sm_max_mhz:.0f} MHz",
                     "algorithmic_gflop_per_launch": flops / 1e9, "algorithmic_mb_per_launch": bytes_ / 1e6,
                     "oracle_counts": counts},
        "cpu_baseline": cpu_baseline(HEADLINE),
        "e2e": {"value": HEADLINE["batch"] / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "workloads": workloads,
        "vs_baseline_ref": "steqr_cta flat, float n=16 V, batch 32,768 on RTX 4090 (other hardware)",
    }
    print(json.dumps(line))
    if world > 1:
        tdist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
