"""Host logic of bench.py, on CPU: the reference arm's JSON line, the
algorithmic byte and flop counts of the roofline, and the source set the
ncu traffic key is digested over."""
import json
import os
import subprocess
import sys

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == bench.wl_name(bench.HEADLINE)


def test_algorithmic_counts_follow_the_stated_formulas():
    """bytes = batch ((3n - 1 + n^2 [V]) s + 4); flops = R (40 + 6n [V]) +
    12 S + D2 (25 + 6n [V]), with the per-problem byte figures of the
    measurement plan (f32 n=16 V 1,216 B, f64 n=12 V 1,436 B)."""
    counts = {"R": 0, "S": 0, "D2": 0}
    _, b = bench.algorithmic(dict(dtype="float32", n=16, batch=1, jobz=True), counts)
    assert b == 1216
    _, b = bench.algorithmic(dict(dtype="float64", n=12, batch=1, jobz=True), counts)
    assert b == 1436
    _, b = bench.algorithmic(dict(dtype="float32", n=16, batch=32768, jobz=False), counts)
    assert b == 192 * 32768
    f, _ = bench.algorithmic(dict(dtype="float32", n=16, batch=1, jobz=True), {"R": 1, "S": 0, "D2": 0})
    assert f == 40 + 6 * 16
    f, _ = bench.algorithmic(dict(dtype="float64", n=12, batch=1, jobz=False), {"R": 0, "S": 1, "D2": 1})
    assert f == 12 + 25


def test_traffic_key_digests_the_timed_kernels_sources():
    src = bench.kernel_sources()
    assert src[0] == bench.HEADLINE_UNIT or bench.HEADLINE_UNIT in src
    for f in ("bstq_split.cuh", "bstq_lane.cuh", "bstq_numerics.cuh"):
        assert f in src
    # the boundary and other kernels are not part of this kernel
    for f in ("bstq_api.cu", "bstq_leaves.cu", "bstq_dyn.cuh", "bstq_syev.cuh"):
        assert f not in src
    assert len(bench.kernel_digest()) == 16
    assert bench.kernel_digest("bstq_kern_dyn_f64_v12.cu") != bench.kernel_digest()


def test_rank_seeds_differ():
    assert len({bench.rank_seed(r) for r in range(8)}) == 8
    assert np.isclose(bench.PAGES_BASELINE, 32768 / 450.9e-6)
