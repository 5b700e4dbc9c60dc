"""The launch plan's block size as a host-only function (csrc/bstq_plan.h),
compiled with g++ and pinned to the shapes the GB300 runs reported through
bstq_describe (a wrong plan still gives correct eigenvalues, so the shape is
asserted directly).  CPU only."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "symmetric_tridiagonal_eigensolver_gb300", "csrc")

# (batch, SMs, block cap, f64) -> (threads per block, grid); the first four
# are the launches bench.py recorded on a GB300 (152 SMs), e.g.
# "dyn<f64,12,V,global,flat> tpb=288 grid=456" at batch 131072
CASES = [
    ((32768, 152, 384, 1), (224, 147)),    # f64 n=12 V: one wave, one block per SM
    ((131072, 152, 384, 1), (288, 456)),   # f64 n=12 V at 4x: three even waves
    ((65536, 152, 416, 0), (128, 512)),    # f32 n=8 V: beyond one wave, 128-thread blocks
    ((65536, 152, 1024, 0), (448, 147)),   # f32 n=8 N: one wave
    ((0, 152, 384, 1), (32, 0)),           # empty batch
    ((1, 152, 384, 0), (32, 1)),           # one problem
    ((152 * 384, 152, 384, 1), (384, 152)),        # exactly one full wave
    ((152 * 384 + 1, 152, 384, 1), (224, 261)),    # one more: two even waves
    ((152 * 384 + 1, 152, 384, 0), (128, 457)),    # float: 128-thread blocks
    ((10 ** 7, 152, 96, 0), (96, 104167)),         # a cap below 128
]


def test_block_size_matches_the_recorded_launches(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "plan_shape_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "plan_shape_check.cpp"), "-o", exe], check=True)
    stdin = "".join(f"{b} {s} {c} {f}\n" for (b, s, c, f), _ in CASES)
    r = subprocess.run([exe], input=stdin, capture_output=True, text=True, timeout=60, check=True)
    got = [tuple(int(x) for x in ln.split()) for ln in r.stdout.splitlines()]
    assert got == [want for _, want in CASES]
    for ((b, s, c, f), (tpb, grid)) in zip([k for k, _ in CASES], got):
        assert tpb % 32 == 0 and tpb <= max(c, 32) and tpb * grid >= b


# Record-and-apply layout: (batch, n, n_pad, log_entries) -> (log entries per
# problem, offsets of the log lengths, maps and logs, total work bytes, apply
# warps).  The first three totals are the `work=` sizes bstq_describe
# reported on a GB300 for the bench workloads f32 n = 64 V (batch 32,768),
# n = 128 V (8,192) and n = 33 V (32,768).
RLOG_CASES = [
    ((32768, 64, 64, 0), (6656, 131072, 262144, 4456448, 1749286912, 32768)),
    ((8192, 128, 128, 0), (25600, 32768, 65536, 2162688, 1679884288, 32768)),
    ((32768, 33, 48, 0), (2048, 131072, 262144, 2424832, 539295744, 32768)),
    ((8192, 96, 96, 0), (14592, 32768, 65536, 1638400, 957939712, 24576)),
    ((300, 40, 48, 1), (256, 1280, 2560, 26624, 641024, 300)),        # one page
    ((300, 40, 48, 300), (512, 1280, 2560, 26624, 1255424, 300)),     # rounded up to pages
    ((1, 127, 128, 0), (25344, 256, 512, 768, 203520, 4)),       # 1.5 * 127^2 + 8 * 127 = 25209 -> 99 pages
]


def test_record_and_apply_layout(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "rlog_layout_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "rlog_layout_check.cpp"), "-o", exe], check=True)
    stdin = "".join(f"{b} {n} {nm} {le}\n" for (b, n, nm, le), _ in RLOG_CASES)
    r = subprocess.run([exe], input=stdin, capture_output=True, text=True, timeout=60, check=True)
    got = [tuple(int(x) for x in ln.split()) for ln in r.stdout.splitlines()]
    assert got == [want for _, want in RLOG_CASES]
    for (b, n, nm, le), (lcap, oc, om, ol, tot, aw) in zip([k for k, _ in RLOG_CASES], got):
        assert lcap % 256 == 0 and lcap >= max(le, 1) and lcap >= n + 4
        assert oc % 256 == 0 and om % 256 == 0 and ol % 256 == 0   # 256-byte aligned regions
        assert om - oc >= 4 * b and ol - om >= 2 * n * b and tot >= ol + 8 * lcap * b
