"""The C ABI from plain C: tests/c_abi_check.c includes include/bstq.h, links
libbstq.so with gcc and runs the checks that need no GPU (version, status
text, argument codes, the no-device status).  CPU only."""
import os
import shutil
import subprocess

import pytest

from symmetric_tridiagonal_eigensolver_gb300 import bstq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    if not os.path.exists(bstq.LIB_PATH):
        from symmetric_tridiagonal_eigensolver_gb300 import build
        build.build()
    libdir = os.path.dirname(bstq.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-lbstq",
           "-Wl,-rpath," + libdir, "-o", exe]
    subprocess.run(cmd, check=True)
    try:
        import torch
        gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        gpu = False
    r = subprocess.run([exe] + (["gpu"] if gpu else []), capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK")
