"""The C-ABI library loads, exports every symbol include/bstq.h declares and
rejects invalid arguments with the documented codes (CPU only: no compute
call is made)."""
import ctypes
import os
import re

import pytest

from symmetric_tridiagonal_eigensolver_gb300 import bstq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bstq.LIB_PATH):
        from symmetric_tridiagonal_eigensolver_gb300 import build
        build.build()
    return bstq.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bstq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bstq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(bstq.EXPORTS)


def test_version_and_status_strings(lib):
    assert bstq.version().startswith("bstq")
    assert bstq.status_string(0) == "success"
    assert "n outside" in bstq.status_string(-3)
    # the allocation-free entry point's size limit is named in the text of -4
    assert "fixed scratch" in bstq.status_string(-4)


def test_invalid_arguments_are_rejected_before_any_device_use(lib):
    vp = ctypes.c_void_p
    buf = (ctypes.c_char * 64)()
    good = ctypes.cast(buf, vp)
    solve = lib.bstq_solve
    assert solve(7, 1, 8, 10, good, good, good, good, None) == -1
    assert solve(0, 5, 8, 10, good, good, good, good, None) == -2
    assert solve(0, 1, 0, 10, good, good, good, good, None) == -3
    assert solve(0, 1, bstq.MAX_N + 1, 10, good, good, good, good, None) == -3
    assert solve(0, 1, 8, -1, good, good, good, good, None) == -4
    assert solve(0, 1, 8, 0, None, None, None, None, None) == 0   # batch 0: no-op
    assert solve(0, 1, 8, 10, None, good, good, good, None) == -5
    assert solve(0, 1, 8, 10, good, None, good, good, None) == -6
    assert solve(0, 1, 8, 10, good, good, None, good, None) == -7
    assert solve(0, 1, 8, 10, good, good, good, None, None) == -8
    mis = ctypes.c_void_p(ctypes.addressof(buf) + 2)
    assert solve(0, 1, 8, 10, mis, good, good, good, None) == -5
    p = bstq.Params(0, 0, 9, 0, 0, 0)
    assert lib.bstq_solve_ex(0, 1, 8, 10, good, good, good, good, None, ctypes.byref(p)) == -10
    p = bstq.Params(0, 0, 0, 0, 48, 0)
    assert lib.bstq_solve_ex(0, 1, 8, 10, good, good, good, good, None, ctypes.byref(p)) == -10
    p = bstq._params(log_entries=-1)   # rotation log capacity: checked before any device query
    assert lib.bstq_solve_ex(0, 1, 64, 10, good, good, good, good, None, ctypes.byref(p)) == -10
    assert lib.bstq_work_size(0, 1, 40, 10) == 0
    assert lib.bstq_solve_host(0, 1, 8, 10, None, good, good, good, good, None, None) == -5
    # the diagnostic entry point
    diag = lib.bstq_diag
    assert diag(99, 0, 10, 0, good, good, good, None) == -1          # unknown op
    assert diag(bstq.DIAG_FASTQ, 0, 10, 5, good, good, good, None) == -1   # double only
    assert diag(bstq.DIAG_RCP, 7, 10, 0, good, good, good, None) == -2
    assert diag(bstq.DIAG_RCP, 0, -1, 0, good, good, good, None) == -3
    assert diag(bstq.DIAG_FASTQ, 1, 10, -1, good, good, good, None) == -4
    assert diag(bstq.DIAG_RCP, 0, 0, 0, None, None, None, None) == 0     # empty: no-op
    assert diag(bstq.DIAG_RCP, 0, 10, 0, None, good, None, None) == -5
    assert diag(bstq.DIAG_RCP, 1, 10, 0, mis, good, None, None) == -5
    assert diag(bstq.DIAG_RCP, 0, 10, 0, good, None, None, None) == -6
    assert diag(bstq.DIAG_PASS_DYN_EXP, 0, 10, 0, good, good, None, None) == -7
    assert lib.bstq_diag_work_size(bstq.DIAG_PASS_DYN_PG, 1, 100) >= 100 * 16 * 16 * 8
    assert lib.bstq_diag_work_size(99, 1, 100) == 0


def test_no_device_is_reported_not_faked(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    vp = ctypes.c_void_p
    buf = (ctypes.c_char * 64)()
    good = ctypes.cast(buf, vp)
    rc = lib.bstq_solve(0, 1, 8, 10, good, good, good, good, None)
    assert rc == bstq.ERR_NODEVICE


def test_product_path_does_not_touch_the_oracle():
    """The library and its binding never import or load the oracle."""
    pkg = os.path.join(ROOT, "symmetric_tridiagonal_eigensolver_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "liboracle" not in text, f


def test_stedc_leaves_arguments(lib):
    vp = ctypes.c_void_p
    buf = (ctypes.c_char * 1024)()
    good = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, vp)
    f = lib.bstq_stedc_leaves
    assert f(7, 1, 70, 32, 10, good, good, good, good, good, None, None) == -1
    assert f(0, 5, 70, 32, 10, good, good, good, good, good, None, None) == -2
    assert f(0, 1, 0, 32, 10, good, good, good, good, good, None, None) == -3
    assert f(0, 1, 70, 0, 10, good, good, good, good, good, None, None) == -3
    assert f(0, 1, 70, bstq.MAX_N + 1, 10, good, good, good, good, good, None, None) == -3
    assert f(0, 1, 70, 32, -1, good, good, good, good, good, None, None) == -4
    assert f(0, 1, 70, 32, 0, None, None, None, None, None, None, None) == 0   # batch 0: no-op
    assert f(0, 1, 70, 32, 10, None, good, good, good, good, None, None) == -5
    assert f(0, 1, 70, 32, 10, good, None, good, good, good, None, None) == -6
    assert f(0, 1, 70, 32, 10, good, good, None, good, good, None, None) == -7
    assert f(0, 1, 70, 32, 10, good, good, good, None, good, None, None) == -8
    assert f(0, 1, 70, 32, 10, good, good, good, good, None, None, None) == -8
    p = bstq.Params(0, 0, 0, 0, 0, 0, 1, 0)   # back_transform: leaves start from the identity
    assert f(0, 1, 70, 32, 10, good, good, good, good, good, None, ctypes.byref(p)) == -10
    ws = lib.bstq_stedc_leaves_work_size
    assert ws(0, 1, 70, 0, 100, None) == 0 and ws(0, 1, 70, 32, 100, ctypes.byref(p)) == 0
    assert bstq.leaf_shape(70, 32) == (32, 2, 6) and bstq.leaf_shape(5, 8) == (5, 1, 0)


def test_stedc_leaves_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    vp = ctypes.c_void_p
    buf = (ctypes.c_char * 1024)()
    good = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, vp)
    assert lib.bstq_stedc_leaves(0, 1, 70, 32, 10, good, good, good, good, good, None, None) == bstq.ERR_NODEVICE


def test_missing_library_fails_loudly(tmp_path):
    """Without libbstq.so the binding raises: there is no CPU fallback."""
    import subprocess
    import sys
    code = ("from symmetric_tridiagonal_eigensolver_gb300 import bstq\n"
            f"bstq.load({str(tmp_path / 'libbstq.so')!r})\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libbstq.so not found" in r.stderr
