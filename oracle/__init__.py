"""CPU oracle for the batched symmetric tridiagonal eigensolver.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package entry's ``smoke()``
check and the benchmark's ``cpu_baseline`` / reference leg may import this
module.  The CUDA library never links, loads or calls it, and it shares no
code with the library.

The oracle is plain C (``steqr_oracle.c`` + ``steqr_oracle_impl.h``): implicit
shifted QL/QR with a Givens bulge chase, one problem at a time, in the
problem's own precision, following the BatchLAS pages "algo_steqr" (the
mathematics of steqr) and "perf_steqr" (steqr_cta notes).  This module
compiles it with gcc (``-O2 -ffp-contract=off``) and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SOURCES = ("steqr_oracle.c", "steqr_oracle_impl.h")
_lock = threading.Lock()
_lib = None

DEFAULT_MAXIT_PER_N = 30


def build(force: bool = False, src_dir: str = _HERE, out_path: str = _LIB_PATH) -> str:
    """Compile liboracle.so (idempotent unless a source is newer).  ``src_dir``
    and ``out_path`` let the tests build a deliberately broken copy."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    srcs = [os.path.join(src_dir, s) for s in _SOURCES]
    if (not force and os.path.exists(out_path)
            and all(os.path.getmtime(out_path) >= os.path.getmtime(s) for s in srcs)):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-fPIC", "-shared", "-o", tmp, srcs[0], "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, cwd=src_dir)
    os.replace(tmp, out_path)
    return out_path


def _bind(lib):
    for suffix in ("f32", "f64"):
        fn = getattr(lib, f"oracle_steqr_batch_{suffix}")
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                       ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_int, ctypes.c_int]
    for suffix in ("f32", "f64"):
        fn = getattr(lib, f"oracle_syev_batch_{suffix}")
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.oracle_constant.restype = ctypes.c_double
    lib.oracle_constant.argtypes = [ctypes.c_int, ctypes.c_int]
    return lib


def load_variant(path: str):
    """Load another build of the oracle (used only by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def constants(dtype) -> dict:
    """eps, safmin, ssfmax, ssfmin exactly as the oracle uses them."""
    code = 0 if np.dtype(dtype) == np.float32 else 1
    lib = _load()
    return {k: lib.oracle_constant(code, i)
            for i, k in enumerate(("eps", "safmin", "ssfmax", "ssfmin"))}


class Result:
    """Oracle output for a batch: eigenvalues ``lam`` (batch, n), eigenvectors
    ``Q`` (batch, n, n) with ``Q[b, :, j]`` the j-th eigenvector (None when
    jobz = N), ``info`` (batch,) int32 and the summed work counters."""

    def __init__(self, lam, Q, info, sweeps, rotations, solves2x2):
        self.lam = lam
        self.Q = Q
        self.info = info
        self.sweeps = sweeps
        self.rotations = rotations
        self.solves2x2 = solves2x2


def steqr(d, e, jobz: bool = True, maxit_per_n: int = DEFAULT_MAXIT_PER_N,
          sort: bool = True, nthreads: int = 1, lib=None, Z=None, scheme: str = "exp") -> Result:
    """Run the oracle on host arrays ``d`` (batch, n) and ``e`` (batch, n-1).

    The dtype of ``d`` (float32 or float64) selects the precision; ``e`` is
    cast to it.  With ``Z`` (batch, n, n) given (and jobz), the rotations are
    right-applied to Z instead of the identity (back_transform, BatchLAS page
    "algo_steqr", eigenvector accumulation): ``Q`` is then Z times the
    eigenvectors.  ``scheme`` selects the implicit step's update: "exp"
    (each local similarity written out, the default) or "pg" (the scalars
    (g, p, c, s) propagated across the sweep), page "algo_steqr", update
    schemes.  Inputs are not modified."""
    if scheme not in ("exp", "pg"):
        raise ValueError("oracle: scheme must be 'exp' or 'pg'")
    d = np.asarray(d)
    if d.dtype not in (np.float32, np.float64):
        raise TypeError("oracle: d must be float32 or float64")
    dt = d.dtype
    if d.ndim == 1:
        d = d[None, :]
    batch, n = d.shape
    e = np.asarray(e, dtype=dt).reshape(batch, max(n - 1, 0))
    lam = np.ascontiguousarray(d, dtype=dt).copy()
    ec = np.ascontiguousarray(e, dtype=dt)
    Qc = np.empty((batch, n, n), dtype=dt) if jobz else None  # column-major per problem
    mode = int(bool(jobz))
    if jobz and Z is not None:
        Zc = np.asarray(Z, dtype=dt).reshape(batch, n, n)
        Qc[...] = np.swapaxes(Zc, 1, 2)  # memory [b][j][i] = Z_ij
        mode = 2
    info = np.zeros(batch, dtype=np.int32)
    cnt = np.zeros(3, dtype=np.int64)
    lib = lib if lib is not None else _load()
    fn = lib.oracle_steqr_batch_f32 if dt == np.float32 else lib.oracle_steqr_batch_f64
    rc = fn(int(n), int(batch), mode, int(maxit_per_n), int(bool(sort)),
            lam.ctypes.data, ec.ctypes.data if ec.size else None,
            Qc.ctypes.data if jobz else None, info.ctypes.data, cnt.ctypes.data,
            int(nthreads), 0 if scheme == "exp" else 1)
    if rc != 0:
        raise ValueError(f"oracle: invalid arguments (n={n}, batch={batch})")
    Q = None
    if jobz:
        # stored column-major per problem: memory [b][j][i] = Q_ij
        Q = np.ascontiguousarray(np.swapaxes(Qc, 1, 2))
    return Result(lam, Q, info, int(cnt[0]), int(cnt[1]), int(cnt[2]))


def syev(A, jobz: bool = True, maxit_per_n: int = DEFAULT_MAXIT_PER_N, sort: bool = True,
         nthreads: int = 1, lib=None, scheme: str = "exp") -> Result:
    """Fused small-n dense symmetric eigensolver on host arrays: ``A``
    (batch, n, n), of which the lower triangle (A[b, i, j], i >= j) is read.
    Householder reduction to tridiagonal form, then the steqr solve with the
    reduction's Q as the basis (back_transform).  Returns a Result with
    ``lam`` (batch, n), ``Q`` (batch, n, n) the eigenvectors of A (None when
    jobz = N), ``info`` and the steqr counters.  Inputs are not modified."""
    A = np.asarray(A)
    if A.dtype not in (np.float32, np.float64):
        raise TypeError("oracle: A must be float32 or float64")
    if scheme not in ("exp", "pg"):
        raise ValueError("oracle: scheme must be 'exp' or 'pg'")
    dt = A.dtype
    if A.ndim == 2:
        A = A[None]
    batch, n, n2 = A.shape
    if n != n2:
        raise ValueError("oracle: A must be (batch, n, n)")
    Ac = np.ascontiguousarray(np.swapaxes(A, 1, 2))  # memory [b][j][i] = A_ij
    W = np.empty((batch, n), dtype=dt)
    Vc = np.empty((batch, n, n), dtype=dt) if jobz else None
    info = np.zeros(batch, dtype=np.int32)
    cnt = np.zeros(3, dtype=np.int64)
    lib = lib if lib is not None else _load()
    fn = lib.oracle_syev_batch_f32 if dt == np.float32 else lib.oracle_syev_batch_f64
    rc = fn(int(n), int(batch), int(bool(jobz)), int(maxit_per_n), int(bool(sort)),
            Ac.ctypes.data, W.ctypes.data, Vc.ctypes.data if jobz else None, info.ctypes.data,
            cnt.ctypes.data, int(nthreads), 0 if scheme == "exp" else 1)
    if rc != 0:
        raise ValueError(f"oracle: invalid arguments (n={n}, batch={batch})")
    V = np.ascontiguousarray(np.swapaxes(Vc, 1, 2)) if jobz else None
    return Result(W, V, info, int(cnt[0]), int(cnt[1]), int(cnt[2]))


class Leaves:
    """Oracle output of the stedc leaf solve for a batch of size-n problems
    torn into leaves: ``starts``/``sizes`` the leaves' first rows and sizes
    (consecutive leaves of ``leaf`` rows, the remainder last), ``d_torn``
    (batch, n) the torn diagonal, ``lam`` (batch, n) each leaf's eigenvalues
    at the leaf's rows (ascending within the leaf), ``Q`` a list with one
    (batch, size, size) array per leaf (``Q[k][b, :, j]`` the j-th
    eigenvector of leaf k, None when jobz = N) and ``info`` (batch, leaves)."""

    def __init__(self, starts, sizes, d_torn, lam, Q, info):
        self.starts = starts
        self.sizes = sizes
        self.d_torn = d_torn
        self.lam = lam
        self.Q = Q
        self.info = info


def leaf_partition(n: int, leaf: int):
    """Leaves of a size-n problem: consecutive runs of ``leaf`` rows from the
    top, the remainder (if any) as a last, shorter leaf.  A leaf size at or
    above n gives one leaf.  Returns (starts, sizes)."""
    if n < 1 or leaf < 1:
        raise ValueError("oracle: n and leaf must be >= 1")
    size = min(leaf, n)
    starts = list(range(0, n, size))
    return starts, [min(size, n - s) for s in starts]


def tear(d, e, leaf: int):
    """The divide step of divide and conquer (BatchLAS page "algo_steqr": the
    leaf solve of stedc; the rank-one tear of Cuppen's method): at every
    boundary between leaves, rows r-1 | r with off-diagonal beta = e[r-1],
    T = diag(T_1, T_2) + |beta| v v^T with v = e_{r-1} + sign(beta) e_r, so
    the leaves are T's diagonal blocks with |beta| taken off the two diagonal
    entries next to the boundary.  Boundaries are applied top to bottom in
    the problem's own precision, so a one-row leaf between two boundaries
    holds (d - |e_left|) - |e_right|.  Returns (starts, sizes, d_torn)."""
    d = np.asarray(d)
    batch, n = d.shape
    e = np.asarray(e, dtype=d.dtype).reshape(batch, max(n - 1, 0))
    starts, sizes = leaf_partition(n, leaf)
    dt = d.copy()
    for r in starts[1:]:
        beta = np.abs(e[:, r - 1])
        dt[:, r - 1] = dt[:, r - 1] - beta
        dt[:, r] = dt[:, r] - beta
    return starts, sizes, dt


def stedc_leaves(d, e, leaf: int, jobz: bool = True, maxit_per_n: int = DEFAULT_MAXIT_PER_N,
                 sort: bool = True, nthreads: int = 1, lib=None) -> Leaves:
    """Leaf solve of divide and conquer on host arrays ``d`` (batch, n) and
    ``e`` (batch, n-1): tear every problem into leaves (``tear``), then solve
    each leaf, a tridiagonal problem of at most ``leaf`` rows whose
    off-diagonal is e inside the leaf, with the steqr oracle (identity start,
    ascending eigenvalues).  Inputs are not modified."""
    d = np.asarray(d)
    if d.dtype not in (np.float32, np.float64):
        raise TypeError("oracle: d must be float32 or float64")
    if d.ndim == 1:
        d = d[None, :]
    batch, n = d.shape
    e = np.asarray(e, dtype=d.dtype).reshape(batch, max(n - 1, 0))
    starts, sizes, dt = tear(d, e, leaf)
    lam = np.empty_like(dt)
    info = np.zeros((batch, len(starts)), dtype=np.int32)
    Qs = []
    for k, (s, m) in enumerate(zip(starts, sizes)):
        r = steqr(dt[:, s:s + m], e[:, s:s + m - 1], jobz=jobz, maxit_per_n=maxit_per_n, sort=sort,
                  nthreads=nthreads, lib=lib)
        lam[:, s:s + m] = r.lam
        info[:, k] = r.info
        Qs.append(r.Q)
    return Leaves(starts, sizes, dt, lam, Qs if jobz else None, info)
