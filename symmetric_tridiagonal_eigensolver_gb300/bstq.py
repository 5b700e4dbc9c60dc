"""Thin ctypes binding of libbstq.so (the C ABI in include/bstq.h).

Argument marshalling only: every step of the solve runs in the CUDA library.
PyTorch supplies device memory and streams.  Importing works without a GPU;
calling into the library without libbstq.so raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbstq.so")

F32, F64 = 0, 1
JOBZ_N, JOBZ_V = 0, 1
SCHED_AUTO, SCHED_FLAT, SCHED_NESTED = 0, 1, 2
QSTORE_AUTO, QSTORE_REGISTERS, QSTORE_SHARED, QSTORE_GLOBAL, QSTORE_HYBRID, QSTORE_SPLIT, QSTORE_LOG = 0, 1, 2, 3, 4, 5, 6
KERNEL_AUTO, KERNEL_STATIC, KERNEL_DYNAMIC = 0, 1, 2
UPDATE_EXP, UPDATE_PG = 0, 1
ERR_CUDA, ERR_NODEVICE = 1, 2
MAX_N = 128

# Every symbol include/bstq.h declares.
EXPORTS = ("bstq_work_size", "bstq_work_size_ex", "bstq_solve", "bstq_solve_ex",
           "bstq_host_work_size", "bstq_solve_host", "bstq_describe",
           "bstq_status_string", "bstq_version", "bstq_last_error", "bstq_solve_noalloc",
           "bstq_syev_work_size", "bstq_syev", "bstq_stedc_leaves_work_size", "bstq_stedc_leaves",
           "bstq_diag_work_size", "bstq_diag")

# Diagnostic ops (bstq_diag): one building block of the solve on a table of
# inputs; values in and out per record.
DIAG_RCP, DIAG_DIV, DIAG_SQRT, DIAG_RSQRT, DIAG_HYP1 = 1, 2, 3, 4, 5
DIAG_LARTG, DIAG_LARTG_FAST, DIAG_SHIFT = 6, 7, 8
DIAG_PASS_STATIC, DIAG_PASS_DYN_EXP, DIAG_PASS_DYN_PG = 20, 21, 22
DIAG_FASTQ = 30
DIAG_SHAPE = {DIAG_RCP: (1, 1), DIAG_DIV: (2, 1), DIAG_SQRT: (1, 1), DIAG_RSQRT: (1, 1), DIAG_HYP1: (1, 1),
              DIAG_LARTG: (2, 3), DIAG_LARTG_FAST: (2, 3), DIAG_SHIFT: (3, 4),
              DIAG_PASS_STATIC: (42, 288), DIAG_PASS_DYN_EXP: (42, 288), DIAG_PASS_DYN_PG: (42, 288)}


class Params(ctypes.Structure):
    """bstq_params; all-zero means the defaults."""
    _fields_ = [("no_sort", ctypes.c_int), ("max_sweeps_per_n", ctypes.c_int),
                ("scheduler", ctypes.c_int), ("qstore", ctypes.c_int),
                ("threads_per_block", ctypes.c_int), ("kernel", ctypes.c_int),
                ("back_transform", ctypes.c_int), ("update_scheme", ctypes.c_int),
                ("log_entries", ctypes.c_int)]


class BstqError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        extra = ""
        if code == ERR_CUDA:
            extra = ": " + load().bstq_last_error().decode()
        super().__init__(f"{where}: {status_string(code)} (code {code}){extra}")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libbstq.so (built by symmetric_tridiagonal_eigensolver_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libbstq.so not found at {path}; run "
                              "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(path)
        vp, sz, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
        P = ctypes.POINTER(Params)
        lib.bstq_work_size.restype = sz
        lib.bstq_work_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64]
        lib.bstq_work_size_ex.restype = sz
        lib.bstq_work_size_ex.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P]
        lib.bstq_solve.restype = ctypes.c_int
        lib.bstq_solve.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp, vp]
        lib.bstq_solve_ex.restype = ctypes.c_int
        lib.bstq_solve_ex.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp, vp, P]
        lib.bstq_host_work_size.restype = sz
        lib.bstq_host_work_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P]
        lib.bstq_solve_host.restype = ctypes.c_int
        lib.bstq_solve_host.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp,
                                        vp, vp, P]
        lib.bstq_describe.restype = ctypes.c_int
        lib.bstq_describe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P,
                                      ctypes.c_char_p, sz]
        lib.bstq_status_string.restype = ctypes.c_char_p
        lib.bstq_status_string.argtypes = [ctypes.c_int]
        lib.bstq_version.restype = ctypes.c_char_p
        lib.bstq_version.argtypes = []
        lib.bstq_last_error.restype = ctypes.c_char_p
        lib.bstq_last_error.argtypes = []
        lib.bstq_syev_work_size.restype = sz
        lib.bstq_syev_work_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P]
        lib.bstq_syev.restype = ctypes.c_int
        lib.bstq_syev.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp, vp, P]
        lib.bstq_stedc_leaves_work_size.restype = sz
        lib.bstq_stedc_leaves_work_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P]
        lib.bstq_stedc_leaves.restype = ctypes.c_int
        lib.bstq_stedc_leaves.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp,
                                          vp, vp, vp, P]
        lib.bstq_diag_work_size.restype = sz
        lib.bstq_diag_work_size.argtypes = [ctypes.c_int, ctypes.c_int, i64]
        lib.bstq_diag.restype = ctypes.c_int
        lib.bstq_diag.argtypes = [ctypes.c_int, ctypes.c_int, i64, ctypes.c_int, vp, vp, vp, vp]
        lib.bstq_solve_noalloc.restype = ctypes.c_int
        lib.bstq_solve_noalloc.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp,
                                           vp, P]
        _lib = lib
        return lib


def _params(no_sort=False, max_sweeps_per_n=0, scheduler=0, qstore=0, threads_per_block=0, kernel=0,
            back_transform=False, update_scheme=0, log_entries=0):
    if isinstance(update_scheme, str):
        update_scheme = {"exp": UPDATE_EXP, "pg": UPDATE_PG}[update_scheme.lower()]
    return Params(int(bool(no_sort)), int(max_sweeps_per_n), int(scheduler), int(qstore),
                  int(threads_per_block), int(kernel), int(bool(back_transform)), int(update_scheme),
                  int(log_entries))


def _dtype_code(dt) -> int:
    import torch
    if dt in (torch.float32, np.float32):
        return F32
    if dt in (torch.float64, np.float64):
        return F64
    raise TypeError(f"bstq: dtype must be float32 or float64, got {dt}")


def status_string(code: int) -> str:
    return load().bstq_status_string(int(code)).decode()


def version() -> str:
    return load().bstq_version().decode()


def work_size(dtype, jobz: bool, n: int, batch: int, **params) -> int:
    code = _dtype_code(dtype)
    p = _params(**params)
    return int(load().bstq_work_size_ex(code, int(bool(jobz)), int(n), int(batch), ctypes.byref(p)))


def describe(dtype, jobz: bool, n: int, batch: int, **params) -> str:
    p = _params(**params)
    buf = ctypes.create_string_buffer(256)
    rc = load().bstq_describe(_dtype_code(dtype), int(bool(jobz)), int(n), int(batch),
                              ctypes.byref(p), buf, 256)
    if rc != 0:
        raise BstqError(rc, "bstq_describe")
    return buf.value.decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def solve(d, e, jobz: bool = True, Q=None, work=None, stream=None, Z=None, **params):
    """Solve on CUDA tensors: ``d`` (batch, n) in/out (eigenvalues on exit),
    ``e`` (batch, n-1).  Returns (d, Q, info) where Q is (batch, n, n) with
    Q[b, :, j] the eigenvector of d[b, j] (None for jobz N) and info (batch,)
    int32.  With ``Z`` (batch, n, n) given, the rotations are right-applied to
    Z (back_transform) and the returned Q is Z times the eigenvectors; ``Q``
    given with ``back_transform=True`` is read as the basis in the library's
    storage layout (memory [b][j][i] = Z_ij).  Work is enqueued on ``stream``
    (default: torch's current stream); nothing is synchronised."""
    import torch
    if Z is not None:
        if not jobz:
            raise ValueError("bstq.solve: Z needs jobz = True")
        # storage layout of the library: memory [b][j][i] = Z_ij
        Q = Z.to(device=d.device, dtype=d.dtype).transpose(1, 2).contiguous()
        params["back_transform"] = True
    if not (d.is_cuda and d.is_contiguous()):
        raise ValueError("bstq.solve: d must be a contiguous CUDA tensor")
    if d.dim() != 2:
        raise ValueError("bstq.solve: d must be (batch, n)")
    batch, n = d.shape
    code = _dtype_code(d.dtype)
    if e is None or e.numel() == 0:
        e_ptr = None
    else:
        if not (e.is_cuda and e.is_contiguous() and e.dtype == d.dtype and e.numel() == batch * (n - 1)):
            raise ValueError("bstq.solve: e must be a contiguous CUDA tensor of d's dtype, (batch, n-1)")
        e_ptr = e.data_ptr()
    p = _params(**params)
    lib = load()
    wbytes = int(lib.bstq_work_size_ex(code, int(bool(jobz)), int(n), int(batch), ctypes.byref(p)))
    if wbytes == 0:
        raise BstqError(-10, "bstq_work_size_ex")
    if work is None:
        work = torch.empty(wbytes, dtype=torch.uint8, device=d.device)
    elif work.numel() * work.element_size() < wbytes:
        raise ValueError(f"bstq.solve: work needs {wbytes} bytes")
    if jobz and Q is None:
        Q = torch.empty((batch, n, n), dtype=d.dtype, device=d.device)
    # the library writes column-major per problem: memory [b][j][i] = Q_ij
    rc = lib.bstq_solve_ex(code, int(bool(jobz)), int(n), int(batch), d.data_ptr(), e_ptr,
                           Q.data_ptr() if jobz else None, work.data_ptr(), _stream_handle(stream),
                           ctypes.byref(p))
    if rc != 0:
        raise BstqError(rc, "bstq_solve_ex")
    info = work[: 4 * batch].view(torch.int32)
    Qout = Q.transpose(1, 2) if jobz else None
    return d, Qout, info


def host_work_size(dtype, jobz: bool, n: int, batch: int, **params) -> int:
    p = _params(**params)
    return int(load().bstq_host_work_size(_dtype_code(dtype), int(bool(jobz)), int(n), int(batch),
                                          ctypes.byref(p)))


def solve_host(h_d, h_e, h_Q, h_info, dev, stream=None, jobz: bool = True, **params):
    """End-to-end call on host buffers (pinned torch CPU tensors): copies in,
    solves and copies out on ``stream``; the caller synchronises."""
    batch, n = h_d.shape
    p = _params(**params)
    rc = load().bstq_solve_host(_dtype_code(h_d.dtype), int(bool(jobz)), int(n), int(batch),
                                h_d.data_ptr(), h_e.data_ptr() if h_e is not None and h_e.numel() else None,
                                h_Q.data_ptr() if jobz else None, h_info.data_ptr(), dev.data_ptr(),
                                _stream_handle(stream), ctypes.byref(p))
    if rc != 0:
        raise BstqError(rc, "bstq_solve_host")


def solve_noalloc(d, e, Q, info, stream=None, **params):
    """bstq_solve_noalloc on CUDA tensors (jobz = V): d (batch, n) in/out,
    e (batch, n-1), Q (batch, n, n) and info (batch,) int32 caller-owned; the
    eigenvector scratch is the library's fixed device array.  Returns
    (d, Q viewed with Q[b, :, j] the j-th eigenvector, info)."""
    batch, n = d.shape
    p = _params(**params)
    e_ptr = e.data_ptr() if e is not None and e.numel() else None
    rc = load().bstq_solve_noalloc(_dtype_code(d.dtype), JOBZ_V, int(n), int(batch), d.data_ptr(), e_ptr,
                                   Q.data_ptr(), info.data_ptr(), _stream_handle(stream), ctypes.byref(p))
    if rc != 0:
        raise BstqError(rc, "bstq_solve_noalloc")
    return d, Q.transpose(1, 2), info


def syev_work_size(dtype, jobz: bool, n: int, batch: int, **params) -> int:
    p = _params(**params)
    return int(load().bstq_syev_work_size(_dtype_code(dtype), int(bool(jobz)), int(n), int(batch),
                                          ctypes.byref(p)))


def syev(A, jobz: bool = True, work=None, stream=None, **params):
    """Fused small-n dense symmetric eigensolver on a CUDA tensor ``A``
    (batch, n, n), n <= 32, of which the lower triangle (A[b, i, j], i >= j)
    is read.  Returns (W, V, info): eigenvalues (batch, n) ascending,
    eigenvectors (batch, n, n) with V[b, :, j] that of W[b, j] (None for
    jobz N), info (batch,) int32.  Nothing is synchronised."""
    import torch
    if not A.is_cuda or A.dim() != 3 or A.shape[1] != A.shape[2]:
        raise ValueError("bstq.syev: A must be a (batch, n, n) CUDA tensor")
    batch, n, _ = A.shape
    code = _dtype_code(A.dtype)
    Ac = A.transpose(1, 2).contiguous()  # library layout: memory [b][j][i] = A_ij
    W = torch.empty((batch, n), dtype=A.dtype, device=A.device)
    Vs = torch.empty((batch, n, n), dtype=A.dtype, device=A.device) if jobz else None
    p = _params(**params)
    lib = load()
    wbytes = int(lib.bstq_syev_work_size(code, int(bool(jobz)), int(n), int(batch), ctypes.byref(p)))
    if wbytes == 0:
        raise BstqError(-10, "bstq_syev_work_size")
    if work is None:
        work = torch.empty(wbytes, dtype=torch.uint8, device=A.device)
    elif work.numel() * work.element_size() < wbytes:
        raise ValueError(f"bstq.syev: work needs {wbytes} bytes")
    rc = lib.bstq_syev(code, int(bool(jobz)), int(n), int(batch), Ac.data_ptr(), W.data_ptr(),
                       Vs.data_ptr() if jobz else None, work.data_ptr(), _stream_handle(stream), ctypes.byref(p))
    if rc != 0:
        raise BstqError(rc, "bstq_syev")
    info = work[: 4 * batch].view(torch.int32)
    return W, (Vs.transpose(1, 2) if jobz else None), info


def leaf_shape(n: int, leaf: int):
    """(L, F, t): the leaf size used, the number of full leaves and the rows
    of the shorter last leaf (0 if none), as bstq_stedc_leaves cuts a
    size-n problem."""
    L = min(int(leaf), int(n))
    return L, n // L, n % L


def stedc_leaves_work_size(dtype, jobz: bool, n: int, leaf: int, batch: int, **params) -> int:
    p = _params(**params)
    return int(load().bstq_stedc_leaves_work_size(_dtype_code(dtype), int(bool(jobz)), int(n), int(leaf),
                                                  int(batch), ctypes.byref(p)))


def stedc_leaves(d, e, leaf: int, jobz: bool = True, work=None, stream=None, **params):
    """Leaf solve of divide and conquer on CUDA tensors: ``d`` (batch, n)
    in/out, ``e`` (batch, n-1).  Each problem is torn into leaves of ``leaf``
    rows (the remainder last) and every leaf solved.  Returns (d, Qf, Qt,
    info): d holds each leaf's eigenvalues at its rows; Qf (batch, F, L, L)
    the full leaves' eigenvectors and Qt (batch, t, t) the last shorter
    leaf's (None if none), both with [..., :, j] the j-th eigenvector (None
    for jobz N); info (batch, leaves) int32.  Nothing is synchronised."""
    import torch
    if not (d.is_cuda and d.is_contiguous() and d.dim() == 2):
        raise ValueError("bstq.stedc_leaves: d must be a contiguous (batch, n) CUDA tensor")
    batch, n = d.shape
    code = _dtype_code(d.dtype)
    L, F, t = leaf_shape(n, leaf)
    e_ptr = None
    if n > 1:
        if not (e.is_cuda and e.is_contiguous() and e.dtype == d.dtype and e.numel() == batch * (n - 1)):
            raise ValueError("bstq.stedc_leaves: e must be a contiguous CUDA tensor of d's dtype, (batch, n-1)")
        e_ptr = e.data_ptr()
    p = _params(**params)
    lib = load()
    wbytes = int(lib.bstq_stedc_leaves_work_size(code, int(bool(jobz)), int(n), int(leaf), int(batch),
                                                 ctypes.byref(p)))
    if wbytes == 0:
        raise BstqError(-10, "bstq_stedc_leaves_work_size")
    if work is None:
        work = torch.empty(wbytes, dtype=torch.uint8, device=d.device)
    elif work.numel() * work.element_size() < wbytes:
        raise ValueError(f"bstq.stedc_leaves: work needs {wbytes} bytes")
    leaves = F + (1 if t else 0)
    info = torch.empty((batch, leaves), dtype=torch.int32, device=d.device)
    Q = torch.empty(batch * (F * L * L + t * t), dtype=d.dtype, device=d.device) if jobz else None
    rc = lib.bstq_stedc_leaves(code, int(bool(jobz)), int(n), int(leaf), int(batch), d.data_ptr(), e_ptr,
                               Q.data_ptr() if jobz else None, info.data_ptr(), work.data_ptr(),
                               _stream_handle(stream), ctypes.byref(p))
    if rc != 0:
        raise BstqError(rc, "bstq_stedc_leaves")
    Qf = Qt = None
    if jobz:
        # library layout: column-major blocks, full leaves first, then tails
        Qf = Q[: batch * F * L * L].view(batch, F, L, L).transpose(2, 3)
        if t:
            Qt = Q[batch * F * L * L:].view(batch, t, t).transpose(1, 2)
    return d, Qf, Qt, info


def diag(op: int, inp, count: int, arg: int = 0, stream=None):
    """bstq_diag on a CUDA tensor ``inp`` (float32 or float64, the records of
    ``count`` inputs back to back).  Returns the (count, values out) result
    tensor.  Nothing is synchronised."""
    import torch
    if not (inp.is_cuda and inp.is_contiguous()):
        raise ValueError("bstq.diag: inp must be a contiguous CUDA tensor")
    code = _dtype_code(inp.dtype)
    out_per = 256 if op == DIAG_FASTQ else DIAG_SHAPE[op][1]
    out = torch.empty((count, out_per), dtype=inp.dtype, device=inp.device)
    lib = load()
    wbytes = int(lib.bstq_diag_work_size(int(op), code, int(count)))
    if wbytes == 0:
        raise BstqError(-1, "bstq_diag_work_size")
    work = torch.empty(wbytes, dtype=torch.uint8, device=inp.device)
    rc = lib.bstq_diag(int(op), code, int(count), int(arg), inp.data_ptr(), out.data_ptr(), work.data_ptr(),
                       _stream_handle(stream))
    if rc != 0:
        raise BstqError(rc, "bstq_diag")
    return out
