"""bstq_solve_noalloc: the allocation-free entry point for callers that must
not allocate device memory while they solve (graph capture, allocator hooks,
fixed-buffer plugins, real-time loops).  It keeps the eigenvector scratch in a
fixed array inside the library.  These tests call it through the C ABI, twice
in a row (the array keeps the previous call's contents), and compare with the
regular entry point under the parity tolerances.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest

from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H
from tests.gpu_helpers import orth_err, run_gpu, tri_residual

pytestmark = pytest.mark.gpu

CASES = [(np.float64, 12, 3000), (np.float32, 16, 2000), (np.float64, 32, 700), (np.float32, 29, 1100),
         (np.float32, 8, 3000), (np.float64, 5, 2500), (np.float32, 1, 300), (np.float32, 48, 700),
         (np.float64, 40, 300)]


def _noalloc(d, e, Z=None, **params):
    """One call through the C ABI; with Z (batch, n, n) the call runs with
    back_transform and Z as the basis."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    lib = bstq.load()
    dev = torch.device("cuda:0")
    batch, n = d.shape
    dg = torch.from_numpy(np.ascontiguousarray(d)).to(dev)
    eg = torch.from_numpy(np.ascontiguousarray(e)).to(dev)
    if Z is not None:
        # library layout: memory [b][j][i] = Z_ij
        Q = torch.from_numpy(np.ascontiguousarray(np.swapaxes(Z, 1, 2))).to(dev)
        params["back_transform"] = True
    else:
        Q = torch.full((batch, n, n), float("nan"), dtype=dg.dtype, device=dev)
    info = torch.full((batch,), 7, dtype=torch.int32, device=dev)
    code = bstq.F32 if d.dtype == np.float32 else bstq.F64
    stream = torch.cuda.current_stream()
    prm = bstq._params(**params)
    rc = lib.bstq_solve_noalloc(code, bstq.JOBZ_V, n, batch, dg.data_ptr(), eg.data_ptr(),
                                Q.data_ptr(), info.data_ptr(), ctypes.c_void_p(stream.cuda_stream),
                                ctypes.byref(prm))
    assert rc == 0, bstq.status_string(rc)
    torch.cuda.synchronize()
    return dg.cpu().numpy(), Q.transpose(1, 2).cpu().numpy(), info.cpu().numpy()


@pytest.mark.parametrize("dt,n,batch", CASES)
def test_noalloc_matches_regular_entry_point_twice(dt, n, batch):
    for call in range(2):
        d, e = inputs.normal_problems(n, batch, dt, seed=40 + call)
        lam, Q, info = _noalloc(d, e)
        lam_r, Q_r, info_r = run_gpu(d, e)
        assert np.array_equal(info, info_r) and np.all(info == 0)
        tn = H.norm1(d, e).astype(np.float64)
        eps = H.eps_of(dt)
        assert np.all(np.abs(lam.astype(np.float64) - lam_r).max(1) <= H.lam_tol(n, dt, tn))
        assert not np.any(np.isnan(Q))
        assert np.all(tri_residual(d, e, lam, Q) <= 64 * n * eps * tn)
        assert np.all(orth_err(Q) <= 64 * n * eps)


def test_noalloc_rejects_what_it_cannot_hold():
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    lib = bstq.load()
    dummy = torch.empty(64, dtype=torch.float64, device="cuda")
    p = dummy.data_ptr()
    # more float64 n = 32 problems than 64 MiB of scratch holds: refused, no launch
    assert lib.bstq_solve_noalloc(bstq.F64, bstq.JOBZ_V, 32, 1 << 20, p, p, p, p, None, None) == -4
    # eigenvalues only need no scratch: this entry point is for jobz = V
    assert lib.bstq_solve_noalloc(bstq.F64, bstq.JOBZ_N, 32, 10, p, p, p, p, None, None) == -2
    # small n: the static-position kernel keeps Q in registers and has no
    # scratch variant, so forcing that family is refused (the default runs the
    # dynamic-position kernel instead)
    prm = bstq.Params(0, 0, 0, 0, 0, bstq.KERNEL_STATIC)
    assert lib.bstq_solve_noalloc(bstq.F32, bstq.JOBZ_V, 8, 10, p, p, p, p, None, ctypes.byref(prm)) == -10


def _regular(d, e, Z=None, **params):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dev = torch.device("cuda:0")
    dg = torch.from_numpy(np.ascontiguousarray(d)).to(dev)
    eg = torch.from_numpy(np.ascontiguousarray(e)).to(dev)
    Zt = torch.from_numpy(np.ascontiguousarray(Z)).to(dev) if Z is not None else None
    lam, Q, info = bstq.solve(dg, eg, jobz=True, Z=Zt, **params)
    torch.cuda.synchronize()
    return lam.cpu().numpy(), Q.cpu().numpy(), info.cpu().numpy()


@pytest.mark.parametrize("dt,n", [(np.float64, 12), (np.float32, 16), (np.float32, 7)])
def test_noalloc_keeps_back_transform_and_pg(dt, n):
    """The entry point rewrites the storage policy (and the kernel family for
    small float n); back_transform, the PG update scheme and the scheduler
    must reach the kernel unchanged.  Compared with the regular entry point
    under the same parameters."""
    batch = 1500
    d, e = inputs.normal_problems(n, batch, dt, seed=77)
    Z = inputs.orthogonal_bases(n, batch, dt, seed=78)
    tn = H.norm1(d, e).astype(np.float64)
    eps = H.eps_of(dt)
    for kw in (dict(Z=Z), dict(update_scheme=1), dict(Z=Z, update_scheme=1), dict(scheduler=2)):
        lam, V, info = _noalloc(d, e, **kw)
        lam_r, V_r, info_r = _regular(d, e, **kw)
        assert np.array_equal(info, info_r) and np.all(info == 0), kw
        assert np.all(np.abs(lam.astype(np.float64) - lam_r).max(1) <= H.lam_tol(n, dt, tn)), kw
        if "Z" in kw:
            res, orth = H.back_residual_orth(d, e, Z, lam, V)
            assert np.all(res <= 64 * n * eps * tn) and np.all(orth <= 64 * n * eps), kw
        else:
            assert np.all(tri_residual(d, e, lam, V) <= 64 * n * eps * tn), kw
            assert np.all(orth_err(V) <= 64 * n * eps), kw


def test_noalloc_large_call_then_small_call():
    """A large call leaves its eigenvectors' scratch in the shared array; a
    smaller call right after must not see any of it."""
    for dt, n, big, small in ((np.float64, 12, 40000, 37), (np.float32, 32, 12000, 5)):
        d, e = inputs.normal_problems(n, big, dt, seed=90)
        _noalloc(d, e)
        d2, e2 = inputs.normal_problems(n, small, dt, seed=91)
        lam, Q, info = _noalloc(d2, e2)
        lam_r, Q_r, info_r = run_gpu(d2, e2)
        tn = H.norm1(d2, e2).astype(np.float64)
        eps = H.eps_of(dt)
        assert np.array_equal(info, info_r) and np.all(info == 0)
        assert np.all(np.abs(lam.astype(np.float64) - lam_r).max(1) <= H.lam_tol(n, dt, tn))
        assert np.all(tri_residual(d2, e2, lam, Q) <= 64 * n * eps * tn)
        assert np.all(orth_err(Q) <= 64 * n * eps)
