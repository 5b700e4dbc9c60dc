"""Fused small-n syev on the GPU (BatchLAS page "perf_steqr": reduction to
tridiagonal form, steqr solve and back-transform in one kernel) against the
oracle's syev on the same seeded dense matrices: eigenvalues within
16 n eps ||A||, the residual ||A V - V Lambda|| within 64 n eps ||A||,
orthogonality within 64 n eps, info exactly."""
import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _gpu_syev(A, jobz=True, **params):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    Ag = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    W, V, info = bstq.syev(Ag, jobz=jobz, **params)
    torch.cuda.synchronize()
    return W.cpu().numpy(), (V.cpu().numpy() if jobz else None), info.cpu().numpy().copy()


def _check(A, W, V, info, ref, what=""):
    dt = A.dtype
    n = A.shape[1]
    eps = H.eps_of(dt)
    np.testing.assert_array_equal(info, ref.info, err_msg=what)
    ok = info == 0
    an = np.abs(A.astype(np.float64)).sum(1).max(1)
    err = np.abs(W[ok].astype(np.float64) - ref.lam[ok].astype(np.float64)).max(1)
    assert np.all(err <= 16 * n * eps * an[ok]), what
    assert np.all(np.diff(W[ok], axis=1) >= 0), what
    if V is not None:
        Al = A[ok].astype(np.longdouble)
        Vl = V[ok].astype(np.longdouble)
        R = Al @ Vl - Vl * W[ok].astype(np.longdouble)[:, None, :]
        assert np.all(np.abs(R).reshape(ok.sum(), -1).max(1).astype(np.float64) <= 64 * n * eps * an[ok]), what
        O = np.swapaxes(Vl, 1, 2) @ Vl - np.eye(n, dtype=np.longdouble)
        assert np.abs(O).max() <= 64 * n * eps, what


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("jobz", [True, False])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 12, 16, 21, 32])
def test_syev_matches_oracle(dt, n, jobz):
    A = inputs.dense_symmetric(n, 1500 + 7 * n, dt, seed=400 + n)
    ref = oracle.syev(A, jobz=jobz, nthreads=8)
    W, V, info = _gpu_syev(A, jobz=jobz)
    _check(A, W, V, info, ref, what=f"syev n={n} jobz={jobz}")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_syev_full_batch_and_schedulers(dt):
    n = 16 if dt == np.float32 else 12
    A = inputs.dense_symmetric(n, 32768, dt, seed=410)
    ref = oracle.syev(A, jobz=True, nthreads=16)
    W, V, info = _gpu_syev(A)
    _check(A, W, V, info, ref, what="full batch")
    W2, V2, info2 = _gpu_syev(A[:3000], scheduler=2)
    np.testing.assert_array_equal(W2, W[:3000])
    np.testing.assert_array_equal(V2, V[:3000])
    W3, V3, info3 = _gpu_syev(A[:3000], update_scheme=1)
    _check(A[:3000], W3, V3, info3, oracle.syev(A[:3000], jobz=True, nthreads=8, scheme="pg"), what="pg")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_syev_of_tridiagonal_input_equals_steqr(dt):
    """No reflector has anything to annihilate: d and e pass through and the
    basis is the identity, so the result is the tridiagonal solve's."""
    from tests.gpu_helpers import run_gpu
    n = 13
    d, e = inputs.normal_problems(n, 2000, dt, seed=411)
    A = H.dense(d, e, dtype=dt)
    W, V, info = _gpu_syev(A)
    lam, Q, inf2 = run_gpu(d, e, kernel=2)
    np.testing.assert_array_equal(W, lam)
    np.testing.assert_array_equal(V, Q)
    np.testing.assert_array_equal(info, inf2)


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_syev_degenerate_and_nonfinite(dt):
    n = 10
    A = inputs.dense_symmetric(n, 300, dt, seed=412)
    A[5] = 0
    A[6] = np.diag(np.arange(n, 0, -1)).astype(dt)
    A[7, 4, 2] = np.nan          # lower triangle: poisons problem 7
    A[8, 1, 6] = np.inf          # upper triangle: not read
    ref = oracle.syev(A, jobz=True)
    W, V, info = _gpu_syev(A)
    assert info[7] == -1 and np.all(np.isnan(W[7])) and np.all(np.isnan(V[7]))
    assert info[8] == 0
    assert np.all(W[5] == 0) and np.all(V[5] == np.eye(n, dtype=dt))
    np.testing.assert_array_equal(W[6], np.arange(1, n + 1, dtype=dt))
    keep = np.ones(len(A), bool)
    keep[7] = False
    A8 = A.copy()
    A8[8, 1, 6] = A8[8, 6, 1]
    _check(A8[keep], W[keep], V[keep], info[keep], oracle.syev(A8[keep], jobz=True))


def test_syev_rejects_what_it_does_not_run():
    import ctypes
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    lib = bstq.load()
    p = ctypes.c_void_p(256)
    assert lib.bstq_syev(bstq.F32, bstq.JOBZ_V, 33, 10, p, p, p, p, None, None) == -3
    prm = bstq.Params(0, 0, 0, 0, 0, 0, 1, 0)  # back_transform
    assert lib.bstq_syev(bstq.F32, bstq.JOBZ_V, 8, 10, p, p, p, p, None, ctypes.byref(prm)) == -10
    assert lib.bstq_syev_work_size(bstq.F32, bstq.JOBZ_V, 33, 10, None) == 0
