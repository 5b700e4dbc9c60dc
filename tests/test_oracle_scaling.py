"""Pins for the oracle's per-block scaling (BatchLAS page "algo_steqr", the
scaling paragraph after the deflation criterion): a block whose max-abs norm
lies above ssfmax or below ssfmin is multiplied by ssfmax/norm or
ssfmin/norm before it is iterated and by the inverse afterwards, a subnormal
norm being first lifted by an exact power of two.

Every input here is N(0,1) times an exact power of two 2^k chosen so that a
branch of that step runs in the problem's precision (above ssfmax, near
overflow, below ssfmin, squares below the smallest normal, subnormal norms).
The stored matrix T_s is scaled back exactly, T = 2^-k T_s, so the reference
is 2^k times the spectrum of a well-scaled matrix: numpy's eigvalsh, or
Sturm bisection in 50-digit arithmetic for n <= 6.  The bound is
16 n eps ||T_s|| plus one subnormal spacing (results below the smallest
normal are rounded to the subnormal grid when they are scaled back).
CPU only."""
import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H

DTYPES = [np.float32, np.float64]
LD = np.longdouble


def _reference(d, e, k):
    """2^k eigvalsh(2^-k T_s) per problem, in long double."""
    dr = np.ldexp(d.astype(np.float64), -k[:, None])
    er = np.ldexp(e.astype(np.float64), -k[:, None])
    lam = np.linalg.eigvalsh(H.dense(dr, er))
    return np.ldexp(lam.astype(LD), k[:, None].astype(np.int32))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [2, 7, 16, 32])
def test_scaled_extremes_against_rescaled_library(dt, n):
    d, e, k = inputs.scaled_problems(n, 14 * len(inputs.SCALE_EXPONENTS[np.dtype(dt)]), dt, seed=40 + n)
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    tn = H.norm1(d, e)
    ref = _reference(d, e, k)
    err = np.abs(r.lam.astype(LD) - ref).max(1)
    tol = H.lam_tol_sub(n, dt, tn)
    assert np.all(err <= tol), [(int(k[i]), float(err[i] / tol[i])) for i in np.nonzero(err > tol)[0][:5]]
    # eigenpairs of the stored (scaled) matrix, computed in long double
    res = H.tri_residual_ld(d, e, r.lam, r.Q)
    eps = H.eps_of(dt)
    assert np.all(res <= LD(64 * n * eps) * tn + LD(H.tiny_of(dt))), (res / tn).max()
    orth = np.abs(np.swapaxes(r.Q.astype(np.float64), 1, 2) @ r.Q.astype(np.float64) - np.eye(n)).max((1, 2))
    assert np.all(orth <= 64 * n * eps)


@pytest.mark.parametrize("dt", DTYPES)
def test_scaled_extremes_against_sturm_bisection(dt):
    """Brute force for n <= 6: bisection on 2^-k T_s in 50 digits, times 2^k."""
    for n in (3, 6):
        d, e, k = inputs.scaled_problems(n, 2 * len(inputs.SCALE_EXPONENTS[np.dtype(dt)]), dt, seed=60 + n)
        r = oracle.steqr(d, e, jobz=False)
        tn = H.norm1(d, e)
        for b in range(len(d)):
            dr = np.ldexp(d[b].astype(np.float64), -int(k[b]))
            er = np.ldexp(e[b].astype(np.float64), -int(k[b]))
            st = np.ldexp(H.sturm_eigenvalues(dr, er).astype(LD), int(k[b]))
            err = np.abs(r.lam[b].astype(LD) - st).max()
            assert err <= H.lam_tol_sub(n, dt, tn[b]), (n, int(k[b]), float(err / tn[b]))


@pytest.mark.parametrize("dt", DTYPES)
def test_scaling_commutes_with_powers_of_two(dt):
    """lambda(2^k T) = 2^k lambda(T) where 2^k T is exact (no subnormal
    result): the scaled runs take the scaling branches, the reference run
    does not."""
    n = 12
    d, e = inputs.normal_problems(n, 60, dt, seed=70)
    base = oracle.steqr(d, e, jobz=False)
    tn = H.norm1(d, e)
    ks = (64, 120, -70, -100) if dt == np.float32 else (520, 1000, -420, -530, -900)
    for kk in ks:
        ds, es = np.ldexp(d, kk).astype(dt), np.ldexp(e, kk).astype(dt)
        assert np.array_equal(np.ldexp(ds, -kk), d)       # exact
        r = oracle.steqr(ds, es, jobz=False)
        assert np.all(r.info == 0)
        err = np.abs(r.lam.astype(LD) - np.ldexp(base.lam.astype(LD), kk)).max(1)
        assert np.all(err <= np.ldexp(2 * H.lam_tol(n, dt, tn).astype(LD), kk)), kk


@pytest.mark.parametrize("dt", DTYPES)
def test_blocks_are_scaled_independently(dt):
    """Two blocks of very different scale in one problem: each block's
    eigenpairs match its own rescaled library spectrum to its own norm, and
    every eigenvector lives on exactly one block."""
    n = 20
    d, e, rsplit, k1, k2 = inputs.block_scaled_problems(n, 300, dt, seed=80)
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    for b in range(len(d)):
        rb = int(rsplit[b])
        top = np.abs(r.Q[b, :rb, :]).sum(0) > 0
        bot = np.abs(r.Q[b, rb:, :]).sum(0) > 0
        assert np.all(top ^ bot), b                          # one block per eigenvector
        for sel, lo, hi, kk in ((top, 0, rb, int(k1[b])), (bot, rb, n, int(k2[b]))):
            db, eb = d[b, lo:hi], e[b, lo:hi - 1]
            assert np.count_nonzero(sel) == hi - lo
            dr = np.ldexp(db.astype(np.float64), -kk)
            er = np.ldexp(eb.astype(np.float64), -kk)
            ref = np.ldexp(np.linalg.eigvalsh(H.dense(dr, er))[0].astype(LD), kk)
            got = np.sort(r.lam[b][sel].astype(LD))
            tn = H.norm1(db[None], eb[None])[0]
            assert np.abs(got - ref).max() <= H.lam_tol_sub(hi - lo, dt, tn), (b, kk)
