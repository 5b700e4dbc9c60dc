"""Helpers for the GPU parity tests: run the CUDA library through the C ABI
and compare with the oracle under the stated tolerances."""
from __future__ import annotations

import os

import numpy as np

import oracle
from tests import helpers as H

ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))


def run_gpu(d, e, jobz=True, **params):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dev = torch.device("cuda:0")
    dg = torch.from_numpy(np.ascontiguousarray(d)).to(dev)
    eg = torch.from_numpy(np.ascontiguousarray(e)).to(dev)
    Q = None
    if jobz:
        batch, n = d.shape
        # poison: every entry must be written
        Q = torch.full((batch, n, n), float("nan"), dtype=dg.dtype, device=dev)
    lam, Qt, info = bstq.solve(dg, eg, jobz=jobz, Q=Q, **params)
    torch.cuda.synchronize()
    return (lam.cpu().numpy(), Qt.cpu().numpy() if jobz else None, info.cpu().numpy().copy())


def tri_residual(d, e, lam, Q):
    """max |T Q - Q Lambda| per problem in float64 using the band structure."""
    d = d.astype(np.float64)
    e = e.astype(np.float64)
    Qd = Q.astype(np.float64)
    TQ = d[:, :, None] * Qd
    if d.shape[1] > 1:
        TQ[:, 1:, :] += e[:, :, None] * Qd[:, :-1, :]
        TQ[:, :-1, :] += e[:, :, None] * Qd[:, 1:, :]
    R = TQ - Qd * lam.astype(np.float64)[:, None, :]
    return np.abs(R).reshape(len(d), -1).max(1)


def orth_err(Q):
    Qd = Q.astype(np.float64)
    n = Qd.shape[-1]
    out = np.empty(len(Qd))
    for s in range(0, len(Qd), 4096):
        O = np.swapaxes(Qd[s:s + 4096], 1, 2) @ Qd[s:s + 4096] - np.eye(n)
        out[s:s + 4096] = np.abs(O).reshape(len(O), -1).max(1)
    return out


def check_parity(d, e, lam, Q, info, ref, what=""):
    """Spec bounds: |lambda - lambda_oracle| <= 16 n eps ||T||,
    ||T Q - Q Lambda||_max <= 64 n eps ||T||, ||Q^T Q - I||_max <= 64 n eps;
    info and non-finite handling exactly equal.  The first two bounds get one
    subnormal spacing added (negligible unless ||T|| is near or below the
    smallest normal number, where scaled-back results are rounded to the
    subnormal grid), and the residual of a float64 problem whose norm is far
    outside [2^-900, 2^900] is computed in long double."""
    dt = d.dtype
    n = d.shape[1]
    eps = H.eps_of(dt)
    tiny = H.tiny_of(dt)
    assert np.array_equal(info, ref.info), f"{what}: info differs at {np.nonzero(info != ref.info)[0][:10]}"
    bad = info == -1
    assert np.all(np.isnan(lam[bad])), f"{what}: poisoned problems must return NaN eigenvalues"
    ok = info == 0
    tnl = H.norm1(d, e)
    tn = tnl.astype(np.float64)
    if n:
        err = np.abs(lam[ok].astype(np.longdouble) - ref.lam[ok].astype(np.longdouble)).max(1)
        tol = H.lam_tol_sub(n, dt, tnl[ok])
        assert np.all(err <= tol), \
            f"{what}: eigenvalue error {float(np.max(err / np.maximum(tnl[ok], 1e-300))):.3e} x||T||"
    if Q is not None:
        assert np.all(np.isnan(Q[bad])), f"{what}: poisoned problems must return NaN eigenvectors"
        assert not np.any(np.isnan(Q[~bad])), f"{what}: unwritten or NaN Q entries"
        res = tri_residual(d[ok], e[ok], lam[ok], Q[ok]).astype(np.longdouble)
        extreme = (tn[ok] < 2.0 ** -900) | (tn[ok] > 2.0 ** 900)
        if dt == np.float64 and np.any(extreme):
            idx = np.nonzero(ok)[0][extreme]
            res[extreme] = H.tri_residual_ld(d[idx], e[idx], lam[idx], Q[idx])
        rtol = np.longdouble(64 * n * eps) * tnl[ok] + np.longdouble(tiny)
        assert np.all(res <= rtol), f"{what}: residual {float(np.max(res / np.maximum(tnl[ok], 1e-300))):.3e}"
        orth = orth_err(Q[~bad])
        assert np.all(orth <= 64 * n * eps), f"{what}: orthogonality {orth.max():.3e}"
    # ascending
    assert np.all(np.diff(lam[ok], axis=1) >= 0), f"{what}: not ascending"


def oracle_ref(d, e, jobz=True, **kw):
    return oracle.steqr(d, e, jobz=jobz, nthreads=ORACLE_THREADS, **kw)
