"""Shared checks for the tests: dense assembly, tolerances from the stated
bounds, and high-precision reference values.  None of this is the solver."""
from __future__ import annotations

import numpy as np

EPS = {np.dtype(np.float32): 2.0 ** -24, np.dtype(np.float64): 2.0 ** -53}


def eps_of(dtype) -> float:
    return EPS[np.dtype(dtype)]


def tiny_of(dtype) -> float:
    """Smallest positive subnormal of the dtype: the spacing of the grid a
    result with a subnormal magnitude is rounded to."""
    return float(np.finfo(dtype).smallest_subnormal)


def dense(d, e, dtype=np.float64):
    """Dense (batch, n, n) symmetric tridiagonal matrices."""
    d = np.asarray(d, dtype=dtype)
    if d.ndim == 1:
        d = d[None]
    batch, n = d.shape
    e = np.asarray(e, dtype=dtype).reshape(batch, max(n - 1, 0))
    T = np.zeros((batch, n, n), dtype=dtype)
    idx = np.arange(n)
    T[:, idx, idx] = d
    if n > 1:
        T[:, idx[:-1], idx[1:]] = e
        T[:, idx[1:], idx[:-1]] = e
    return T


def norm1(d, e):
    """||T||_1 (= ||T||_inf, the largest absolute row sum) in long double."""
    d = np.abs(np.asarray(d, dtype=np.longdouble))
    if d.ndim == 1:
        d = d[None]
    batch, n = d.shape
    e = np.abs(np.asarray(e, dtype=np.longdouble)).reshape(batch, max(n - 1, 0))
    rows = d.copy()
    if n > 1:
        rows[:, :-1] += e
        rows[:, 1:] += e
    return rows.max(axis=1)


def lam_tol(n, dtype, tnorm):
    """|lambda - lambda_ref| <= 16 n eps ||T||."""
    return 16.0 * n * eps_of(dtype) * np.asarray(tnorm, dtype=np.float64)


def lam_tol_sub(n, dtype, tnorm):
    """16 n eps ||T|| plus one subnormal spacing: where ||T|| is itself near or
    below the smallest normal number, every eigenvalue is rounded to the
    subnormal grid when it is scaled back, so two correct results can differ
    by that spacing however small 16 n eps ||T|| is.  For normal ||T|| the
    extra term is negligible.  Returned in long double, so that tolerances
    far below the dtype's own range stay exact."""
    return (np.longdouble(16.0 * n * eps_of(dtype)) * np.asarray(tnorm, dtype=np.longdouble)
            + np.longdouble(tiny_of(dtype)))


def tri_residual_ld(d, e, lam, Q):
    """max |T Q - Q Lambda| per problem from the band structure, in long
    double (exact products of subnormal entries, no overflow near the top of
    float64's range)."""
    ld = np.longdouble
    d = np.asarray(d, dtype=ld)
    e = np.asarray(e, dtype=ld).reshape(len(d), max(d.shape[1] - 1, 0))
    Qd = np.asarray(Q, dtype=ld)
    TQ = d[:, :, None] * Qd
    if d.shape[1] > 1:
        TQ[:, 1:, :] += e[:, :, None] * Qd[:, :-1, :]
        TQ[:, :-1, :] += e[:, :, None] * Qd[:, 1:, :]
    R = TQ - Qd * np.asarray(lam, dtype=ld)[:, None, :]
    return np.abs(R).reshape(len(d), -1).max(1)


def residual_orth(d, e, lam, Q):
    """max |T Q - Q Lambda| and max |Q^T Q - I| per problem, in long double."""
    T = dense(d, e, np.longdouble)
    Ql = np.asarray(Q, dtype=np.longdouble)
    L = np.asarray(lam, dtype=np.longdouble)
    n = T.shape[-1]
    R = T @ Ql - Ql * L[:, None, :]
    O = np.swapaxes(Ql, 1, 2) @ Ql - np.eye(n, dtype=np.longdouble)
    return (np.abs(R).reshape(len(T), -1).max(axis=1).astype(np.float64),
            np.abs(O).reshape(len(T), -1).max(axis=1).astype(np.float64))


def sturm_eigenvalues(d, e, dps: int = 50):
    """All eigenvalues of one tridiagonal matrix by Sturm-sequence bisection in
    mpmath at ``dps`` decimal digits (brute force for small n)."""
    import mpmath as mp
    mp.mp.dps = dps
    n = len(d)
    D = [mp.mpf(float(x)) for x in d]
    E = [mp.mpf(float(x)) for x in e]

    def count_below(x):
        cnt = 0
        q = D[0] - x
        if q < 0:
            cnt += 1
        for i in range(1, n):
            if q == 0:
                q = mp.mpf(10) ** (-2 * dps)
            q = D[i] - x - E[i - 1] ** 2 / q
            if q < 0:
                cnt += 1
        return cnt

    bound = sum(abs(x) for x in D) + 2 * sum(abs(x) for x in E) + 1
    out = []
    for k in range(n):
        lo, hi = -bound, bound
        for _ in range(int(dps * 3.33) + 10):
            mid = (lo + hi) / 2
            if count_below(mid) > k:
                hi = mid
            else:
                lo = mid
        out.append((lo + hi) / 2)
    return np.array([float(v) for v in out])


def toeplitz_eigenvalues(n, a, b):
    """Closed form for tridiag(b; a; b): a + 2 b cos(k pi / (n + 1)), k=1..n,
    evaluated in long double and returned ascending."""
    k = np.arange(1, n + 1, dtype=np.longdouble)
    pi = np.longdouble("3.14159265358979323846264338327950288")
    v = np.longdouble(a) + 2 * np.longdouble(b) * np.cos(k * pi / (n + 1))
    return np.sort(v)


def back_residual_orth(d, e, Z, lam, V):
    """For back_transform output V = Z Q: max |A V - V Lambda| with
    A = Z T Z^T, and max |V^T V - I|, per problem, in long double."""
    T = dense(d, e, np.longdouble)
    Zl = np.asarray(Z, dtype=np.longdouble)
    A = Zl @ T @ np.swapaxes(Zl, 1, 2)
    Vl = np.asarray(V, dtype=np.longdouble)
    L = np.asarray(lam, dtype=np.longdouble)
    n = T.shape[-1]
    R = A @ Vl - Vl * L[:, None, :]
    O = np.swapaxes(Vl, 1, 2) @ Vl - np.eye(n, dtype=np.longdouble)
    return (np.abs(R).reshape(len(T), -1).max(axis=1).astype(np.float64),
            np.abs(O).reshape(len(T), -1).max(axis=1).astype(np.float64))
