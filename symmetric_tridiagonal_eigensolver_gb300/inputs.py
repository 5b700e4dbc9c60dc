"""Seeded synthetic inputs for the batched tridiagonal eigensolver.

This module only draws numbers: it holds none of the solver's arithmetic and
is shared by the tests, the benchmark and the CPU oracle's callers, so that
the oracle and the CUDA library consume the very same arrays.

Workload (BatchLAS page "perf_steqr", setup paragraph): random normal d and e.
Generator: ``numpy.random.default_rng(seed)`` (PCG64); standard normals are
drawn in float64, in the order d (batch x n), then e (batch x (n-1)), then any
class extras, and are rounded to the problem's dtype last.
"""
from __future__ import annotations

import numpy as np

# Mixed hard-case batch: class name -> share of the batch.
MIXED_CLASSES = (
    ("normal", 0.60),      # d, e i.i.d. N(0,1)
    ("graded", 0.10),      # d_i = N(0,1) 10^(-i/2), e_i = N(0,1) 10^(-i/2)
    ("presplit", 0.10),    # each e_i zeroed with probability 1/4, at least one
    ("zero", 0.05),        # d = e = 0
    ("big", 0.05),         # N(0,1) scaled by 1e+18
    ("tiny", 0.05),        # N(0,1) scaled by 1e-18
    ("toeplitz", 0.05),    # d = a, e = b with a, b ~ N(0,1) per problem
)
CLASS_INDEX = {name: i for i, (name, _) in enumerate(MIXED_CLASSES)}


def _as_dtype(dtype) -> np.dtype:
    dt = np.dtype(dtype)
    if dt not in (np.float32, np.float64):
        raise TypeError("dtype must be float32 or float64")
    return dt


def normal_problems(n: int, batch: int, dtype, seed: int = 0):
    """d (batch, n) and e (batch, n-1), i.i.d. N(0,1), rounded to dtype."""
    dt = _as_dtype(dtype)
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((batch, n))
    e = rng.standard_normal((batch, max(n - 1, 0)))
    return d.astype(dt), e.astype(dt)


def class_counts(batch: int):
    """Problems per mixed class; the remainder of the rounding goes to
    'normal'."""
    counts = [int(np.floor(batch * share + 1e-9)) for _, share in MIXED_CLASSES]
    counts[0] += batch - sum(counts)
    return counts


def mixed_problems(n: int, batch: int, dtype, seed: int = 0, big: float = 1e18, tiny: float = 1e-18):
    """Mixed hard-case batch.  Returns d, e (rounded to dtype), the class label
    of each problem (int8, index into MIXED_CLASSES) and the Toeplitz (a, b)
    pair of each problem (float64 before rounding; meaningful only for the
    'toeplitz' class, whose stored d and e are a and b rounded to dtype).
    ``big`` and ``tiny`` are the factors of the 'big' and 'tiny' classes
    (1e+18 and 1e-18 as the workload states; other values, e.g. powers of two
    beyond float64's scaling thresholds, give the same draws rescaled)."""
    dt = _as_dtype(dtype)
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((batch, n))
    e = rng.standard_normal((batch, max(n - 1, 0)))
    counts = class_counts(batch)
    labels = rng.permutation(np.repeat(np.arange(len(MIXED_CLASSES), dtype=np.int8), counts))
    split_mask = rng.random((batch, max(n - 1, 0))) < 0.25
    forced = rng.integers(0, max(n - 1, 1), size=batch)
    ab = rng.standard_normal((batch, 2))

    grade = 10.0 ** (-np.arange(n) / 2.0)
    g = labels == CLASS_INDEX["graded"]
    d[g] *= grade[None, :]
    e[g] *= grade[None, : max(n - 1, 0)]

    p = labels == CLASS_INDEX["presplit"]
    if n > 1:
        m = split_mask.copy()
        m[np.arange(batch), forced] = True
        e[p] = np.where(m[p], 0.0, e[p])

    z = labels == CLASS_INDEX["zero"]
    d[z] = 0.0
    e[z] = 0.0

    b = labels == CLASS_INDEX["big"]
    d[b] *= big
    e[b] *= big
    t = labels == CLASS_INDEX["tiny"]
    d[t] *= tiny
    e[t] *= tiny

    tp = labels == CLASS_INDEX["toeplitz"]
    d[tp] = ab[tp, 0:1]
    e[tp] = ab[tp, 1:2]
    return d.astype(dt), e.astype(dt), labels, ab


# Exponents k of the scaled-extremes inputs (N(0,1) problems times 2^k), per
# precision: unscaled, above the down-scaling threshold ssfmax (twice, the
# second close to overflow), below the up-scaling threshold ssfmin, low
# enough that squared entries fall under the smallest normal number, and two
# with a subnormal block norm (the second, in float32, so deep that
# ssfmin / norm would overflow without the exact power-of-two lift).
SCALE_EXPONENTS = {
    np.dtype(np.float32): (0, 64, 120, -70, -100, -140, -146),
    np.dtype(np.float64): (0, 520, 1000, -420, -530, -1060),
}


def scaled_problems(n: int, batch: int, dtype, seed: int = 0, exponents=None):
    """N(0,1) problems, problem b multiplied by 2^k_b with k_b taken in turn
    from ``exponents`` (default SCALE_EXPONENTS of the dtype).  The product is
    formed exactly in float64 (np.ldexp) and rounded to dtype last, so
    subnormal results are the correctly rounded values.  Returns d, e and k
    (int32, per problem)."""
    dt = _as_dtype(dtype)
    exps = np.asarray(SCALE_EXPONENTS[dt] if exponents is None else exponents, dtype=np.int32)
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((batch, n))
    e = rng.standard_normal((batch, max(n - 1, 0)))
    k = exps[np.arange(batch) % len(exps)]
    d = np.ldexp(d, k[:, None])
    e = np.ldexp(e, k[:, None])
    return d.astype(dt), e.astype(dt), k


def block_scaled_problems(n: int, batch: int, dtype, seed: int = 0, exponents=None):
    """Two blocks per problem with different scales: N(0,1) d and e, the
    off-diagonal at a random row r (1 <= r <= n-1) set to zero, rows [0, r)
    multiplied by 2^k1 and rows [r, n) by 2^k2, k1 and k2 drawn from
    ``exponents`` (default SCALE_EXPONENTS of the dtype).  n >= 2.  Returns
    d, e, r, k1, k2."""
    dt = _as_dtype(dtype)
    exps = np.asarray(SCALE_EXPONENTS[dt] if exponents is None else exponents, dtype=np.int32)
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((batch, n))
    e = rng.standard_normal((batch, n - 1))
    r = rng.integers(1, n, size=batch)
    k1 = exps[rng.integers(0, len(exps), size=batch)]
    k2 = exps[rng.integers(0, len(exps), size=batch)]
    rows = np.arange(n)[None, :]
    kd = np.where(rows < r[:, None], k1[:, None], k2[:, None])
    e[np.arange(batch), r - 1] = 0.0
    d = np.ldexp(d, kd)
    e = np.ldexp(e, kd[:, : n - 1])
    return d.astype(dt), e.astype(dt), r, k1, k2


def problems(kind: str, n: int, batch: int, dtype, seed: int = 0):
    """``kind`` is 'normal' or 'mixed'; returns (d, e)."""
    if kind == "normal":
        return normal_problems(n, batch, dtype, seed)
    if kind == "mixed":
        d, e, _, _ = mixed_problems(n, batch, dtype, seed)
        return d, e
    raise ValueError(f"unknown input kind {kind!r}")


def orthogonal_bases(n: int, batch: int, dtype, seed: int = 0):
    """Z (batch, n, n) with Z[b] orthogonal (to the dtype's rounding): the Q
    factor of a matrix of i.i.d. N(0,1) entries (numpy's QR in float64),
    columns signed so that R has a positive diagonal, rounded to dtype.  Used
    as the basis Z of the back_transform case (Q on exit = Z times the
    eigenvectors)."""
    dt = _as_dtype(dtype)
    rng = np.random.default_rng(seed)
    G = rng.standard_normal((batch, n, n))
    Qf, R = np.linalg.qr(G)
    sgn = np.sign(np.diagonal(R, axis1=1, axis2=2))
    sgn[sgn == 0] = 1.0
    return (Qf * sgn[:, None, :]).astype(dt)


def dense_symmetric(n: int, batch: int, dtype, seed: int = 0):
    """A (batch, n, n) symmetric with i.i.d. N(0,1) entries on and below the
    diagonal (mirrored above), rounded to dtype: the dense input of the fused
    small-n syev."""
    dt = _as_dtype(dtype)
    rng = np.random.default_rng(seed)
    G = rng.standard_normal((batch, n, n))
    L = np.tril(G)
    A = L + np.swapaxes(np.tril(G, -1), 1, 2)
    return A.astype(dt)
