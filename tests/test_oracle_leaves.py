"""Pins for the oracle's stedc leaf solve (the divide step of divide and
conquer followed by a steqr solve per leaf).  Each check compares against
something other than the oracle's own index arithmetic: the dense rank-one
identity T = diag(T_1, ..., T_m) + sum |beta| v v^T, a library eigensolver on
the dense torn blocks, the trace, and the exact special cases (no coupling at
the boundaries, a single leaf).  Planted tear mistakes must fail the
reassembly pin.  CPU only."""
import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H

DTYPES = [np.float32, np.float64]
SHAPES = [(1, 1), (5, 1), (5, 2), (16, 8), (37, 8), (64, 32), (70, 32), (33, 32), (12, 5), (9, 100)]


def _torn_dense(d_torn, e, starts, sizes):
    """Block-diagonal dense matrix of the leaves (long double)."""
    batch, n = d_torn.shape
    T = np.zeros((batch, n, n), dtype=np.longdouble)
    for s, m in zip(starts, sizes):
        T[:, s:s + m, s:s + m] = H.dense(d_torn[:, s:s + m], e[:, s:s + m - 1], np.longdouble)
    return T


def _reassembly_error(d, e, starts, sizes, d_torn):
    """max |diag(T_k) + sum_r |beta_r| v_r v_r^T - T| per problem, relative to
    the rounding a tear may commit (one ulp of each torn diagonal entry)."""
    batch, n = d.shape
    T = H.dense(d, e, np.longdouble)
    R = _torn_dense(d_torn, e, starts, sizes)
    el = np.asarray(e, dtype=np.longdouble)
    for r in starts[1:]:
        beta = el[:, r - 1]
        v = np.zeros((batch, n), dtype=np.longdouble)
        v[:, r - 1] = 1
        v[:, r] = np.sign(beta)
        R += np.abs(beta)[:, None, None] * v[:, :, None] * v[:, None, :]
    eps = H.eps_of(d.dtype)
    ea = np.abs(el)
    # row scale |d_i| + |e_{i-1}| + |e_i|: what the two subtractions can round
    scale = np.abs(np.asarray(d, dtype=np.longdouble))
    scale[:, 1:] += ea
    scale[:, :-1] += ea
    scale = np.maximum(scale, np.finfo(d.dtype).tiny)
    diag_err = np.abs(np.diagonal(R - T, axis1=1, axis2=2)) / (2 * eps * scale)
    off = R - T
    idx = np.arange(n)
    off[:, idx, idx] = 0
    # off-diagonal entries must reassemble exactly (|beta| sign(beta) = beta)
    return np.maximum(diag_err.max(axis=1).astype(np.float64),
                      np.where(np.abs(off).reshape(batch, -1).max(axis=1) > 0, np.inf, 0.0))


def test_partition():
    assert oracle.leaf_partition(70, 32) == ([0, 32, 64], [32, 32, 6])
    assert oracle.leaf_partition(64, 32) == ([0, 32], [32, 32])
    assert oracle.leaf_partition(5, 8) == ([0], [5])
    assert oracle.leaf_partition(1, 1) == ([0], [1])
    assert oracle.leaf_partition(7, 3) == ([0, 3, 6], [3, 3, 1])
    with pytest.raises(ValueError):
        oracle.leaf_partition(4, 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n,leaf", SHAPES)
def test_tear_reassembles_T(dt, n, leaf):
    d, e = inputs.normal_problems(n, 40, dt, seed=7 + n)
    starts, sizes, dtn = oracle.tear(d, e, leaf)
    assert dtn.dtype == d.dtype and sum(sizes) == n
    assert np.all(_reassembly_error(d, e, starts, sizes, dtn) <= 1.0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n,leaf", SHAPES)
def test_leaf_eigenpairs_solve_the_torn_blocks(dt, n, leaf):
    """Each leaf's eigenpairs against the dense torn block built from the
    definition (T's diagonal block with |beta| taken off next to each
    boundary), by numpy's eigvalsh and the residual / orthogonality bounds."""
    d, e = inputs.normal_problems(n, 40, dt, seed=70 + n)
    r = oracle.stedc_leaves(d, e, leaf, jobz=True)
    assert np.all(r.info == 0)
    T = H.dense(d, e, np.float64)
    el = np.asarray(e, dtype=np.float64)
    eps = H.eps_of(dt)
    for k, (s, m) in enumerate(zip(r.starts, r.sizes)):
        B = T[:, s:s + m, s:s + m].copy()
        if s > 0:
            B[:, 0, 0] -= np.abs(el[:, s - 1])
        if s + m < n:
            B[:, m - 1, m - 1] -= np.abs(el[:, s + m - 1])
        ref = np.linalg.eigvalsh(B)
        lam = r.lam[:, s:s + m].astype(np.float64)
        bn = np.abs(B).sum(axis=2).max(axis=1)
        # the torn entries carry one rounding each, inside the bound's slack
        assert np.all(np.abs(lam - ref).max(axis=1) <= H.lam_tol(m, dt, bn) + 4 * eps * bn)
        assert np.all(np.diff(lam, axis=1) >= 0)
        Q = r.Q[k].astype(np.longdouble)
        R = B.astype(np.longdouble) @ Q - Q * r.lam[:, None, s:s + m].astype(np.longdouble)
        O = np.swapaxes(Q, 1, 2) @ Q - np.eye(m, dtype=np.longdouble)
        assert np.all(np.abs(R).reshape(40, -1).max(axis=1) <= 64 * m * eps * bn + 4 * eps * bn)
        assert np.all(np.abs(O).reshape(40, -1).max(axis=1) <= 64 * m * eps)


@pytest.mark.parametrize("dt", DTYPES)
def test_trace_identity(dt):
    n, leaf = 50, 16
    d, e = inputs.normal_problems(n, 64, dt, seed=3)
    r = oracle.stedc_leaves(d, e, leaf, jobz=False)
    el = np.abs(np.asarray(e, dtype=np.longdouble))
    want = np.asarray(d, dtype=np.longdouble).sum(axis=1) - 2 * sum(el[:, s - 1] for s in r.starts[1:])
    got = np.asarray(r.lam, dtype=np.longdouble).sum(axis=1)
    tn = H.norm1(d, e)
    assert np.all(np.abs(got - want) <= 4 * n * H.eps_of(dt) * tn * n)


@pytest.mark.parametrize("dt", DTYPES)
def test_uncoupled_boundaries_give_the_spectrum(dt):
    """With e = 0 at every boundary the tear changes nothing (d_torn == d
    bit for bit) and the leaves' eigenvalues together are T's."""
    n, leaf = 40, 8
    d, e = inputs.normal_problems(n, 32, dt, seed=5)
    for s in range(leaf, n, leaf):
        e[:, s - 1] = 0
    r = oracle.stedc_leaves(d, e, leaf, jobz=True)
    assert np.array_equal(r.d_torn, d)
    ref = np.linalg.eigvalsh(H.dense(d, e))
    tn = H.norm1(d, e)
    got = np.sort(r.lam.astype(np.float64), axis=1)
    assert np.all(np.abs(got - ref).max(axis=1) <= H.lam_tol(n, dt, tn))


@pytest.mark.parametrize("dt", DTYPES)
def test_single_leaf_is_the_plain_solve(dt):
    n = 20
    d, e = inputs.normal_problems(n, 50, dt, seed=9)
    r = oracle.stedc_leaves(d, e, 32, jobz=True)
    s = oracle.steqr(d, e, jobz=True)
    assert r.starts == [0] and np.array_equal(r.d_torn, d)
    assert np.array_equal(r.lam, s.lam) and np.array_equal(r.Q[0], s.Q)
    assert np.array_equal(r.info[:, 0], s.info)


@pytest.mark.parametrize("dt", DTYPES)
def test_nonfinite_coupling_poisons_both_neighbours(dt):
    n, leaf = 24, 8
    d, e = inputs.normal_problems(n, 4, dt, seed=11)
    e[1, leaf - 1] = np.nan      # boundary between leaves 0 and 1
    e[2, 3] = np.inf             # inside leaf 0 only
    r = oracle.stedc_leaves(d, e, leaf, jobz=True)
    assert r.info[0].tolist() == [0, 0, 0] and r.info[3].tolist() == [0, 0, 0]
    assert r.info[1].tolist() == [-1, -1, 0]
    assert r.info[2].tolist() == [-1, 0, 0]
    assert np.all(np.isnan(r.lam[1, :2 * leaf])) and not np.any(np.isnan(r.lam[1, 2 * leaf:]))


# Planted tear mistakes: each must fail the reassembly pin.
def _mut_plus(d, e, leaf):
    starts, sizes, dt = oracle.tear(d, e, leaf)
    out = dt.copy()
    for r in starts[1:]:
        out[:, r] = out[:, r] + 2 * np.abs(e[:, r - 1])   # added instead of taken off
    return starts, sizes, out


def _mut_signed(d, e, leaf):
    starts, sizes, dt = oracle.tear(d, e, leaf)
    out = dt.copy()
    for r in starts[1:]:
        out[:, r - 1] = out[:, r - 1] + np.abs(e[:, r - 1]) - e[:, r - 1]   # beta, not |beta|
    return starts, sizes, out


def _mut_one_side(d, e, leaf):
    starts, sizes, dt = oracle.tear(d, e, leaf)
    out = dt.copy()
    for r in starts[1:]:
        out[:, r] = d[:, r] if r + 1 not in starts else out[:, r]   # upper side only
    return starts, sizes, out


def _mut_shifted(d, e, leaf):
    starts, sizes, dt = oracle.tear(d, e, leaf)
    out = d.copy()
    for r in starts[1:]:
        beta = np.abs(e[:, r - 2]) if r >= 2 else 0
        out[:, r - 1] = out[:, r - 1] - beta                # off by one boundary index
        out[:, r] = out[:, r] - beta
    return starts, sizes, out


@pytest.mark.parametrize("mutant", [_mut_plus, _mut_signed, _mut_one_side, _mut_shifted])
def test_planted_tear_mistakes_fail_the_pin(mutant):
    n, leaf = 37, 8
    d, e = inputs.normal_problems(n, 40, np.float64, seed=21)
    starts, sizes, dtn = mutant(d, e, leaf)
    assert np.any(_reassembly_error(d, e, starts, sizes, dtn) > 1.0)
