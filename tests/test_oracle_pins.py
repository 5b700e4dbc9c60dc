"""Pins for the CPU oracle: each test checks the oracle against something other
than itself (closed forms, Sturm bisection, a library eigensolver, invariants,
exact special cases).  CPU only."""
import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H

DTYPES = [np.float32, np.float64]


def test_constants_match_definitions():
    for dt in DTYPES:
        c = oracle.constants(dt)
        fi = np.finfo(dt)
        eps = float(fi.eps) / 2.0                      # unit roundoff
        safmin = float(fi.smallest_normal)
        assert c["eps"] == eps
        assert c["safmin"] == safmin
        assert c["ssfmax"] == float(dt(np.sqrt(1.0 / safmin)) / dt(3.0))
        assert c["ssfmin"] == float(np.sqrt(safmin) / eps ** 2)


@pytest.mark.parametrize("dt", DTYPES)
def test_n1_is_exact(dt):
    d = np.array([[3.5], [-0.0], [1e-30]], dtype=dt)
    r = oracle.steqr(d, np.zeros((3, 0), dt), jobz=True)
    assert np.array_equal(r.lam, d)
    assert np.all(r.Q == 1) and np.all(r.info == 0)
    assert (r.sweeps, r.rotations, r.solves2x2) == (0, 0, 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_n2_closed_form(dt):
    import mpmath as mp
    mp.mp.dps = 40
    rng = np.random.default_rng(11)
    d = rng.standard_normal((200, 2)).astype(dt)
    e = rng.standard_normal((200, 1)).astype(dt)
    d[:20, 1] = d[:20, 0]                                  # tau = 0 case
    r = oracle.steqr(d, e, jobz=True)
    assert r.solves2x2 == 200 and r.sweeps == 0 and r.rotations == 0
    tn = H.norm1(d, e)
    for b in range(200):
        a, c, bb = (mp.mpf(float(x)) for x in (d[b, 0], d[b, 1], e[b, 0]))
        rt = mp.sqrt(((a - c) / 2) ** 2 + bb ** 2)
        ref = sorted([float((a + c) / 2 - rt), float((a + c) / 2 + rt)])
        assert np.max(np.abs(r.lam[b] - ref)) <= H.lam_tol(2, dt, tn[b])
    res, orth = H.residual_orth(d, e, r.lam, r.Q)
    assert np.all(res <= 64 * 2 * H.eps_of(dt) * tn)
    assert np.all(orth <= 64 * 2 * H.eps_of(dt))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [3, 4, 5, 7, 8, 12, 16, 17, 24, 31, 32])
def test_toeplitz_closed_form(dt, n):
    rng = np.random.default_rng(100 + n)
    ab = rng.standard_normal((64, 2)).astype(dt)
    d = np.repeat(ab[:, :1], n, axis=1)
    e = np.repeat(ab[:, 1:], n - 1, axis=1)
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    tn = H.norm1(d, e)
    for b in range(64):
        ref = H.toeplitz_eigenvalues(n, ab[b, 0], ab[b, 1])
        err = np.max(np.abs(r.lam[b].astype(np.longdouble) - ref))
        assert err <= H.lam_tol(n, dt, tn[b]), (b, err)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [3, 4, 5, 6])
def test_sturm_bisection_small_n(dt, n):
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(7 * n)
    d = rng.standard_normal((12, n)).astype(dt)
    e = rng.standard_normal((12, n - 1)).astype(dt)
    d[0] *= 1e-3                                       # a graded-ish item
    r = oracle.steqr(d, e, jobz=False)
    tn = H.norm1(d, e)
    for b in range(12):
        ref = H.sturm_eigenvalues(d[b], e[b])
        err = np.max(np.abs(r.lam[b].astype(np.float64) - ref))
        assert err <= H.lam_tol(n, dt, tn[b]), (b, err)
        # much tighter than the stated bound in practice
        assert err <= 4 * n * H.eps_of(dt) * tn[b]


def test_sturm_spot_check_n32():
    pytest.importorskip("mpmath")
    d, e = inputs.normal_problems(32, 3, np.float64, seed=5)
    r = oracle.steqr(d, e, jobz=False)
    tn = H.norm1(d, e)
    for b in range(3):
        ref = H.sturm_eigenvalues(d[b], e[b], dps=30)
        assert np.max(np.abs(r.lam[b] - ref)) <= H.lam_tol(32, np.float64, tn[b])


@pytest.mark.parametrize("dt", DTYPES)
def test_against_library_eigh_all_n(dt):
    for n in range(1, 33):
        d, e = inputs.normal_problems(n, 48, dt, seed=n)
        r = oracle.steqr(d, e, jobz=True)
        assert np.all(r.info == 0)
        T = H.dense(d, e)
        ref = np.linalg.eigvalsh(T)
        tn = H.norm1(d, e)
        err = np.abs(r.lam.astype(np.float64) - ref).max(axis=1)
        assert np.all(err <= H.lam_tol(n, dt, tn)), (n, err.max())
        res, orth = H.residual_orth(d, e, r.lam, r.Q)
        assert np.all(res <= 64 * n * H.eps_of(dt) * tn), (n, res.max())
        assert np.all(orth <= 64 * n * H.eps_of(dt)), (n, orth.max())
        # ascending
        assert np.all(np.diff(r.lam, axis=1) >= 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [40, 64, 65, 96, 127, 128])
def test_against_library_eigh_large_n(dt, n):
    """Sizes above the sub-group width, up to the oracle's largest (128)."""
    d, e = inputs.normal_problems(n, 12, dt, seed=500 + n)
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    tn = H.norm1(d, e)
    ref = np.linalg.eigvalsh(H.dense(d, e))
    assert np.all(np.abs(r.lam.astype(np.float64) - ref).max(axis=1) <= H.lam_tol(n, dt, tn))
    res, orth = H.residual_orth(d, e, r.lam, r.Q)
    assert np.all(res <= 64 * n * H.eps_of(dt) * tn) and np.all(orth <= 64 * n * H.eps_of(dt))
    # Toeplitz closed form at the same size
    cf = H.toeplitz_eigenvalues(n, 0.5, -1.25)
    rt = oracle.steqr(np.full((1, n), 0.5, dt), np.full((1, n - 1), -1.25, dt), jobz=False)
    assert np.max(np.abs(rt.lam[0] - cf)) <= H.lam_tol(n, dt, 0.5 + 2.5)
    with pytest.raises(ValueError):
        oracle.steqr(np.zeros((1, 129), dt), np.zeros((1, 128), dt))


@pytest.mark.parametrize("dt", DTYPES)
def test_trace_and_frobenius_invariants(dt):
    n = 20
    d, e = inputs.normal_problems(n, 200, dt, seed=3)
    r = oracle.steqr(d, e, jobz=False)
    L = r.lam.astype(np.longdouble)
    dl, el = d.astype(np.longdouble), e.astype(np.longdouble)
    tn = H.norm1(d, e).astype(np.float64)
    tr_err = np.abs(L.sum(1) - dl.sum(1)).astype(np.float64)
    fr_err = np.abs((L ** 2).sum(1) - (dl ** 2).sum(1) - 2 * (el ** 2).sum(1)).astype(np.float64)
    assert np.all(tr_err <= n * H.lam_tol(n, dt, tn))
    assert np.all(fr_err <= 2 * n * H.lam_tol(n, dt, tn) * tn)


@pytest.mark.parametrize("dt", DTYPES)
def test_eigenvectors_match_library_up_to_sign(dt):
    n = 12
    d, e = inputs.normal_problems(n, 100, np.float64, seed=21)
    d, e = d.astype(dt), e.astype(dt)
    r = oracle.steqr(d, e, jobz=True)
    w, V = np.linalg.eigh(H.dense(d, e))
    checked = 0
    for b in range(100):
        gaps = np.diff(w[b])
        for j in range(n):
            gap = min(gaps[j - 1] if j > 0 else np.inf, gaps[j] if j < n - 1 else np.inf)
            if gap < 0.1:
                continue
            q = r.Q[b, :, j].astype(np.float64)
            v = V[b, :, j]
            s = 1.0 if q @ v >= 0 else -1.0
            assert np.max(np.abs(s * q - v)) <= 64 * n * H.eps_of(dt) * 10 / gap
            checked += 1
    assert checked > 500


@pytest.mark.parametrize("dt", DTYPES)
def test_zero_matrix_exact(dt):
    n = 9
    r = oracle.steqr(np.zeros((4, n), dt), np.zeros((4, n - 1), dt), jobz=True)
    assert np.all(r.lam == 0) and np.all(r.info == 0)
    assert np.array_equal(r.Q, np.broadcast_to(np.eye(n, dtype=dt), (4, n, n)))
    assert (r.sweeps, r.rotations, r.solves2x2) == (0, 0, 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_presplit_structure_exact(dt):
    n = 16
    d, e = inputs.normal_problems(n, 64, dt, seed=9)
    rng = np.random.default_rng(4)
    e[rng.random(e.shape) < 0.3] = 0
    e[:, 5] = 0
    e[:, 6] = 0                     # index 6 is an isolated 1x1 block
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    for b in range(64):
        block = np.zeros(n, dtype=int)
        for i in range(n - 1):
            block[i + 1] = block[i] + (1 if e[b, i] == 0 else 0)
        # every eigenvector lives on exactly one block
        for j in range(n):
            rows = np.nonzero(r.Q[b, :, j])[0]
            assert len(set(block[rows])) == 1
        # the isolated diagonal entry comes back bitwise
        assert d[b, 6] in r.lam[b]
        # the spectrum is the union of the block spectra
        ref = []
        for k in np.unique(block):
            idx = np.nonzero(block == k)[0]
            ref.extend(np.linalg.eigvalsh(H.dense(d[b, idx], e[b, idx[:-1]])[0]))
        tn = H.norm1(d[b], e[b])[0]
        assert np.max(np.abs(np.sort(ref) - r.lam[b])) <= H.lam_tol(n, dt, tn)


@pytest.mark.parametrize("dt", DTYPES)
def test_presplit_1x1_unscaled_in_scaled_matrix(dt):
    """Blocks open on exact zeros before any scaling, so an isolated diagonal
    entry of a matrix whose other block is scaled returns bitwise."""
    n = 12
    d, e = inputs.normal_problems(n, 32, np.float64, seed=13)
    fac = 1e-20 if dt == np.float32 else 1e-140
    d, e = (d * fac).astype(dt), (e * fac).astype(dt)
    e[:, 7] = 0
    e[:, 8] = 0
    r = oracle.steqr(d, e, jobz=True)
    for b in range(32):
        assert d[b, 8] in r.lam[b]
        j = int(np.nonzero(r.lam[b] == d[b, 8])[0][0])
        assert r.Q[b, 8, j] == 1 and np.count_nonzero(r.Q[b, :, j]) == 1


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [8, 16, 32])
def test_graded_direction_rate_and_relative_accuracy(dt, n):
    """perf_steqr, chase micro-structure decisions: QL/QR chosen as LAPACK
    does (small end first) converges a graded block's small end first; the
    inverted rule took about twice the steps and lost relative accuracy on
    graded input.  Pin both: about one step per eigenvalue, and small
    eigenvalues to relative accuracy, whichever end the grading starts at."""
    rng = np.random.default_rng(n)
    d = rng.standard_normal((200, n))
    e = rng.standard_normal((200, n - 1))
    g = 10.0 ** (-np.arange(n) / 2.0)
    d, e = (d * g).astype(dt), (e * g[: n - 1]).astype(dt)
    for dd, ee in ((d, e), (d[:, ::-1].copy(), e[:, ::-1].copy())):
        r = oracle.steqr(dd, ee, jobz=False)
        assert r.sweeps <= 1.5 * n * 200
        ref = np.linalg.eigvalsh(H.dense(dd, ee))
        rel = np.abs((r.lam.astype(np.float64) - ref) / ref).max(1)
        assert np.median(rel) <= 100 * H.eps_of(dt)


@pytest.mark.parametrize("dt", DTYPES)
def test_normal_input_convergence_rate(dt):
    """Cubically convergent shifted QL: well under 3 implicit steps per
    eigenvalue on N(0,1) input."""
    d, e = inputs.normal_problems(16, 400, dt, seed=1)
    r = oracle.steqr(d, e, jobz=False)
    assert r.sweeps <= 3 * 16 * 400


@pytest.mark.parametrize("dt", DTYPES)
def test_nonfinite_poisons_only_its_problem(dt):
    n = 6
    d, e = inputs.normal_problems(n, 5, dt, seed=1)
    d[1, 2] = np.nan
    e[2, 4] = np.inf
    d[3, 0] = -np.inf
    r = oracle.steqr(d, e, jobz=True)
    assert list(r.info) == [0, -1, -1, -1, 0]
    for b in (1, 2, 3):
        assert np.all(np.isnan(r.lam[b])) and np.all(np.isnan(r.Q[b]))
    ok = oracle.steqr(d[[0, 4]], e[[0, 4]], jobz=True)
    assert np.array_equal(ok.lam, r.lam[[0, 4]])
    assert np.array_equal(ok.Q, r.Q[[0, 4]])


@pytest.mark.parametrize("dt", DTYPES)
def test_zero_budget_fails_untouched(dt):
    n = 16
    d, e = inputs.normal_problems(n, 50, dt, seed=2)
    r = oracle.steqr(d, e, jobz=True, maxit_per_n=0)
    # no sweep may run: the first active block fails before any rotation,
    # every off-diagonal is still nonzero and nothing was sorted or rotated
    assert np.all(r.info == n - 1)
    assert np.array_equal(r.lam, d)
    assert np.array_equal(r.Q, np.broadcast_to(np.eye(n, dtype=dt), (50, n, n)))


@pytest.mark.parametrize("dt", DTYPES)
def test_small_budget_reports_unconverged(dt):
    n = 16
    d, e = inputs.normal_problems(n, 50, dt, seed=2)
    r = oracle.steqr(d, e, jobz=True, maxit_per_n=1)
    assert np.all((r.info > 0) & (r.info < n))
    # still a similarity: trace preserved
    tn = H.norm1(d, e).astype(np.float64)
    assert np.all(np.abs(r.lam.sum(1).astype(np.float64) - d.sum(1).astype(np.float64))
                  <= n * H.lam_tol(n, dt, tn))


@pytest.mark.parametrize("dt", DTYPES)
def test_reversed_problem_gives_identical_spectrum(dt):
    """QR on a block is QL on the mirrored block: reversing d and e must give
    the same eigenvalues bit for bit and row-reversed eigenvectors."""
    n = 15
    d, e = inputs.normal_problems(n, 200, dt, seed=8)
    keep = np.abs(d[:, 0]) != np.abs(d[:, -1])
    d, e = d[keep], e[keep]
    r1 = oracle.steqr(d, e, jobz=True)
    r2 = oracle.steqr(d[:, ::-1].copy(), e[:, ::-1].copy(), jobz=True)
    assert np.array_equal(r1.lam, r2.lam)
    assert np.array_equal(r1.Q, r2.Q[:, ::-1, :])
    # and both directions occur in this set
    assert 0 < np.count_nonzero(np.abs(d[:, 0]) > np.abs(d[:, -1])) < len(d)


@pytest.mark.parametrize("dt", DTYPES)
def test_power_of_two_scaling_is_exact(dt):
    n = 10
    d, e = inputs.normal_problems(n, 100, dt, seed=12)
    r1 = oracle.steqr(d, e, jobz=True)
    r2 = oracle.steqr(d * dt(4), e * dt(4), jobz=True)
    tn = H.norm1(d, e).astype(np.float64)
    assert np.all(np.abs(r2.lam - 4 * r1.lam).max(1) <= 4 * H.lam_tol(n, dt, tn))
    assert np.count_nonzero(np.all(r2.lam == 4 * r1.lam, axis=1)) >= 90


@pytest.mark.parametrize("dt", DTYPES)
def test_mixed_hard_cases(dt):
    n = 32
    d, e, labels, ab = inputs.mixed_problems(n, 600, dt, seed=0)
    r = oracle.steqr(d, e, jobz=True)
    assert np.all(r.info == 0)
    tn = H.norm1(d, e).astype(np.float64)
    ref = np.linalg.eigvalsh(H.dense(d, e))
    err = np.abs(r.lam.astype(np.float64) - ref).max(1)
    assert np.all(err <= H.lam_tol(n, dt, tn))
    res, orth = H.residual_orth(d, e, r.lam, r.Q)
    assert np.all(res <= 64 * n * H.eps_of(dt) * tn)
    assert np.all(orth <= 64 * n * H.eps_of(dt))
    z = labels == inputs.CLASS_INDEX["zero"]
    assert np.all(r.lam[z] == 0) and np.all(r.Q[z] == np.eye(n, dtype=dt))
    tp = np.nonzero(labels == inputs.CLASS_INDEX["toeplitz"])[0]
    for b in tp:
        cf = H.toeplitz_eigenvalues(n, d[b, 0], e[b, 0])
        assert np.max(np.abs(r.lam[b] - cf)) <= H.lam_tol(n, dt, tn[b])


def test_scaling_extremes_float32():
    """Blocks with norm above ssfmax or below ssfmin are scaled; results must
    track the float64 spectrum of the same rounded input."""
    n = 12
    d, e = inputs.normal_problems(n, 64, np.float64, seed=30)
    for fac in (3e19, 1e18, 1e-18, 1e-30, 1e-40):
        d32 = (d * fac).astype(np.float32)
        e32 = (e * fac).astype(np.float32)
        r = oracle.steqr(d32, e32, jobz=True)
        assert np.all(r.info == 0)
        ref = np.linalg.eigvalsh(H.dense(d32, e32))
        tn = H.norm1(d32, e32).astype(np.float64)
        err = np.abs(r.lam.astype(np.float64) - ref).max(1)
        assert np.all(err <= H.lam_tol(n, np.float32, tn)), (fac, (err / tn).max())
        res, orth = H.residual_orth(d32, e32, r.lam, r.Q)
        assert np.all(orth <= 64 * n * H.eps_of(np.float32))


def test_float32_oracle_close_to_float64_oracle():
    n = 16
    d, e = inputs.normal_problems(n, 300, np.float32, seed=0)
    r32 = oracle.steqr(d, e, jobz=False)
    r64 = oracle.steqr(d.astype(np.float64), e.astype(np.float64), jobz=False)
    tn = H.norm1(d, e).astype(np.float64)
    assert np.all(np.abs(r32.lam - r64.lam).max(1) <= H.lam_tol(n, np.float32, tn))


def test_counters_are_consistent():
    d, e = inputs.normal_problems(16, 100, np.float64, seed=0)
    r = oracle.steqr(d, e, jobz=False)
    # each sweep has at least 2 rotations (sweeps of length 1 are 2x2 solves)
    assert r.rotations >= 2 * r.sweeps
    # every eigenvalue is found by deflation or by a 2x2 solve
    assert r.solves2x2 <= 8 * 100
    assert r.sweeps <= 30 * 16 * 100


def test_multithreaded_batch_matches_single_thread():
    d, e = inputs.normal_problems(12, 500, np.float64, seed=44)
    a = oracle.steqr(d, e, jobz=True, nthreads=1)
    b = oracle.steqr(d, e, jobz=True, nthreads=4)
    assert np.array_equal(a.lam, b.lam) and np.array_equal(a.Q, b.Q)
    assert (a.sweeps, a.rotations, a.solves2x2) == (b.sweeps, b.rotations, b.solves2x2)


# --- back_transform (BatchLAS page "algo_steqr", eigenvector accumulation:
# with back_transform the rotations are right-applied to the caller's basis
# instead of the identity) ---

@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_back_transform_identity_basis_is_bitwise_plain(dt):
    d, e = inputs.normal_problems(11, 50, dt, seed=31)
    a = oracle.steqr(d, e, jobz=True)
    b = oracle.steqr(d, e, jobz=True, Z=np.broadcast_to(np.eye(11, dtype=dt), (50, 11, 11)))
    np.testing.assert_array_equal(a.lam, b.lam)
    np.testing.assert_array_equal(a.Q, b.Q)
    np.testing.assert_array_equal(a.info, b.info)


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_back_transform_permutation_basis_permutes_rows_exactly(dt):
    """Z = P (a row permutation): Z Q has the rows of Q permuted, bit for bit,
    since each row of the basis is rotated on its own."""
    n, batch = 9, 40
    d, e = inputs.normal_problems(n, batch, dt, seed=32)
    rng = np.random.default_rng(5)
    perms = np.stack([rng.permutation(n) for _ in range(batch)])
    P = np.zeros((batch, n, n), dtype=dt)
    P[np.arange(batch)[:, None], np.arange(n)[None, :], perms] = 1
    a = oracle.steqr(d, e, jobz=True)
    b = oracle.steqr(d, e, jobz=True, Z=P)
    np.testing.assert_array_equal(b.lam, a.lam)
    np.testing.assert_array_equal(b.Q, np.take_along_axis(a.Q, perms[:, :, None], axis=1))


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("n", [2, 7, 16, 32])
def test_back_transform_solves_the_dense_problem(dt, n):
    """With an orthogonal Z, V = Z Q holds the eigenvectors of A = Z T Z^T:
    residual and orthogonality within the stated bounds, and V agrees with
    Z times the plain eigenvectors."""
    batch = 60
    d, e = inputs.normal_problems(n, batch, dt, seed=33 + n)
    Z = inputs.orthogonal_bases(n, batch, dt, seed=n)
    eps = H.eps_of(dt)
    tn = H.norm1(d, e).astype(np.float64)
    r = oracle.steqr(d, e, jobz=True, Z=Z)
    assert np.all(r.info == 0)
    res, orth = H.back_residual_orth(d, e, Z, r.lam, r.Q)
    assert np.all(res <= 64 * n * eps * tn)
    assert np.all(orth <= 64 * n * eps)
    plain = oracle.steqr(d, e, jobz=True)
    np.testing.assert_array_equal(r.lam, plain.lam)
    zq = Z.astype(np.float64) @ plain.Q.astype(np.float64)
    assert np.abs(zq - r.Q).max() <= 64 * n * eps


# --- PG update scheme (BatchLAS page "algo_steqr", update schemes: PG
# propagates (g, p, c, s) across the sweep; EXP writes each local similarity;
# both perform the same implicit step) ---

@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("n", [2, 3, 6, 12, 17, 32])
def test_pg_scheme_solves_like_exp(dt, n):
    batch = 300
    d, e = inputs.normal_problems(n, batch, dt, seed=60 + n)
    eps = H.eps_of(dt)
    tn = H.norm1(d, e).astype(np.float64)
    pg = oracle.steqr(d, e, jobz=True, scheme="pg")
    ex = oracle.steqr(d, e, jobz=True, scheme="exp")
    assert np.all(pg.info == 0)
    ref = np.linalg.eigvalsh(H.dense(d, e))
    assert np.all(np.abs(pg.lam.astype(np.float64) - ref).max(1) <= H.lam_tol(n, dt, tn))
    res, orth = H.residual_orth(d, e, pg.lam, pg.Q)
    assert np.all(res <= 64 * n * eps * tn)
    assert np.all(orth <= 64 * n * eps)
    # the same implicit steps: sweep and rotation counts within 2 %
    assert abs(pg.sweeps - ex.sweeps) <= 0.02 * ex.sweeps + 2
    assert abs(pg.rotations - ex.rotations) <= 0.02 * ex.rotations + 2


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_pg_scheme_toeplitz_and_hard_cases(dt):
    n = 16
    rng = np.random.default_rng(7)
    a, b = rng.standard_normal(2)
    d = np.full((1, n), a, dtype=dt)
    e = np.full((1, n - 1), b, dtype=dt)
    r = oracle.steqr(d, e, jobz=False, scheme="pg")
    k = np.arange(1, n + 1)
    closed = np.sort(a + 2 * b * np.cos(k * np.pi / (n + 1)))
    tn = H.norm1(d, e).astype(np.float64)
    assert np.abs(r.lam[0].astype(np.float64) - closed).max() <= H.lam_tol(n, dt, tn)[0]
    dm, em, _, _ = inputs.mixed_problems(32, 400, dt, seed=3)
    pg = oracle.steqr(dm, em, jobz=False, scheme="pg")
    ex = oracle.steqr(dm, em, jobz=False, scheme="exp")
    np.testing.assert_array_equal(pg.info, ex.info)
    tn = H.norm1(dm, em).astype(np.float64)
    ok = np.isfinite(ex.lam).all(1)
    assert np.all(np.abs(pg.lam[ok].astype(np.float64) - ex.lam[ok]).max(1) <= 2 * H.lam_tol(32, dt, tn[ok]))


# --- fused small-n syev (BatchLAS page "perf_steqr": the fused kernel runs
# the reduction to tridiagonal form, the steqr solve and the back-transform;
# the reduction is the plain Householder one) ---

def _dense_checks(A, r, dt):
    n = A.shape[1]
    eps = H.eps_of(dt)
    Ad = np.asarray(A, dtype=np.longdouble)
    an = np.abs(Ad).sum(1).max(1).astype(np.float64)
    ref = np.linalg.eigvalsh(A.astype(np.float64))
    assert np.all(np.abs(r.lam.astype(np.float64) - ref).max(1) <= 16 * n * eps * an)
    if r.Q is not None:
        V = np.asarray(r.Q, dtype=np.longdouble)
        R = Ad @ V - V * np.asarray(r.lam, dtype=np.longdouble)[:, None, :]
        O = np.swapaxes(V, 1, 2) @ V - np.eye(n, dtype=np.longdouble)
        assert np.all(np.abs(R).reshape(len(A), -1).max(1).astype(np.float64) <= 64 * n * eps * an)
        assert np.abs(O).max() <= 64 * n * eps


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 2, 5, 12, 16, 31, 64])
def test_syev_against_library_and_residual(dt, n):
    A = inputs.dense_symmetric(n, 120, dt, seed=90 + n)
    r = oracle.syev(A, jobz=True)
    assert np.all(r.info == 0)
    _dense_checks(A, r, dt)
    rn = oracle.syev(A, jobz=False)
    np.testing.assert_array_equal(rn.lam, r.lam)


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_syev_of_a_tridiagonal_matrix_is_steqr_bitwise(dt):
    """A reflector has nothing to annihilate below the subdiagonal, so the
    reduction returns d and e untouched and Q = I."""
    n = 13
    d, e = inputs.normal_problems(n, 80, dt, seed=91)
    A = H.dense(d, e, dtype=dt)
    a = oracle.syev(A, jobz=True)
    b = oracle.steqr(d, e, jobz=True)
    np.testing.assert_array_equal(a.lam, b.lam)
    np.testing.assert_array_equal(a.Q, b.Q)
    np.testing.assert_array_equal(a.info, b.info)


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_syev_degenerate_inputs(dt):
    n = 9
    rng = np.random.default_rng(4)
    diag = rng.standard_normal((10, n)).astype(dt)
    A = np.zeros((10, n, n), dtype=dt)
    A[:, np.arange(n), np.arange(n)] = diag
    r = oracle.syev(A, jobz=True)
    np.testing.assert_array_equal(r.lam, np.sort(diag, axis=1))
    assert np.all(np.isin(r.Q, (-1, 0, 1)))
    z = oracle.syev(np.zeros((3, n, n), dtype=dt), jobz=True)
    assert np.all(z.lam == 0) and np.all(z.Q == np.eye(n, dtype=dt))
    # only the lower triangle is read: NaN above it changes nothing, below it
    # poisons the problem
    A = inputs.dense_symmetric(n, 4, dt, seed=5)
    ref = oracle.syev(A, jobz=True)
    Au = A.copy()
    Au[0, 1, 5] = np.nan
    up = oracle.syev(Au, jobz=True)
    np.testing.assert_array_equal(up.lam, ref.lam)
    Al = A.copy()
    Al[1, 5, 1] = np.nan
    lo = oracle.syev(Al, jobz=True)
    assert lo.info[1] == -1 and np.all(np.isnan(lo.lam[1])) and np.all(np.isnan(lo.Q[1]))
    np.testing.assert_array_equal(lo.lam[0], ref.lam[0])
