"""Unit layer under the parity tests: each building block of the solve, run
on a table of inputs through the library's diagnostic entry point
(bstq_diag), against exact or higher-precision arithmetic.

- The reciprocal, quotient, square-root and reciprocal-square-root
  refinements (Newton-Raphson / third-order Householder steps on the
  hardware approximations) against correctly rounded results, element by
  element: at most one unit in the last place, over normal numbers of every
  exponent, values next to the smallest normal and to the overflow bound,
  and powers of two.
- lartg, the copysign shift with the 2x2 tangent and rotation (BatchLAS page
  "algo_steqr": Givens rotation, shift, 2x2 solve) against long double.
- One pass of the bulge chase in both kernel families, EXP and PG (page
  "algo_steqr": implicit step, update schemes): the pass's rotations Q are
  orthogonal, the new tridiagonal is Q^T T Q (a dense explicit similarity in
  long double, so the bulge left the matrix), the first rotation is the one
  of the shifted seed (d_m - mu, e_{m-1}), and entries outside the active
  range are untouched, including under the identity positions of a lockstep
  pass.
- The factored double eigenvector update (fast Givens) over thousands of
  rotations per column, where the column scales would underflow without
  their guard, against the plain product in long double."""
import numpy as np
import pytest

from tests import helpers as H

pytestmark = pytest.mark.gpu

F32, F64 = np.float32, np.float64
LD = np.longdouble


def _diag(op, arr, count, arg=0):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    t = torch.from_numpy(np.ascontiguousarray(arr)).cuda()
    out = bstq.diag(op, t, count, arg)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _bstq():
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    return bstq


def _positive_inputs(dt, count, seed):
    """Normal positive numbers of every exponent, the ends of the normal
    range, and powers of two."""
    fi = np.finfo(dt)
    rng = np.random.default_rng(seed)
    lo, hi = np.log2(float(fi.smallest_normal)), np.log2(float(fi.max))
    x = np.exp2(rng.uniform(lo + 1, hi - 2, count)) * rng.uniform(1, 2, count)
    edge = np.array([float(fi.smallest_normal) * k for k in (1, 1.5, 2, 3)]
                    + [float(fi.max) / k for k in (2, 3, 4, 8)], dtype=np.float64)
    pw = np.exp2(np.arange(int(lo) + 2, int(hi) - 2, 7, dtype=np.float64))
    return np.concatenate([x, edge, pw]).astype(dt)


def _ulps(got, ref, dt):
    ref = np.asarray(ref, dtype=dt)
    return np.abs(got.astype(LD) - ref.astype(LD)) / np.spacing(np.abs(ref)).astype(LD)


@pytest.mark.parametrize("dt", [F32, F64])
def test_reciprocal_square_root_and_quotient_refinements(dt):
    b = _bstq()
    x = _positive_inputs(dt, 20000, 1)
    xl = x.astype(LD)
    # correctly rounded references: numpy's own division and square root in
    # the dtype (IEEE), and 1/sqrt through long double
    ref_rcp = (dt(1) / x)
    ref_sqrt = np.sqrt(x)
    ref_rsqrt = (LD(1) / np.sqrt(xl)).astype(dt)
    # x below the overflow bound's reciprocal range keeps 1/x normal
    ok = x < dt(np.finfo(dt).max) / dt(4)
    ok &= x > dt(4) / dt(np.finfo(dt).max)
    got = _diag(b.DIAG_RCP, x, len(x))[:, 0]
    assert np.all(_ulps(got[ok], ref_rcp[ok], dt) <= 1), "rcp"
    got = _diag(b.DIAG_SQRT, x, len(x))[:, 0]
    assert np.all(_ulps(got, ref_sqrt, dt) <= 1), "sqrt"
    got = _diag(b.DIAG_RSQRT, x, len(x))[:, 0]
    assert np.all(_ulps(got, ref_rsqrt, dt) <= 1), "rsqrt"
    # a / b with a normal quotient
    rng = np.random.default_rng(2)
    a = (rng.standard_normal(len(x)) * np.exp2(rng.uniform(-40, 40, len(x)))).astype(dt)
    den = (np.sign(rng.standard_normal(len(x))) * np.exp2(rng.uniform(-40, 40, len(x)))
           * rng.uniform(1, 2, len(x))).astype(dt)
    got = _diag(b.DIAG_DIV, np.stack([a, den], 1), len(x))[:, 0]
    ref = a / den
    assert np.all(_ulps(got, ref, dt) <= 1), "div"
    # sqrt(1 + x^2) for |x| across the range the shift uses
    h = (rng.standard_normal(4000) * np.exp2(rng.uniform(-30, 30, 4000))).astype(dt)
    got = _diag(b.DIAG_HYP1, h, len(h))[:, 0]
    ref = np.sqrt(LD(1) + h.astype(LD) ** 2).astype(dt)
    assert np.all(_ulps(got, ref, dt) <= 2), "hyp1"


@pytest.mark.parametrize("op,dt", [("lartg", F32), ("lartg", F64), ("lartg_fast", F64)])
def test_lartg(op, dt):
    b = _bstq()
    code = b.DIAG_LARTG if op == "lartg" else b.DIAG_LARTG_FAST
    rng = np.random.default_rng(3)
    m = 6000
    span = 60 if dt == F32 else 400
    f = rng.standard_normal(m) * np.exp2(rng.uniform(-span, span, m))
    g = rng.standard_normal(m) * np.exp2(rng.uniform(-span, span, m))
    f[:200] = 0.0
    g[200:400] = 0.0
    g[400:600] = f[400:600] * 1e-30     # negligible bulge
    f, g = f.astype(dt), g.astype(dt)
    out = _diag(code, np.stack([f, g], 1), m)
    c, s, r = out[:, 0], out[:, 1], out[:, 2]
    z = g == 0
    # g = 0: (1, 0, f) exactly (page perf_steqr: identity rotations)
    assert np.all(c[z] == 1) and np.all(s[z] == 0) and np.array_equal(r[z], f[z])
    fl, gl = f.astype(LD), g.astype(LD)
    rr = np.sqrt(fl * fl + gl * gl)
    eps = H.eps_of(dt)
    nz = ~z
    assert np.all(r[nz] >= 0)
    # a few roundings each (the scaled squares, the refined 1/sqrt, the
    # products): within 3 ulps (6 eps) of the long-double values
    er = float((np.abs(r[nz].astype(LD) - rr[nz]) / rr[nz]).max() / eps)
    ec = float(np.abs(c[nz].astype(LD) - fl[nz] / rr[nz]).max() / eps)
    es = float(np.abs(s[nz].astype(LD) - gl[nz] / rr[nz]).max() / eps)
    assert er <= 6 and ec <= 6 and es <= 6, (er, ec, es)
    # G^T [f; g] = [r; 0]
    cl, sl = c.astype(LD), s.astype(LD)
    ea = float((np.abs(-sl[nz] * fl[nz] + cl[nz] * gl[nz]) / rr[nz]).max() / eps)
    assert ea <= 8, ea


@pytest.mark.parametrize("dt", [F32, F64])
def test_shift_and_two_by_two_rotation(dt):
    b = _bstq()
    rng = np.random.default_rng(4)
    m = 8000
    d1 = rng.standard_normal(m)
    d2 = rng.standard_normal(m)
    e1 = rng.standard_normal(m) * np.exp2(rng.uniform(-12, 4, m))
    d2[:300] = d1[:300]                  # delta = 0: the tie goes to sgn(e1)
    d1, d2, e1 = d1.astype(dt), d2.astype(dt), e1.astype(dt)
    out = _diag(b.DIAG_SHIFT, np.stack([d1, d2, e1], 1), m)
    t, mu, cs, sn = (out[:, k].astype(LD) for k in range(4))
    a, c, e = d1.astype(LD), d2.astype(LD), e1.astype(LD)
    tau = (c - a) / (2 * e)
    sg = np.where(tau > 0, 1, np.where(tau < 0, -1, np.sign(e)))
    tr = sg / (np.abs(tau) + np.sqrt(tau * tau + 1))
    eps = H.eps_of(dt)
    nrm = np.maximum(np.abs(a), np.abs(c)) + np.abs(e)
    assert np.all(np.abs(t - tr) <= 8 * eps * np.maximum(np.abs(tr), 1e-300) + 2 * eps * np.abs(e) / nrm)
    # mu: the eigenvalue of the 2x2 nearer to d1 (the copysign shift)
    half = (c - a) / 2
    root = np.sqrt(half * half + e * e)
    lam_a, lam_b = (a + c) / 2 - root, (a + c) / 2 + root
    near = np.where(np.abs(lam_a - a) <= np.abs(lam_b - a), lam_a, lam_b)
    assert np.all(np.abs(mu - near) <= 4 * eps * nrm)
    # (cs, sn) = (1, t) / sqrt(1 + t^2) diagonalises the 2x2: with the chase's
    # column convention on the pair (k+1, k), the rotated off-diagonal vanishes
    assert np.all(np.abs(cs * cs + sn * sn - 1) <= 4 * eps)
    off = cs * sn * (a - c) + (cs * cs - sn * sn) * e
    assert np.all(np.abs(off) <= 8 * eps * nrm)


def _pass_records(dt, count, seed, task):
    """Random passes on tridiagonals of n <= 16: the active range [lo, m]
    closed by zeros at e_{lo-1} and e_m, the copysign shift of the leading
    2x2 at lo, and a union of positions around [lo+1, m]."""
    rng = np.random.default_rng(seed)
    rec = np.zeros((count, 42), dtype=np.float64)
    for k in range(count):
        n = int(rng.integers(3, 17))
        d = np.zeros(16)
        e = np.zeros(16)
        d[:n] = rng.standard_normal(n)
        e[: n - 1] = rng.standard_normal(n - 1)
        if task == 2:
            lo = int(rng.integers(0, n - 1))
            m = lo + 1
        else:
            lo = int(rng.integers(0, n - 2))
            m = int(rng.integers(lo + 2, n))
        if lo > 0:
            e[lo - 1] = 0.0
        if m < n - 1:
            e[m] = 0.0
        d, e = d.astype(dt).astype(np.float64), e.astype(dt).astype(np.float64)
        a, c, b = LD(d[lo]), LD(d[lo + 1]), LD(e[lo])
        tau = (c - a) / (2 * b)
        sg = 1 if tau > 0 else (-1 if tau < 0 else np.sign(b))
        t = sg / (abs(tau) + np.sqrt(tau * tau + 1))
        mu = a - b * t
        cs2 = 1 / np.sqrt(1 + t * t)
        sn2 = t * cs2
        rhi = int(rng.integers(m, 16))
        rlo = int(rng.integers(1, lo + 2))
        f0 = dt(LD(d[m]) - mu) if task == 1 else 0.0
        g0 = e[m - 1] if task == 1 else 0.0
        rec[k, :10] = [n, lo, m, task, rhi, rlo, f0, g0, dt(cs2), dt(sn2)]
        rec[k, 10:26] = d
        rec[k, 26:42] = e
    return rec.astype(dt)


def _check_pass(rec, out, dt, what):
    eps = H.eps_of(dt)
    for k in range(len(rec)):
        n, lo, m, task = (int(v) for v in rec[k, :4])
        d0, e0 = rec[k, 10:26].astype(LD), rec[k, 26:42].astype(LD)
        d1, e1 = out[k, :16], out[k, 16:32]
        Q = out[k, 32:].reshape(16, 16).T.astype(LD)     # column-major
        tn = float(H.norm1(d0[None, :n], e0[None, : n - 1])[0])
        # orthogonal, and the identity outside the active range
        assert np.abs(Q.T @ Q - np.eye(16)).max() <= 16 * 16 * eps, (what, k)
        act = np.zeros(16, bool)
        act[lo:m + 1] = True
        assert np.all(Q[~act][:, ~act] == np.eye(16)[~act][:, ~act]), (what, k)
        # untouched entries outside [lo, m], as values (identity rotations of
        # a lockstep pass keep them)
        assert np.all(d1[~act] == d0[~act].astype(dt)), (what, k)
        eo = np.ones(16, bool)
        eo[lo:m] = False
        assert np.all(e1[eo] == e0[eo].astype(dt)), (what, k)
        # the new tridiagonal is the dense similarity Q^T T Q (long double):
        # its band matches, and nothing is left outside the band (the bulge
        # was chased out)
        T0 = H.dense(d0[None], e0[None, :15], LD)[0]
        S = Q.T @ T0 @ Q
        tol = 64 * 16 * eps * max(tn, 1e-30)
        assert np.abs(np.diag(S) - d1.astype(LD)).max() <= tol, (what, k)
        assert np.abs(np.diag(S, 1) - e1[:15].astype(LD)).max() <= tol, (what, k)
        band = np.abs(np.subtract.outer(np.arange(16), np.arange(16))) <= 1
        assert np.abs(S[~band]).max(initial=0) <= tol, (what, k)
        if task == 1:
            # the first rotation is that of the seed: column m of Q is
            # c e_m + s e_{m-1}, (c, s) = (f0, g0) / r with r >= 0
            f0, g0 = LD(rec[k, 6]), LD(rec[k, 7])
            r = np.hypot(f0, g0)
            assert abs(Q[m, m] - f0 / r) <= 4 * eps and abs(Q[m - 1, m] - g0 / r) <= 4 * eps, (what, k)
        else:
            assert e1[lo] == 0, (what, k)


@pytest.mark.parametrize("family", ["static", "dyn_exp", "dyn_pg"])
@pytest.mark.parametrize("task", [1, 2])
@pytest.mark.parametrize("dt", [F32, F64])
def test_one_pass_of_the_chase(dt, task, family):
    b = _bstq()
    op = {"static": b.DIAG_PASS_STATIC, "dyn_exp": b.DIAG_PASS_DYN_EXP, "dyn_pg": b.DIAG_PASS_DYN_PG}[family]
    rec = _pass_records(dt, 400, 10 + task, task)
    out = _diag(op, rec, len(rec))
    _check_pass(rec, out, dt, f"{family} task={task}")


@pytest.mark.parametrize("dt", [F32, F64])
def test_lockstep_identity_positions_change_nothing(dt):
    """A pass entered above the lane's sweep and run below it (the union of
    a warp's positions) gives the same values as the lane's own range."""
    b = _bstq()
    rec = _pass_records(dt, 300, 20, 1)
    own = rec.copy()
    own[:, 4] = own[:, 2]          # rhi = m
    own[:, 5] = own[:, 1] + 1      # rlo = lo + 1
    a = _diag(b.DIAG_PASS_STATIC, rec, len(rec))
    c = _diag(b.DIAG_PASS_STATIC, own, len(own))
    assert np.all(a == c)


@pytest.mark.parametrize("angle", ["near_45", "random"])
def test_factored_update_over_thousands_of_rotations(angle):
    """K = 2000 sweeps over a 16 x 16 Q: 4,000 rotations per column.  Near
    45 degrees every rotation halves a column's scale squared, so without the
    guard the scales would reach 2^-2000; the result must still be the plain
    product of the rotations (long double) to accumulated rounding."""
    b = _bstq()
    K, count = 2000, 16
    rng = np.random.default_rng(30)
    if angle == "near_45":
        th = np.pi / 4 + rng.uniform(-0.05, 0.05, (count, K, 15))
    else:
        th = rng.uniform(-np.pi, np.pi, (count, K, 15))
    c, s = np.cos(th), np.sin(th)
    rot = np.stack([c, s], -1)
    out = _diag(b.DIAG_FASTQ, rot, count, arg=K)
    Qg = out.reshape(count, 16, 16).transpose(0, 2, 1)   # column-major
    assert np.all(np.isfinite(Qg))
    Q = np.broadcast_to(np.eye(16, dtype=LD), (count, 16, 16)).copy()
    cl, sl = c.astype(LD), s.astype(LD)
    for k in range(K):
        for j in range(15):
            C = 15 - j
            x, y = Q[:, :, C].copy(), Q[:, :, C - 1].copy()
            cc, ss = cl[:, k, j, None], sl[:, k, j, None]
            Q[:, :, C] = cc * x + ss * y
            Q[:, :, C - 1] = -ss * x + cc * y
    err = np.abs(Qg.astype(LD) - Q).max()
    assert err <= 1e-10, float(err)
    orth = np.abs(np.swapaxes(Qg, 1, 2) @ Qg - np.eye(16)).max()
    assert orth <= 1e-10, orth
