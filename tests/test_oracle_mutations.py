"""The oracle's pins must be able to fail.  Each case below plants one
plausible mistake (a wrong sign, a dropped term, a wrong index, an inverted
choice) in a private copy of the oracle's C source, builds it with gcc, and
requires the compact pin suite ``pin_failures`` to report at least one
failure; the unmodified source must report none.  CPU only."""
import os
import shutil

import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))
IMPL = "steqr_oracle_impl.h"
CONSTS = "steqr_oracle.c"

# (name, exact source text, replacement) in the generic body; entries of
# four are (name, file, exact source text, replacement)
MUTATIONS = [
    ("exp_sign_2csb", "DD(i0) = c * c * aa + (real_t)2 * c * s * bb + s * s * cc;",
     "DD(i0) = c * c * aa - (real_t)2 * c * s * bb + s * s * cc;"),
    ("exp_dropped_s2", "EE(i1) = c * s * (cc - aa) + (c * c - s * s) * bb;",
     "EE(i1) = c * s * (cc - aa) + (c * c) * bb;"),
    ("exp_transposed_operands", "DD(i1) = s * s * aa - (real_t)2 * c * s * bb + c * c * cc;",
     "DD(i1) = s * s * cc - (real_t)2 * c * s * bb + c * c * aa;"),
    ("bulge_sign", "gg = s * eo;", "gg = -s * eo;"),
    ("bulge_not_damped", "EE(i1 - 1) = c * eo;", "EE(i1 - 1) = eo;"),
    ("seed_wrong_index", "real_t gg = EE(m - 1);", "real_t gg = EE(lo);"),
    ("shift_far_root", "real_t mu = d1 - e1 / (g + R_COPYSIGN(r, g));",
     "real_t mu = d1 - e1 / (g - R_COPYSIGN(r, g));"),
    ("deflation_eps_not_squared", "if (tst <= (eps2 * R_ABS(DD(m))) * R_ABS(DD(m + 1)) + R_SAFMIN)",
     "if (tst <= (R_EPS * R_ABS(DD(m))) * R_ABS(DD(m + 1)) + R_SAFMIN)"),
    ("direction_inverted", "if (R_ABS(d[lb]) <= R_ABS(d[le])) {",
     "if (R_ABS(d[lb]) > R_ABS(d[le])) {"),
    ("qrot_sign", "qb[i] = -s * x + c * y;", "qb[i] = s * x + c * y;"),
    ("two_by_two_sign", "DD(lo) = a - t * b;", "DD(lo) = a + t * b;"),
    ("unscale_wrong_factor", "real_t us = a_eff / R_SSFMIN;", "real_t us = R_SSFMIN / a_eff;"),
    ("sort_unstable_descending", "while (j >= 0 && val[j] > x) {", "while (j >= 0 && val[j] < x) {"),
    ("budget_off_by_all", "if (jtot == budget) {", "if (jtot == budget + 1000000) {"),
    ("block_ignores_exact_zero", "while (le < n - 1 && e[le] != (real_t)0)",
     "while (le < n - 1 && e[le] != (real_t)-12345)"),
    ("back_transform_ignored", "    if (jobz == 1)\n", "    if (jobz >= 1)\n"),
    ("pg_dropped_2cb", "real_t rs = (DD(i1) - gs) * sp + (real_t)2 * cp * b;",
     "real_t rs = (DD(i1) - gs) * sp + cp * b;"),
    ("pg_missing_fixup", "DD(lo) = DD(lo) - p;", "DD(lo) = DD(lo);"),
    ("pg_bulge_unscaled", "real_t f = sp * EE(i1), b = cp * EE(i1), rr;",
     "real_t f = EE(i1), b = cp * EE(i1), rr;"),
    ("sytd2_rank1_only", "A[r + (size_t)c * n] -= v[r] * p[c] + p[r] * v[c];",
     "A[r + (size_t)c * n] -= v[r] * p[c];"),
    ("sytd2_beta_sign", "real_t beta = -R_COPYSIGN(FN(hypot2)(alpha, xnorm), alpha);",
     "real_t beta = R_COPYSIGN(FN(hypot2)(alpha, xnorm), alpha);"),
    ("sytd2_q_forward_order", "for (int i = n - 2; i >= 0; --i) {\n            if (tau[i] == (real_t)0)",
     "for (int i = 0; i <= n - 2; ++i) {\n            if (tau[i] == (real_t)0)"),
    # scaling (algo_steqr, the scaling paragraph): thresholds, the exact
    # lift of a subnormal norm, and the scale-back
    ("f64_ssfmax_never_scales", CONSTS, "#define R_SSFMAX (0x1p511 / 3.0)", "#define R_SSFMAX (0x1p1023)"),
    ("f64_ssfmin_never_scales", CONSTS, "#define R_SSFMIN 0x1p-405", "#define R_SSFMIN 0x1p-1020"),
    ("f32_ssfmax_never_scales", CONSTS, "#define R_SSFMAX (0x1p63f / 3.0f)", "#define R_SSFMAX (0x1p127f)"),
    ("f32_prescale_dropped", CONSTS, "#define R_PRESCALE_F32 16777216.0f", "#define R_PRESCALE_F32 1.0f"),
    ("prescale_not_undone", "real_t upre = (real_t)1 / pre;", "real_t upre = (real_t)1;"),
    ("prescale_skips_e", "e[i] = (e[i] * pre) * sc;", "e[i] = e[i] * sc;"),
    ("unscale_down_inverted", "real_t us = anorm / R_SSFMAX;", "real_t us = R_SSFMAX / anorm;"),
]


def pin_failures(lib):
    """Compact pin suite; returns the names of failed pins."""
    bad = []

    def check(name, ok):
        if not ok:
            bad.append(name)

    for dt in (np.float32, np.float64):
        eps = H.eps_of(dt)
        # library eigensolver + residual + orthogonality, several n
        for n in (3, 8, 13):
            d, e = inputs.normal_problems(n, 40, dt, seed=n)
            r = oracle.steqr(d, e, jobz=True, lib=lib)
            tn = H.norm1(d, e).astype(np.float64)
            ref = np.linalg.eigvalsh(H.dense(d, e))
            check(f"info{n}", np.all(r.info == 0))
            lam = np.nan_to_num(r.lam.astype(np.float64), nan=1e300)
            check(f"eigvalsh{n}", np.all(np.abs(lam - ref).max(1) <= H.lam_tol(n, dt, tn)))
            if np.all(np.isfinite(r.Q)):
                res, orth = H.residual_orth(d, e, r.lam, r.Q)
                check(f"res{n}", np.all(res <= 64 * n * eps * tn))
                check(f"orth{n}", np.all(orth <= 64 * n * eps))
            else:
                bad.append(f"finite{n}")
            check(f"ascending{n}", np.all(np.diff(r.lam, axis=1) >= 0))
        # convergence rate: cubically convergent shifted QL needs well under
        # 3 implicit steps per eigenvalue on N(0,1) input
        d, e = inputs.normal_problems(16, 100, dt, seed=1)
        r = oracle.steqr(d, e, jobz=False, lib=lib)
        check("rate", r.sweeps <= 3 * 16 * 100)
        # zero budget leaves everything untouched and reports n-1
        d, e = inputs.normal_problems(10, 20, dt, seed=2)
        r = oracle.steqr(d, e, jobz=True, maxit_per_n=0, lib=lib)
        check("budget", np.all(r.info == 9) and np.array_equal(r.lam, d))
        # scaled extremes
        d, e = inputs.normal_problems(8, 20, np.float64, seed=3)
        for fac in (1e-30, 1e30) if dt == np.float64 else (1e-20, 1e20):
            ds, es = (d * fac).astype(dt), (e * fac).astype(dt)
            r = oracle.steqr(ds, es, jobz=False, lib=lib)
            tn = H.norm1(ds, es).astype(np.float64)
            ref = np.linalg.eigvalsh(H.dense(ds, es))
            lam = np.nan_to_num(r.lam.astype(np.float64), nan=1e300)
            check(f"scaled{fac}", np.all(np.abs(lam - ref).max(1) <= H.lam_tol(8, dt, tn)))
        # scaled extremes: N(0,1) times 2^k across every scaling branch,
        # against 2^k times the library spectrum of the exactly rescaled
        # matrix
        d, e, k = inputs.scaled_problems(8, 4 * len(inputs.SCALE_EXPONENTS[np.dtype(dt)]), dt, seed=90)
        r = oracle.steqr(d, e, jobz=True, lib=lib)
        check("scaled_info", np.all(r.info == 0))
        dr = np.ldexp(d.astype(np.float64), -k[:, None])
        er = np.ldexp(e.astype(np.float64), -k[:, None])
        ref = np.ldexp(np.linalg.eigvalsh(H.dense(dr, er)).astype(np.longdouble), k[:, None])
        lam = np.nan_to_num(r.lam.astype(np.longdouble), nan=np.longdouble(1e300))
        check("scaled_lam", np.all(np.abs(lam - ref).max(1) <= H.lam_tol_sub(8, dt, H.norm1(d, e))))
        # pre-split: every eigenvector on one block
        d, e = inputs.normal_problems(9, 10, dt, seed=4)
        e[:, 3] = 0
        r = oracle.steqr(d, e, jobz=True, lib=lib)
        check("split", np.all(r.Q[:, :4, :] * r.Q[:, 4:, :].sum(1, keepdims=True) == 0)
              if np.all(np.isfinite(r.Q)) else False)
        # an isolated 1x1 block inside a matrix that needs scaling comes back
        # bitwise (it is never scaled)
        ds, es = (d * 1e-20).astype(dt), (e * 1e-20).astype(dt)
        es[:, 5] = 0
        es[:, 6] = 0
        r = oracle.steqr(ds, es, jobz=False, lib=lib)
        check("split1x1", all(ds[b, 6] in r.lam[b] for b in range(len(ds))))
        # graded input: QL/QR chosen so the small end converges first takes
        # about one step per eigenvalue and keeps small eigenvalues to high
        # relative accuracy (the inverted rule takes about twice the steps)
        d, e = graded(16, 100, dt)
        r = oracle.steqr(d, e, jobz=False, lib=lib)
        ref = np.linalg.eigvalsh(H.dense(d, e))
        rel = np.abs((r.lam.astype(np.float64) - ref) / ref).max(1)
        check("graded_rate", r.sweeps <= 1.5 * 16 * 100)
        check("graded_relacc", np.median(rel) <= 100 * eps)
        # PG update scheme: same spectrum and eigenpair bounds as EXP
        for n in (5, 12):
            d, e = inputs.normal_problems(n, 40, dt, seed=50 + n)
            r = oracle.steqr(d, e, jobz=True, lib=lib, scheme="pg")
            tn = H.norm1(d, e).astype(np.float64)
            ref = np.linalg.eigvalsh(H.dense(d, e))
            check(f"pg_info{n}", np.all(r.info == 0))
            lam = np.nan_to_num(r.lam.astype(np.float64), nan=1e300)
            check(f"pg_eigvalsh{n}", np.all(np.abs(lam - ref).max(1) <= H.lam_tol(n, dt, tn)))
            if np.all(np.isfinite(r.Q)):
                res, orth = H.residual_orth(d, e, r.lam, r.Q)
                check(f"pg_res{n}", np.all(res <= 64 * n * eps * tn))
            else:
                bad.append(f"pg_finite{n}")
        # fused syev: eigenpairs of a dense symmetric matrix
        for n in (6, 11):
            A = inputs.dense_symmetric(n, 30, dt, seed=70 + n)
            r = oracle.syev(A, jobz=True, lib=lib)
            an = np.abs(A.astype(np.float64)).sum(1).max(1)
            ref = np.linalg.eigvalsh(A.astype(np.float64))
            lam = np.nan_to_num(r.lam.astype(np.float64), nan=1e300)
            check(f"syev_lam{n}", np.all(np.abs(lam - ref).max(1) <= 16 * n * eps * an))
            if np.all(np.isfinite(r.Q)):
                V = r.Q.astype(np.float64)
                res = np.abs(A.astype(np.float64) @ V - V * r.lam[:, None, :]).reshape(30, -1).max(1)
                check(f"syev_res{n}", np.all(res <= 64 * n * eps * an))
            else:
                bad.append(f"syev_finite{n}")
        # back_transform: the rotations are right-applied to an orthogonal Z,
        # so Z Q holds the eigenvectors of Z T Z^T
        d, e = inputs.normal_problems(7, 20, dt, seed=6)
        Z = inputs.orthogonal_bases(7, 20, dt, seed=6)
        r = oracle.steqr(d, e, jobz=True, Z=Z, lib=lib)
        tn = H.norm1(d, e).astype(np.float64)
        if np.all(np.isfinite(r.Q)):
            res, orth = H.back_residual_orth(d, e, Z, r.lam, r.Q)
            check("back_res", np.all(res <= 64 * 7 * eps * tn))
        else:
            bad.append("back_finite")
    return bad


def graded(n, batch, dt, seed=0):
    """d_i, e_i = N(0,1) 10^(-i/2), largest entries at the top."""
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((batch, n))
    e = rng.standard_normal((batch, n - 1))
    g = 10.0 ** (-np.arange(n) / 2.0)
    return (d * g).astype(dt), (e * g[: n - 1]).astype(dt)


@pytest.fixture(scope="module")
def build_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


def _build_variant(build_dir, name, old, new, fname=IMPL):
    src = build_dir / name
    src.mkdir()
    for f in oracle._SOURCES:
        shutil.copy(os.path.join(ORACLE_DIR, f), src / f)
    if old is not None:
        text = (src / fname).read_text()
        assert text.count(old) == 1, f"mutation anchor not unique: {name}"
        (src / fname).write_text(text.replace(old, new))
    out = oracle.build(force=True, src_dir=str(src), out_path=str(src / "lib.so"))
    return oracle.load_variant(out)


def test_unmodified_oracle_passes_compact_pins(build_dir):
    lib = _build_variant(build_dir, "clean", None, None)
    assert pin_failures(lib) == []


def _spec(m):
    return (m[0], IMPL, m[1], m[2]) if len(m) == 3 else m


@pytest.mark.parametrize("name,fname,old,new", [_spec(m) for m in MUTATIONS], ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(build_dir, name, fname, old, new):
    lib = _build_variant(build_dir, name, old, new, fname)
    assert pin_failures(lib) != [], f"mutation {name} slipped through every pin"
