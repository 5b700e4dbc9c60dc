/*
 * Generic body of the CPU oracle: implicit shifted QL/QR with a Givens bulge
 * chase for one symmetric tridiagonal problem.  TEST INFRASTRUCTURE ONLY.
 *
 * Included twice by steqr_oracle.c, once with real_t = float and once with
 * real_t = double; the including file defines real_t, FN(name), R_ABS,
 * R_SQRT, R_COPYSIGN and the constants R_EPS, R_SAFMIN, R_SSFMAX, R_SSFMIN,
 * R_PRESCALE.
 *
 * Every step follows the BatchLAS documentation page "algo_steqr" (the
 * mathematics of steqr) and the BatchLAS page "perf_steqr" (performance notes
 * of steqr_cta), cited per function.  The code is written to be read against
 * those pages: no blocking, fusion or reordering beyond what they describe.
 * Arithmetic runs in real_t, compiled with -ffp-contract=off (no FMA).
 */

/* sqrt(1 + x^2) without overflow for large |x|.
 * Used by the copysign shift (algo_steqr, shift equation r = sqrt(g^2 + 1))
 * and by the 2x2 direct solve. */
static real_t FN(hyp1)(real_t x)
{
    real_t ax = R_ABS(x);
    if (ax <= (real_t)1)
        return R_SQRT((real_t)1 + ax * ax);
    real_t y = (real_t)1 / ax;
    return ax * R_SQRT((real_t)1 + y * y);
}

/* sqrt(f^2 + g^2) by the max-scaled formula w * sqrt(1 + (z/w)^2). */
static real_t FN(hypot2)(real_t f, real_t g)
{
    real_t af = R_ABS(f), ag = R_ABS(g);
    real_t w = af > ag ? af : ag;
    real_t z = af > ag ? ag : af;
    if (w == (real_t)0)
        return (real_t)0;
    real_t q = z / w;
    return w * R_SQRT((real_t)1 + q * q);
}

/* lartg: plane rotation G(c,s) = [[c,-s],[s,c]] with G^T [f; g] = [r; 0].
 * algo_steqr, Givens rotation definition; perf_steqr, "CTA STEQR: chase
 * micro-structure decisions" (g = 0 returns (1, 0, f)).
 * Otherwise r = hypot(f, g) >= 0, c = f / r, s = g / r. */
static void FN(lartg)(real_t f, real_t g, real_t *c, real_t *s, real_t *r)
{
    if (g == (real_t)0) {
        *c = (real_t)1;
        *s = (real_t)0;
        *r = f;
        return;
    }
    real_t h = FN(hypot2)(f, g);
    *c = f / h;
    *s = g / h;
    *r = h;
}

/* Right-apply the plane rotation G = [[c,-s],[s,c]] acting on the column pair
 * (ja, jb) of the n x n column-major Q:  Q[:, {ja, jb}] <- Q[:, {ja, jb}] G.
 * algo_steqr, eigenvector accumulation paragraph. */
static void FN(rot_cols)(int n, real_t *Q, int ja, int jb, real_t c, real_t s)
{
    real_t *qa = Q + (size_t)ja * n;
    real_t *qb = Q + (size_t)jb * n;
    for (int i = 0; i < n; ++i) {
        real_t x = qa[i], y = qb[i];
        qa[i] = c * x + s * y;
        qb[i] = -s * x + c * y;
    }
}

/* Block-local view in "converging" coordinates: local index p = 0 is the end
 * of the active block that converges first; p grows toward the other end.
 * For QL the converging end is the top of the block (dir = +1), for QR it is
 * the bottom (dir = -1), as perf_steqr "CTA STEQR: chase micro-structure
 * decisions" (QL if |D_l| <= |D_lend|) and algo_steqr (QL runs the QR
 * formulas on reversed local indices) describe. */
typedef struct {
    int lconv; /* physical index of local p = 0 */
    int dir;   /* +1 or -1 */
} FN(view_t);

static int FN(pidx)(FN(view_t) v, int p) { return v.lconv + v.dir * p; }
/* physical index of the off-diagonal coupling local p and p + 1 */
static int FN(eidx)(FN(view_t) v, int p)
{
    return v.dir > 0 ? v.lconv + p : v.lconv - p - 1;
}

/*
 * Solve one problem.  d[n] is overwritten with the eigenvalues; e_in[n-1] is
 * read only; ework[n] is scratch; Q[n*n] (column-major, used iff jobz != 0)
 * receives the eigenvectors (jobz == 1), or holds a basis Z on entry and
 * receives Z times the eigenvectors (jobz == 2, back_transform).
 * cnt[0..2] accumulate (implicit steps,
 * rotations, 2x2 direct solves).  Returns info: 0 converged, k > 0 the sweep
 * budget ran out with k off-diagonals still nonzero, -1 non-finite input.
 */
static int FN(steqr_one)(int n, int jobz, int maxit_per_n, int sort, int scheme,
                         real_t *d, const real_t *e_in, real_t *Q,
                         real_t *e, long *cnt)
{
    const real_t eps2 = R_EPS * R_EPS;
    int i;

    /* Non-finite input poisons the problem (reading of the pages: they only
     * state that NaN items are part of the checked set). */
    int bad = 0;
    for (i = 0; i < n; ++i)
        if (!isfinite(d[i]))
            bad = 1;
    for (i = 0; i + 1 < n; ++i)
        if (!isfinite(e_in[i]))
            bad = 1;
    if (bad) {
        for (i = 0; i < n; ++i)
            d[i] = (real_t)NAN;
        if (jobz)
            for (i = 0; i < n * n; ++i)
                Q[i] = (real_t)NAN;
        return -1;
    }

    for (i = 0; i + 1 < n; ++i)
        e[i] = e_in[i];
    /* algo_steqr, eigenvector accumulation: back_transform = false starts
     * from Q = I (jobz == 1); back_transform = true (jobz == 2) takes the
     * caller's Q as the basis the rotations are right-applied to. */
    if (jobz == 1)
        for (i = 0; i < n * n; ++i)
            Q[i] = (i % (n + 1) == 0) ? (real_t)1 : (real_t)0;

    /* Sweep budget: 30 implicit steps per eigenvalue, counted over the whole
     * problem (perf_steqr setup paragraph). */
    const long budget = (long)maxit_per_n * (long)n;
    long jtot = 0;

    /* algo_steqr, CTA split bookkeeping: running left boundary b_next. */
    int b_next = 0;
    while (b_next < n) {
        int lb = b_next;
        if (lb > 0)
            e[lb - 1] = (real_t)0;
        int le = lb;
        while (le < n - 1 && e[le] != (real_t)0)
            ++le;
        b_next = le + 1;
        if (le == lb)
            continue; /* a 1x1 block is final */

        /* algo_steqr, scaling paragraph: block infinity-norm estimate
         * max(|d_i|, |e_i|), then scale into [ssfmin, ssfmax]. */
        real_t anorm = 0;
        for (i = lb; i <= le; ++i)
            if (R_ABS(d[i]) > anorm)
                anorm = R_ABS(d[i]);
        for (i = lb; i < le; ++i)
            if (R_ABS(e[i]) > anorm)
                anorm = R_ABS(e[i]);
        if (anorm == (real_t)0)
            continue;
        int iscale = 0;
        real_t pre = 1, sc = 1, a_eff = anorm;
        if (anorm > R_SSFMAX) {
            iscale = 1;
            sc = R_SSFMAX / anorm;
        } else if (anorm < R_SSFMIN) {
            iscale = 2;
            if (anorm < R_SAFMIN) {
                /* subnormal norm: lift by an exact power of two first */
                pre = R_PRESCALE;
                a_eff = anorm * pre;
            }
            sc = R_SSFMIN / a_eff;
        }
        if (iscale) {
            for (i = lb; i <= le; ++i)
                d[i] = (d[i] * pre) * sc;
            for (i = lb; i < le; ++i)
                e[i] = (e[i] * pre) * sc;
        }

        /* Direction: converge the end of smaller magnitude first. */
        FN(view_t) v;
        if (R_ABS(d[lb]) <= R_ABS(d[le])) {
            v.lconv = lb;
            v.dir = 1; /* QL */
        } else {
            v.lconv = le;
            v.dir = -1; /* QR */
        }
        const int nloc = le - lb;
#define DD(p) d[FN(pidx)(v, (p))]
#define EE(p) e[FN(eidx)(v, (p))]
#define QC(p) FN(pidx)(v, (p))

        int lo = 0;
        int failed = 0;
        while (lo <= nloc) {
            /* algo_steqr, deflation criterion:
             * |e_i|^2 <= eps^2 |d_i| |d_{i+1}| + safmin  ->  e_i = 0. */
            int m = lo;
            while (m < nloc) {
                real_t tst = R_ABS(EE(m));
                tst = tst * tst;
                if (tst <= (eps2 * R_ABS(DD(m))) * R_ABS(DD(m + 1)) + R_SAFMIN)
                    break;
                ++m;
            }
            if (m < nloc)
                EE(m) = (real_t)0;
            if (m == lo) { /* eigenvalue DD(lo) has converged */
                ++lo;
                continue;
            }
            if (m == lo + 1) {
                /* algo_steqr, 2x2 block direct solve: Q2^T T2 Q2 = diag. */
                real_t a = DD(lo), b = EE(lo), c2 = DD(lo + 1);
                real_t tau = (c2 - a) / ((real_t)2 * b);
                real_t sgn = tau < (real_t)0 ? (real_t)-1 : (real_t)1;
                real_t t = sgn / (R_ABS(tau) + FN(hyp1)(tau));
                real_t cs = (real_t)1 / FN(hyp1)(t);
                real_t sn = -t * cs;
                DD(lo) = a - t * b;
                DD(lo + 1) = c2 + t * b;
                EE(lo) = (real_t)0;
                if (jobz)
                    FN(rot_cols)(n, Q, QC(lo), QC(lo + 1), cs, sn);
                cnt[2] += 1;
                lo += 2;
                continue;
            }
            if (jtot == budget) {
                failed = 1;
                break;
            }
            ++jtot;
            cnt[0] += 1;

            /* algo_steqr, copysign shift from the 2x2 block at the
             * converging end: g = (d2 - d1) / (2 e1), r = sqrt(g^2 + 1),
             * mu = d1 - e1 / (g + copysign(r, g)). */
            real_t d1 = DD(lo), d2 = DD(lo + 1), e1 = EE(lo);
            real_t g = (d2 - d1) / ((real_t)2 * e1);
            real_t r = FN(hyp1)(g);
            real_t mu = d1 - e1 / (g + R_COPYSIGN(r, g));

            if (scheme == 1) {
                /* algo_steqr, update schemes: PG propagates (g, p, c, s)
                 * across the sweep.  The page gives the QR form; this is the
                 * mirrored recurrence with the sweep reversed (QL form, in
                 * converging coordinates), seeded with g = d_m - mu,
                 * c = s = 1, p = 0:
                 *   f = s e, b = c e, (c, s, r) = lartg(g, f), e_prev <- r,
                 *   g* = d_i0 - p, r* = (d_i1 - g*) s + 2 c b, p = s r*,
                 *   d_i0 <- g* + p, g = c r* - b;
                 * after the last step d_lo <- d_lo - p and e_lo <- g. */
                real_t g = DD(m) - mu, sp = 1, cp = 1, p = 0;
                for (int q = 0; q < m - lo; ++q) {
                    int i0 = m - q, i1 = m - q - 1;
                    real_t f = sp * EE(i1), b = cp * EE(i1), rr;
                    FN(lartg)(g, f, &cp, &sp, &rr);
                    if (q > 0)
                        EE(i0) = rr;
                    real_t gs = DD(i0) - p;
                    real_t rs = (DD(i1) - gs) * sp + (real_t)2 * cp * b;
                    p = sp * rs;
                    DD(i0) = gs + p;
                    g = cp * rs - b;
                    if (jobz)
                        FN(rot_cols)(n, Q, QC(i0), QC(i1), cp, sp);
                    cnt[1] += 1;
                }
                DD(lo) = DD(lo) - p;
                EE(lo) = g;
                continue;
            }

            /* algo_steqr, implicit bulge chase: the first rotation comes from
             * the shifted corner (d_m - mu, e_{m-1}) at the far end of the
             * sweep, every later one from (e_current, bulge).  Each step is
             * the similarity T+ = G^T T G on the pair (i0, i1), written out
             * from that definition (EXP form), with the new bulge s * e. */
            real_t f = DD(m) - mu;
            real_t gg = EE(m - 1);
            for (int q = 0; q < m - lo; ++q) {
                int i0 = m - q, i1 = m - q - 1;
                real_t c, s, rr;
                FN(lartg)(f, gg, &c, &s, &rr);
                if (q > 0)
                    EE(i0) = rr;
                real_t aa = DD(i0), bb = EE(i1), cc = DD(i1);
                DD(i0) = c * c * aa + (real_t)2 * c * s * bb + s * s * cc;
                DD(i1) = s * s * aa - (real_t)2 * c * s * bb + c * c * cc;
                EE(i1) = c * s * (cc - aa) + (c * c - s * s) * bb;
                if (i1 > lo) {
                    real_t eo = EE(i1 - 1);
                    gg = s * eo;
                    EE(i1 - 1) = c * eo;
                    f = EE(i1);
                }
                if (jobz)
                    FN(rot_cols)(n, Q, QC(i0), QC(i1), c, s);
                cnt[1] += 1;
            }
        }
#undef DD
#undef EE
#undef QC

        /* algo_steqr, scaling paragraph: scale back by alpha^-1. */
        if (iscale == 1) {
            real_t us = anorm / R_SSFMAX;
            for (i = lb; i <= le; ++i)
                d[i] = d[i] * us;
            if (failed)
                for (i = lb; i < le; ++i)
                    e[i] = e[i] * us;
        } else if (iscale == 2) {
            real_t us = a_eff / R_SSFMIN;
            real_t upre = (real_t)1 / pre;
            for (i = lb; i <= le; ++i)
                d[i] = (d[i] * us) * upre;
            if (failed)
                for (i = lb; i < le; ++i)
                    e[i] = (e[i] * us) * upre;
        }
        if (failed) {
            int info = 0;
            for (i = 0; i + 1 < n; ++i)
                if (e[i] != (real_t)0)
                    ++info;
            return info; /* output left unsorted */
        }
    }

    /* algo_steqr, final paragraph: ascending order, same permutation on the
     * columns of Q.  Stable: equal values keep their original order. */
    if (sort && n > 1) {
        int perm[ORACLE_MAX_N];
        real_t val[ORACLE_MAX_N];
        for (i = 0; i < n; ++i) {
            perm[i] = i;
            val[i] = d[i];
        }
        for (i = 1; i < n; ++i) { /* insertion sort, strict comparison */
            real_t x = val[i];
            int pi = perm[i];
            int j = i - 1;
            while (j >= 0 && val[j] > x) {
                val[j + 1] = val[j];
                perm[j + 1] = perm[j];
                --j;
            }
            val[j + 1] = x;
            perm[j + 1] = pi;
        }
        for (i = 0; i < n; ++i)
            d[i] = val[i];
        if (jobz) {
            real_t tmp[ORACLE_MAX_N * ORACLE_MAX_N];
            for (i = 0; i < n * n; ++i)
                tmp[i] = Q[i];
            for (int j = 0; j < n; ++j)
                for (i = 0; i < n; ++i)
                    Q[(size_t)j * n + i] = tmp[(size_t)perm[j] * n + i];
        }
    }
    return 0;
}

/* 2-norm of x[0..m-1], scaled by the largest magnitude so that squares
 * neither overflow nor underflow. */
static real_t FN(nrm2)(int m, const real_t *x)
{
    real_t sc = 0;
    for (int k = 0; k < m; ++k)
        if (R_ABS(x[k]) > sc)
            sc = R_ABS(x[k]);
    if (sc == (real_t)0)
        return (real_t)0;
    real_t ss = 0;
    for (int k = 0; k < m; ++k) {
        real_t y = x[k] / sc;
        ss += y * y;
    }
    return sc * R_SQRT(ss);
}

/*
 * Dense symmetric A (n x n, column-major, lower triangle read) to tridiagonal
 * form by Householder reflectors, the plain unblocked lower reduction: for
 * i = 0 .. n-2 the reflector H_i = I - tau v v^T (v_{i+1} = 1, v_k = 0 for
 * k <= i) annihilates A[i+2:n, i] and is applied from both sides to the
 * trailing block, so T = Q^T A Q with Q = H_0 H_1 ... H_{n-2}.  The fused
 * small-n syev (BatchLAS page "perf_steqr": sytrd, then the steqr solve, then
 * the back-transform in one kernel) names this step; the pages give no
 * formulas for it, so this is the standard form.  d[n], e[n-1] receive T;
 * A is overwritten with the reflectors; Z (if not null) receives Q.
 */
static void FN(sytd2_lower)(int n, real_t *A, real_t *d, real_t *e, real_t *Z)
{
    real_t tau[64], v[64], p[64];
    for (int i = 0; i + 1 < n; ++i) {
        real_t *col = A + (size_t)i * n;
        real_t alpha = col[i + 1];
        real_t xnorm = FN(nrm2)(n - i - 2, col + i + 2);
        real_t t = 0;
        if (xnorm != (real_t)0) {
            real_t beta = -R_COPYSIGN(FN(hypot2)(alpha, xnorm), alpha);
            t = (beta - alpha) / beta;
            real_t scal = (real_t)1 / (alpha - beta);
            for (int k = i + 2; k < n; ++k)
                col[k] = col[k] * scal;
            alpha = beta;
        }
        e[i] = alpha;
        tau[i] = t;
        if (t != (real_t)0) {
            v[i + 1] = 1;
            for (int k = i + 2; k < n; ++k)
                v[k] = col[k];
            /* p = tau A22 v with A22 = A[i+1:n, i+1:n] (symmetric, lower) */
            for (int r = i + 1; r < n; ++r) {
                real_t acc = 0;
                for (int c = i + 1; c < n; ++c) {
                    real_t arc = r >= c ? A[r + (size_t)c * n] : A[c + (size_t)r * n];
                    acc += arc * v[c];
                }
                p[r] = t * acc;
            }
            /* w = p - (tau/2) (p^T v) v;  A22 <- A22 - v w^T - w v^T */
            real_t pv = 0;
            for (int r = i + 1; r < n; ++r)
                pv += p[r] * v[r];
            real_t a2 = -(real_t)0.5 * t * pv;
            for (int r = i + 1; r < n; ++r)
                p[r] = p[r] + a2 * v[r];
            for (int c = i + 1; c < n; ++c)
                for (int r = c; r < n; ++r)
                    A[r + (size_t)c * n] -= v[r] * p[c] + p[r] * v[c];
        }
        d[i] = A[i + (size_t)i * n];
    }
    d[n - 1] = A[(n - 1) + (size_t)(n - 1) * n];
    if (Z) {
        /* Q = H_0 (H_1 (... H_{n-2})): start from I and left-apply the
         * reflectors last to first; H_i changes rows i+1.. of columns i+1.. */
        for (int k = 0; k < n * n; ++k)
            Z[k] = (k % (n + 1) == 0) ? (real_t)1 : (real_t)0;
        for (int i = n - 2; i >= 0; --i) {
            if (tau[i] == (real_t)0)
                continue;
            const real_t *col = A + (size_t)i * n;
            v[i + 1] = 1;
            for (int k = i + 2; k < n; ++k)
                v[k] = col[k];
            for (int c = i + 1; c < n; ++c) {
                real_t s = 0;
                for (int r = i + 1; r < n; ++r)
                    s += v[r] * Z[r + (size_t)c * n];
                s = s * tau[i];
                for (int r = i + 1; r < n; ++r)
                    Z[r + (size_t)c * n] -= s * v[r];
            }
        }
    }
}

/* Fused small-n syev of one problem: reduction, then the steqr solve with the
 * reduction's Q as the basis (back_transform).  A (n x n, column-major, lower
 * read) is overwritten; W[n] receives the eigenvalues, V[n*n] (if jobz) the
 * eigenvectors of A. */
static int FN(syev_one)(int n, int jobz, int maxit_per_n, int sort, int scheme,
                        real_t *A, real_t *W, real_t *V, real_t *ework, long *cnt)
{
    real_t e[64];
    int bad = 0;
    for (int c = 0; c < n; ++c)
        for (int r = c; r < n; ++r)
            if (!isfinite(A[r + (size_t)c * n]))
                bad = 1;
    if (bad) {
        for (int k = 0; k < n; ++k)
            W[k] = (real_t)NAN;
        if (jobz)
            for (int k = 0; k < n * n; ++k)
                V[k] = (real_t)NAN;
        return -1;
    }
    FN(sytd2_lower)(n, A, W, e, jobz ? V : (real_t *)0);
    return FN(steqr_one)(n, jobz ? 2 : 0, maxit_per_n, sort, scheme, W, e, V, ework, cnt);
}

/* Batch driver arguments, one worker per contiguous slice of the batch. */
typedef struct {
    int n, jobz, maxit_per_n, sort, scheme;
    long b0, b1;
    real_t *d;
    const real_t *e;
    real_t *Q;
    int *info;
    long cnt[3];
} FN(job_t);

static void *FN(worker)(void *arg)
{
    FN(job_t) *jb = (FN(job_t) *)arg;
    const int n = jb->n;
    real_t ework[ORACLE_MAX_N];
    for (long b = jb->b0; b < jb->b1; ++b) {
        real_t *db = jb->d + b * n;
        const real_t *eb = jb->e + b * (n > 1 ? n - 1 : 0);
        real_t *Qb = jb->jobz ? jb->Q + b * (long)n * n : (real_t *)0;
        jb->info[b] = FN(steqr_one)(n, jb->jobz, jb->maxit_per_n, jb->sort, jb->scheme,
                                    db, eb, Qb, ework, jb->cnt);
    }
    return (void *)0;
}

typedef struct {
    int n, jobz, maxit_per_n, sort, scheme;
    long b0, b1;
    real_t *A, *W, *V;
    int *info;
    long cnt[3];
} FN(sjob_t);

static void *FN(sworker)(void *arg)
{
    FN(sjob_t) *jb = (FN(sjob_t) *)arg;
    const int n = jb->n;
    real_t ework[64];
    for (long b = jb->b0; b < jb->b1; ++b)
        jb->info[b] = FN(syev_one)(n, jb->jobz, jb->maxit_per_n, jb->sort, jb->scheme,
                                   jb->A + b * (long)n * n, jb->W + b * n,
                                   jb->jobz ? jb->V + b * (long)n * n : (real_t *)0, ework, jb->cnt);
    return (void *)0;
}

/* Fused syev of a batch (A: batch x n x n column-major, lower read and
 * overwritten; W: batch x n; V: batch x n x n when jobz).  Same threading and
 * counters as oracle_steqr_batch.  Returns 0, or -1 for invalid arguments. */
int FN(oracle_syev_batch)(int n, long batch, int jobz, int maxit_per_n, int sort,
                          real_t *A, real_t *W, real_t *V, int *info, long *counters,
                          int nthreads, int scheme)
{
    if (n < 1 || n > 64 || batch < 0 || maxit_per_n < 0 || scheme < 0 || scheme > 1)
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((long)nthreads > batch)
        nthreads = batch > 0 ? (int)batch : 1;
    FN(sjob_t) jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].n = n;
        jobs[t].jobz = jobz;
        jobs[t].maxit_per_n = maxit_per_n;
        jobs[t].sort = sort;
        jobs[t].scheme = scheme;
        jobs[t].b0 = batch * t / nthreads;
        jobs[t].b1 = batch * (t + 1) / nthreads;
        jobs[t].A = A;
        jobs[t].W = W;
        jobs[t].V = V;
        jobs[t].info = info;
        jobs[t].cnt[0] = jobs[t].cnt[1] = jobs[t].cnt[2] = 0;
    }
    if (nthreads == 1) {
        FN(sworker)(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], (void *)0, FN(sworker), &jobs[t]);
        for (int t = 0; t < nthreads; ++t)
            pthread_join(th[t], (void *)0);
    }
    if (counters) {
        counters[0] = counters[1] = counters[2] = 0;
        for (int t = 0; t < nthreads; ++t)
            for (int k = 0; k < 3; ++k)
                counters[k] += jobs[t].cnt[k];
    }
    return 0;
}

/* Solve a batch of problems (d: batch x n, e: batch x (n-1), Q: batch x n x n
 * column-major per problem) on nthreads host threads, static partition.
 * scheme: 0 the EXP update, 1 the PG update (algo_steqr, update schemes).
 * counters[0..2] receive the summed (implicit steps, rotations, 2x2 solves).
 * Returns 0, or -1 for invalid arguments. */
int FN(oracle_steqr_batch)(int n, long batch, int jobz, int maxit_per_n,
                           int sort, real_t *d, const real_t *e, real_t *Q,
                           int *info, long *counters, int nthreads, int scheme)
{
    if (n < 1 || n > ORACLE_MAX_N || batch < 0 || maxit_per_n < 0 || scheme < 0 || scheme > 1)
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((long)nthreads > batch)
        nthreads = batch > 0 ? (int)batch : 1;
    FN(job_t) jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].n = n;
        jobs[t].jobz = jobz;
        jobs[t].maxit_per_n = maxit_per_n;
        jobs[t].sort = sort;
        jobs[t].scheme = scheme;
        jobs[t].b0 = batch * t / nthreads;
        jobs[t].b1 = batch * (t + 1) / nthreads;
        jobs[t].d = d;
        jobs[t].e = e;
        jobs[t].Q = Q;
        jobs[t].info = info;
        jobs[t].cnt[0] = jobs[t].cnt[1] = jobs[t].cnt[2] = 0;
    }
    if (nthreads == 1) {
        FN(worker)(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], (void *)0, FN(worker), &jobs[t]);
        for (int t = 0; t < nthreads; ++t)
            pthread_join(th[t], (void *)0);
    }
    if (counters) {
        counters[0] = counters[1] = counters[2] = 0;
        for (int t = 0; t < nthreads; ++t)
            for (int k = 0; k < 3; ++k)
                counters[k] += jobs[t].cnt[k];
    }
    return 0;
}
