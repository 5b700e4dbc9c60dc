// Lane-per-problem steqr kernel, dynamic-position form.
//
// One CUDA thread owns one problem of size n <= NM, as in bstq_lane.cuh, but
// d and e live in shared memory (entry i of the lane's d at sd[i * blockDim],
// of e at se[i * blockDim]: the lanes of a warp hit consecutive words whatever
// index each one is at, so no access conflicts) and every lane chases its own
// positions.  A sweep of L rotations is L steps of a rolled loop; the warp
// runs max(L) steps per pass (flat scheduler) and a lane past its own sweep
// sits the rest out.  Compared with the static-position kernel there is no
// union of position ranges to pay for and the loop body is small.
//
// The per-problem operations are those of the BatchLAS page "algo_steqr"
// (deflation, scaling, copysign shift, lartg + EXP bulge chase, direct 2x2
// solve, eigenvector accumulation, ascending sort) with QR blocks mirrored at
// load as in bstq_lane.cuh ("perf_steqr", direction unification), and the
// schedulers of "perf_steqr", section "Lockstep flat solver".
#pragma once

#include <type_traits>

#include "bstq_lane.cuh"

namespace bstq {

// Q columns in memory (global scratch or shared), one 16-byte vector per
// group of rows, vector g of column k of thread t at base[(k*G + g)*stride+t].
template <typename T, int NM>
struct DynQ {
    using Tr = El<T>;
    using E = typename Tr::E;
    static constexpr int RPE = Tr::RPE;
    static constexpr int W = 16 / (int)sizeof(T);
    static constexpr int NR = ((NM + W - 1) / W) * W;  // stored rows
    static constexpr int NE = NR / RPE;
    static constexpr int G = NE / 2;
    struct V16 {
        E a, b;
    };
    V16 *base;
    int stride;

    __device__ __forceinline__ void load(int k, E (&x)[NE]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const V16 v = base[(k * G + g) * stride];
            x[2 * g] = v.a;
            x[2 * g + 1] = v.b;
        }
    }
    __device__ __forceinline__ void store(int k, const E (&x)[NE]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g)
            base[(k * G + g) * stride] = V16{x[2 * g], x[2 * g + 1]};
    }
    __device__ __forceinline__ V16 &vec(int k, int g) const { return base[(k * G + g) * stride]; }
    // Column s from a basis stored interleaved: row r at zc[r * st] (the
    // fused syev's reduction), zero below n.
    __device__ __forceinline__ void init_col_strided(int s, const T *zc, int st, int n) const
    {
        T col[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r)
            col[r] = r < n ? zc[(size_t)r * st] : T(0);
        E x[NE];
#pragma unroll
        for (int j = 0; j < NE; ++j)
            x[j] = Tr::pack(&col[j * RPE]);
        store(s, x);
    }
    // Column s from the caller's basis: rows 0 .. n-1 of zc, zero below
    // (back_transform).
    __device__ __forceinline__ void init_col_from(int s, const T *zc, int n, bool vec) const
    {
        T col[NR];
        load_col(zc, col, n, vec);
        E x[NE];
#pragma unroll
        for (int j = 0; j < NE; ++j)
            x[j] = Tr::pack(&col[j * RPE]);
        store(s, x);
    }
    __device__ __forceinline__ void init_col(int s, int row_of_one) const
    {
        E x[NE];
#pragma unroll
        for (int j = 0; j < NE; ++j)
            x[j] = Tr::unit(row_of_one, j * RPE);
        store(s, x);
    }
};

// One bit per entry for problems of 65 to 128 entries: two 64-bit words,
// kept as two scalars (an array member, even indexed with constants, sent
// the whole lane structure to local memory), with the few operations the
// lane's block bookkeeping needs; the 32- and 64-bit masks use the plain
// integer operators.
struct Mask128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ void mask_clear(unsigned &m) { m = 0u; }
__device__ __forceinline__ void mask_clear(unsigned long long &m) { m = 0ull; }
__device__ __forceinline__ void mask_clear(Mask128 &m) { m.lo = m.hi = 0ull; }
__device__ __forceinline__ void mask_set(unsigned &m, int i) { m |= 1u << i; }
__device__ __forceinline__ void mask_set(unsigned long long &m, int i) { m |= 1ull << i; }
__device__ __forceinline__ void mask_set(Mask128 &m, int i)
{
    const unsigned long long bit = 1ull << (i & 63);
    m.lo |= i < 64 ? bit : 0ull;
    m.hi |= i < 64 ? 0ull : bit;
}
__device__ __forceinline__ bool mask_test(unsigned m, int i) { return (m >> i) & 1u; }
__device__ __forceinline__ bool mask_test(unsigned long long m, int i) { return (m >> i) & 1ull; }
__device__ __forceinline__ bool mask_test(const Mask128 &m, int i)
{
    return ((i < 64 ? m.lo : m.hi) >> (i & 63)) & 1ull;
}
// every bit from i on (i >= 0)
__device__ __forceinline__ void mask_set_from(unsigned &m, int i) { m |= i < 32 ? (~0u << i) : 0u; }
__device__ __forceinline__ void mask_set_from(unsigned long long &m, int i) { m |= i < 64 ? (~0ull << i) : 0ull; }
__device__ __forceinline__ void mask_set_from(Mask128 &m, int i)
{
    m.lo |= i < 64 ? (~0ull << i) : 0ull;
    m.hi |= i <= 64 ? ~0ull : (i < 128 ? (~0ull << (i - 64)) : 0ull);
}
__device__ __forceinline__ bool mask_any(unsigned m) { return m != 0u; }
__device__ __forceinline__ bool mask_any(unsigned long long m) { return m != 0ull; }
__device__ __forceinline__ bool mask_any(const Mask128 &m) { return (m.lo | m.hi) != 0ull; }
// Block [lb, le] containing index s from a boundary mask (bit i set when
// e_i is an exact zero or i >= n-1): the first set bit at or after s, and
// one past the last set bit before s.
__device__ __forceinline__ int block_hi(const Mask128 &m, int s)
{
    const unsigned long long xl = s < 64 ? (m.lo >> s) << s : 0ull;
    const unsigned long long xh = s <= 64 ? m.hi : (m.hi >> (s - 64)) << (s - 64);
    return xl ? __ffsll((long long)xl) - 1 : (xh ? 64 + __ffsll((long long)xh) - 1 : 127);
}
__device__ __forceinline__ int block_lo(const Mask128 &m, int s)
{
    const unsigned long long xl = s >= 64 ? m.lo : (s > 0 ? m.lo & ((1ull << s) - 1ull) : 0ull);
    const unsigned long long xh = s >= 128 ? m.hi : (s > 64 ? m.hi & ((1ull << (s - 64)) - 1ull) : 0ull);
    return xh ? 128 - __clzll((long long)xh) : (xl ? 64 - __clzll((long long)xl) : 0);
}

// double eigenvectors are accumulated in factored form Q = Qt diag(delta)
// (fast Givens, after Gentleman): a rotation then costs two FMAs per row
// instead of two multiplies and two FMAs, plus a dozen scalar operations for
// the column scales; delta and its inverse live in shared memory.
template <typename T, bool WANTZ>
constexpr bool dyn_fastq()
{
    return WANTZ && sizeof(T) == 8;
}

// With LOG set (float, eigenvalues-only chase) every pass is also appended
// to the problem's rotation log (the record-and-apply kernels,
// bstq_rlog.cuh): a header entry (top position m and count, as integer
// bits), the rotations (cs, sn) of positions m, m-1, ..., lo + 1, and
// identity rotations (1, 0) for positions lo, ..., down to the next
// multiple of kRlogGroup, so that every logged pass ends on a group
// boundary and its reader tests for the end once per group.
constexpr int kRlogGroup = 4;

template <typename T, int NM, bool WANTZ, bool LOG = false>
struct DynLane {
    static_assert(!LOG || (sizeof(T) == 4 && !WANTZ), "the rotation log is for the float chase without Q");
    using C_ = Consts<T>;
    using Q_ = DynQ<T, NM>;
    using E = typename Q_::E;
    static constexpr int NE = Q_::NE;
    static constexpr bool FASTQ = dyn_fastq<T, WANTZ>();
    // Block-boundary and mirror masks: one bit per entry.
    static_assert(NM <= 128, "block masks hold up to 128 entries");
    using Mask = typename std::conditional<
        (NM > 64), Mask128, typename std::conditional<(NM > 32), unsigned long long, unsigned>::type>::type;
    // The column shared by successive rotations of a sweep stays in
    // registers.  For double above n = 32, and float above n = 64, the whole
    // next column would not fit beside it, so that column is read and
    // rotated in groups of vectors and the carried one is kept in shared
    // memory (step_q_carry_chunked); float up to n = 64 reads the whole
    // next column at once (up to 32 packed pairs), which measured faster.
    static constexpr bool CHUNKED = (sizeof(T) == 8 && NM > 32) || NM > 64;
    // Above n = 64 the carried column itself lives in shared memory; at
    // n = 48 and 64 (double) it stays in registers, which measured faster
    // (f64 n = 64 V 169 against 221 ms, n = 48 45 against 77 ms): the extra
    // shared memory per thread cost a warp of occupancy.
    static constexpr bool CARRY_SMEM = NM > 64;
    // From n = 48 on, the double column scales live in global scratch next
    // to Q (element j of thread t at [j * blockDim + t], L1-resident)
    // instead of shared memory: shared memory per thread, not registers,
    // limited these kernels to three warps per SM.
    static constexpr bool DELTA_GLOBAL = FASTQ && NM >= 48;

    T *sd, *se;  // this lane's d and e in shared memory
    T *sdl, *sil;  // column scales delta_j and 1/delta_j (FASTQ)
    int ms;      // their stride (blockDim.x)
    T da, ia;    // scale and inverse scale of the carried column C (FASTQ)
    int n, status, info;
    Mask zmask, revmask;
    bool inblock;
    int bnext, lb, le, lo;
    int iscale;
    T pre, sc, aeff, anorm;
    int jtot, budget;
    int task, m;
    T f, g;        // running pair (PG: f is the running g of the recurrence)
    T cs2, sn2;    // pending 2x2 rotation
    bool pg;       // PG update scheme for sweeps (else EXP)
    T pg_c, pg_s, pg_p;  // PG: previous rotation and p
    // pass state
    int L, C;      // steps of the current task, current position
    T a_reg, b_reg;  // d_C and e_{C-1} as updated by the previous step
    Q_ q;
    E cur[CARRY_SMEM ? 1 : NE];  // Q column C (the column shared with the next rotation)
    E *scr;        // CARRY_SMEM: that column in shared memory instead,
                   // element j at scr[j * ms]
    float2 *lg;    // LOG: this problem's rotation log, its entry count and
    int cnt, lpad; // the identity entries that end the current pass
    __device__ __forceinline__ E &carry(int j)
    {
        if constexpr (CARRY_SMEM)
            return scr[j * ms];
        else
            return cur[j];
    }

    __device__ __forceinline__ T D(int i) const { return sd[i * ms]; }
    __device__ __forceinline__ T Ev(int i) const { return se[i * ms]; }
    __device__ __forceinline__ void setD(int i, T v) { sd[i * ms] = v; }
    __device__ __forceinline__ void setE(int i, T v) { se[i * ms] = v; }

    __device__ __forceinline__ int phys(int s) const
    {
        int a = block_lo(zmask, s), b = block_hi(zmask, s);
        return mask_test(revmask, a) ? (a + b - s) : s;
    }

    __device__ __forceinline__ void scale_factors(T an, int &isc, T &pr, T &s, T &ae) const
    {
        isc = 0;
        pr = T(1);
        s = T(1);
        ae = an;
        if (an > C_::ssfmax) {
            isc = 1;
            s = C_::ssfmax / an;
        } else if (an < C_::ssfmin) {
            isc = 2;
            if (an < C_::safmin) {
                pr = C_::prescale;
                ae = an * pr;
            }
            s = C_::ssfmin / ae;
        }
    }

    __device__ __forceinline__ T block_norm(int a, int b) const
    {
        T an = T(0);
        for (int i = a; i <= b; ++i)
            an = fmax(an, dabs(D(i)));
        for (int i = a; i < b; ++i)
            an = fmax(an, dabs(Ev(i)));
        return an;
    }

    __device__ void load(const KParams &p, long long b, bool live)
    {
        n = p.n;
        budget = p.budget;
        jtot = 0;
        task = TASK_NONE;
        inblock = false;
        bnext = 0;
        lb = le = lo = m = 0;
        info = 0;
        mask_clear(revmask);
        iscale = 0;
        pre = sc = aeff = anorm = T(1);
        f = g = cs2 = sn2 = a_reg = b_reg = T(0);
        L = 0;
        C = 0;
        if (!live) {
            status = ST_DEAD;
            mask_clear(zmask);
            mask_set_from(zmask, 0);
            return;
        }
        const T *dg = reinterpret_cast<const T *>(p.d) + b * n;
        const T *eg = reinterpret_cast<const T *>(p.e) + b * (n - 1);
        bool bad = false;
        mask_clear(zmask);
        for (int i = 0; i < n; ++i) {
            const T di = dg[i];
            const T ei = i < n - 1 ? eg[i] : T(0);
            setD(i, di);
            setE(i, ei);
            bad |= !isfinite(di) || !isfinite(ei);
            if (i >= n - 1 || ei == T(0))
                mask_set(zmask, i);
        }
        mask_set_from(zmask, n);
        status = bad ? ST_BAD : ST_RUN;
        if (bad)
            return;
        for (int a = 0; a < n;) {
            const int z = block_hi(zmask, a);
            if (z > a) {
                const T an = block_norm(a, z);
                if (an > T(0)) {
                    int isc;
                    T pr, s, ae;
                    scale_factors(an, isc, pr, s, ae);
                    T x = D(a), y = D(z);
                    if (isc) {
                        x = (x * pr) * s;
                        y = (y * pr) * s;
                    }
                    if (dabs(x) > dabs(y))
                        mask_set(revmask, a);
                }
            }
            a = z + 1;
        }
        if (mask_any(revmask)) {
            for (int s = 0; s < n; ++s) {
                const int ps = phys(s);
                setD(s, dg[ps]);
                if (s < n - 1 && !mask_test(zmask, s)) {
                    const int pn = phys(s + 1);
                    setE(s, eg[ps < pn ? ps : pn]);
                }
            }
        }
    }

    __device__ __forceinline__ void scale_range(T f1, T f2, bool with_e)
    {
        for (int i = lb; i <= le; ++i)
            setD(i, (D(i) * f1) * f2);
        if (with_e)
            for (int i = lb; i < le; ++i)
                setE(i, (Ev(i) * f1) * f2);
    }

    __device__ __forceinline__ void unscale_block(bool with_e)
    {
        if (iscale == 0)
            return;
        T us, up = T(1);
        if (iscale == 1) {
            us = anorm / C_::ssfmax;
        } else {
            us = aeff / C_::ssfmin;
            up = T(1) / pre;
        }
        scale_range(us, up, with_e);
    }

    __device__ __forceinline__ void close_block()
    {
        unscale_block(false);
        inblock = false;
    }

    // Settle the lane (advance past converged eigenvalues and blocks until
    // it has a task, is done or has exhausted its budget); consecutive
    // deflations are handled in one call.
    __device__ void settle_step()
    {
        int mm;
        for (;;) {
            if (!inblock) {
                if (bnext >= n) {
                    status = ST_DONE;
                    return;
                }
                lb = bnext;
                le = block_hi(zmask, lb);
                bnext = le + 1;
                if (le == lb)
                    continue;
                anorm = block_norm(lb, le);
                if (anorm == T(0))
                    continue;
                scale_factors(anorm, iscale, pre, sc, aeff);
                if (iscale)
                    scale_range(pre, sc, true);
                lo = lb;
                inblock = true;
            }
            // first negligible off-diagonal from lo (page "algo_steqr")
            mm = le;
            T dcur = D(lo);
            for (int i = lo; i < le; ++i) {
                const T dn = D(i + 1);
                const T ev = Ev(i);
                bool neg;
                if constexpr (sizeof(T) == 8) {
                    // Exponent bounds first (integer pipe).  With k the biased
                    // exponent field, 2^(k-1023) <= |x| < 2^(k-1022) (the upper
                    // bound holds for zero and subnormals too), so
                    // e^2 >= 2^(2 k_e - 2046), eps^2 |d_i d_i+1| < 2^(k_1 + k_2 - 2150)
                    // and safmin = 2^-1022.  When 2 k_e >= k_1 + k_2 - 99 and
                    // 2 k_e >= 1037, e^2 exceeds each term of the threshold by a
                    // factor of 8 or more, so the off-diagonal is certainly not
                    // negligible and the FP64 test is skipped.  (Scaled inputs
                    // are finite here.)
                    const int ke = (__double2hiint(ev) >> 20) & 0x7ff;
                    const int k1 = (__double2hiint(dcur) >> 20) & 0x7ff;
                    const int k2 = (__double2hiint(dn) >> 20) & 0x7ff;
                    const bool clear = (2 * ke > k1 + k2 - 100) && (2 * ke > 1036);
                    neg = false;
                    if (!clear) {
                        const T ae = dabs(ev);
                        const T tst = ae * ae;
                        const T thr = fma(C_::eps2 * dabs(dcur), dabs(dn), C_::safmin);
                        // non-negative doubles order as their bit patterns
                        neg = __double_as_longlong(tst) <= __double_as_longlong(thr);
                    }
                } else {
                    const T ae = dabs(ev);
                    const T tst = ae * ae;
                    const T thr = fma(C_::eps2 * dabs(dcur), dabs(dn), C_::safmin);
                    neg = tst <= thr;
                }
                if (neg) {
                    mm = i;
                    break;
                }
                dcur = dn;
            }
            if (mm < le)
                setE(mm, T(0));
            if (mm != lo)
                break;
            ++lo;  // eigenvalue at lo has converged
            if (lo > le)
                close_block();
        }
        const T d1 = D(lo), d2 = D(lo + 1), e1 = Ev(lo);
        T t, mu;
        shift_tangent(d1, d2, e1, t, mu);
        if (mm == lo + 1) {  // 2x2 direct solve
            rot_from_tangent(t, cs2, sn2);
            task = TASK_2X2;
            m = lo + 1;
            return;
        }
        if (jtot == budget) {
            unscale_block(true);
            int cnt = 0;
            for (int i = 0; i < n - 1; ++i)
                cnt += Ev(i) != T(0) ? 1 : 0;
            info = cnt;
            status = ST_FAIL;
            return;
        }
        ++jtot;
        f = D(mm) - mu;
        g = Ev(mm - 1);
        m = mm;
        task = TASK_SWEEP;
    }

    __device__ __forceinline__ bool has_task() const { return status == ST_RUN && task != TASK_NONE; }

    __device__ __forceinline__ void begin_pass()
    {
        if (!has_task()) {
            L = 0;
            return;
        }
        C = m;
        L = m - lo;  // 1 for a 2x2 task
        if constexpr (LOG) {
            lpad = lo % kRlogGroup;
            lg[cnt] = make_float2(__int_as_float(m), __int_as_float(L + lpad));
            for (int i = 0; i < lpad; ++i)
                lg[cnt + 1 + L + i] = make_float2(1.f, 0.f);
            ++cnt;
        }
        a_reg = D(C);
        b_reg = Ev(C - 1);
        pg_c = pg_s = T(1);
        pg_p = T(0);
        if constexpr (WANTZ) {
            if constexpr (CARRY_SMEM) {
                for (int g = 0; g < Q_::G; ++g) {
                    const typename Q_::V16 v = q.vec(C, g);
                    scr[(2 * g) * ms] = v.a;
                    scr[(2 * g + 1) * ms] = v.b;
                }
            } else {
                q.load(C, cur);
            }
        }
        if constexpr (FASTQ) {
            da = sdl[C * ms];
            ia = sil[C * ms];
        }
    }

    // Rotation k of the lane's task, on the pair (C, C-1).
    __device__ __forceinline__ void step(int k)
    {
        const bool sweep = task == TASK_SWEEP;
        T cs, sn, r = T(0);
        if (sweep && pg) {
            // PG (page "algo_steqr", update schemes), QL form: the scalars
            // (g, p, c, s) run across the sweep; d_C is final after this
            // step, e_C takes r, and the last step closes d_lo and e_lo.
            const T ev = Ev(C - 1);
            const T fb = pg_s * ev, bb = pg_c * ev;
            if constexpr (sizeof(T) == 8)
                lartg_fast(f, fb, cs, sn, r);
            else
                lartg(f, fb, cs, sn, r);
            if (k > 0)
                setE(C, r);
            const T gs = D(C) - pg_p;
            const T rs = fma(D(C - 1) - gs, sn, T(2) * cs * bb);
            pg_p = sn * rs;
            setD(C, gs + pg_p);
            f = fma(cs, rs, -bb);
            pg_c = cs;
            pg_s = sn;
            if (C - 1 == lo) {
                setD(lo, D(lo) - pg_p);
                setE(lo, f);
            }
        } else {
            step_exp(k, sweep, cs, sn, r);
        }
        step_q(cs, sn);
        if constexpr (LOG)
            lg[cnt++] = make_float2(cs, sn);
        --C;
    }

    // EXP step (and the 2x2 solve of either scheme): the similarity written
    // out on the pair (C, C-1).
    __device__ __forceinline__ void step_exp(int k, bool sweep, T &cs, T &sn, T &r)
    {
        if (sweep) {
            if constexpr (sizeof(T) == 8)
                lartg_fast(f, g, cs, sn, r);
            else
                lartg(f, g, cs, sn, r);
        } else {
            cs = cs2;
            sn = sn2;
        }
        const T a = a_reg, b = b_reg, cc = D(C - 1);
        // T+ = G^T T G on rows/columns (C, C-1) (page "algo_steqr", EXP)
        const T p1 = fma(cs, a, sn * b);
        const T p2 = fma(cs, b, sn * cc);
        const T dn = fma(cs, p1, sn * p2);
        T en = fma(cs, p2, -sn * p1);
        const T dm = (a + cc) - dn;
        setD(C, dn);
        if (sweep && k > 0)
            setE(C, r);
        if (!sweep)
            en = T(0);
        if (C - 1 > lo) {
            const T eo = Ev(C - 2);
            g = sn * eo;  // new bulge
            b_reg = cs * eo;
            f = en;
            a_reg = dm;
        } else {
            setD(C - 1, dm);
            setE(C - 1, en);
        }
    }

    // Eigenvector update of the step's rotation on columns (C, C-1).
    __device__ __forceinline__ void step_q(T cs, T sn)
    {
        if constexpr (!WANTZ)
            return;  // eigenvalues only: no Q (q.base is not set)
        else if constexpr (CHUNKED)
            step_q_carry_chunked(cs, sn);
        else
            step_q_carry(cs, sn);
    }

    // Fast-Givens scales drift: every rotation multiplies the two deltas it
    // touches by max(|cs|, |sn|) >= 1/sqrt(2) and nothing restores them, so
    // a column rotated a couple of thousand times (a large sweep budget at
    // large n) would see delta underflow and 1/delta overflow.  Before each
    // rotation a delta below 2^-128 is folded into its column of Qt
    // (Q = Qt diag(delta) is unchanged) and reset to one, which keeps every
    // delta above 2^-129 and every entry of Qt below 2^129.  The exponent
    // tests run on the integer pipe; the folds themselves are rare.
    __device__ __forceinline__ static bool scale_low(T x)
    {
        return ((unsigned)(__double2hiint(x) >> 20) & 0x7ffu) < 1023u - 128u;
    }
    // the carried column (registers)
    __device__ __forceinline__ void renorm_carried()
    {
        if (scale_low(da)) {
            if constexpr (CARRY_SMEM) {
                for (int j = 0; j < NE; ++j)
                    scr[j * ms] *= da;
            } else {
#pragma unroll
                for (int j = 0; j < NE; ++j)
                    cur[j] *= da;
            }
            da = T(1);
            ia = T(1);
        }
    }
    // column k in the scratch, with its scale dk and inverse ik
    __device__ __forceinline__ void renorm_mem(int k, T &dk, T &ik)
    {
        if (scale_low(dk)) {
            for (int g = 0; g < Q_::G; ++g) {
                typename Q_::V16 v = q.vec(k, g);
                v.a *= dk;
                v.b *= dk;
                q.vec(k, g) = v;
            }
            dk = T(1);
            ik = T(1);
            sdl[k * ms] = T(1);
            sil[k * ms] = T(1);
        }
    }

    // step_q_carry for double above n = 32: column C-1 is read four 16-byte
    // vectors at a time, the next group's reads issued before this group's
    // writes, so only the carried column and two groups are live in
    // registers (above n = 64 the carried column moves to shared memory).
    __device__ __forceinline__ void step_q_carry_chunked(T cs, T sn)
    {
        constexpr int G = Q_::G;
        constexpr int K = 4;  // vectors per group
        static_assert(G % K == 0, "column vectors in whole groups");
        using V = typename Q_::V16;
        T c1, c2, da2 = T(0), db2 = T(0), ia2 = T(0), ib2 = T(0);
        bool f1 = true;
        typename El<T>::R rr;
        if constexpr (FASTQ) {
            T db = sdl[(C - 1) * ms], ib = sil[(C - 1) * ms];
            renorm_carried();
            renorm_mem(C - 1, db, ib);
            f1 = (__double_as_longlong(cs) & 0x7fffffffffffffffll) >=
                 (__double_as_longlong(sn) & 0x7fffffffffffffffll);
            const T rp = rcp_nr(f1 ? cs : sn);
            const T t = (f1 ? sn : cs) * rp;
            const T P = t * (db * ia), M = t * (da * ib);
            c1 = f1 ? P : M;
            c2 = f1 ? -M : -P;
            da2 = (f1 ? cs : sn) * (f1 ? da : db);
            db2 = (f1 ? cs : -sn) * (f1 ? db : da);
            ia2 = (f1 ? ia : ib) * rp;
            ib2 = (f1 ? ib : -ia) * rp;
        } else {
            rr = El<T>::make(cs, sn);
        }
        V nx[2][K];
#pragma unroll
        for (int k = 0; k < K; ++k)
            nx[0][k] = q.vec(C - 1, k);
#pragma unroll
        for (int grp = 0; grp < G / K; ++grp) {
            const int bsel = grp & 1;
            if (grp + 1 < G / K) {
#pragma unroll
                for (int k = 0; k < K; ++k)
                    nx[bsel ^ 1][k] = q.vec(C - 1, (grp + 1) * K + k);
            }
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int j = 2 * (grp * K + k);
                E u0 = carry(j), u1 = carry(j + 1);
                E v0 = nx[bsel][k].a, v1 = nx[bsel][k].b;
                if constexpr (FASTQ) {
                    const E s10 = f1 ? v0 : u0, s20 = f1 ? u0 : v0;
                    const E s11 = f1 ? v1 : u1, s21 = f1 ? u1 : v1;
                    u0 = fma(c1, s10, s20);
                    v0 = fma(c2, s20, s10);
                    u1 = fma(c1, s11, s21);
                    v1 = fma(c2, s21, s11);
                } else {
                    El<T>::rot(u0, v0, rr);
                    El<T>::rot(u1, v1, rr);
                }
                q.vec(C, grp * K + k) = V{u0, u1};
                carry(j) = v0;
                carry(j + 1) = v1;
            }
        }
        if constexpr (FASTQ) {
            sdl[C * ms] = da2;
            sil[C * ms] = ia2;
            da = db2;
            ia = ib2;
        }
        if (C - 1 == lo) {
            // end of the sweep: the carried column is final
#pragma unroll
            for (int g = 0; g < G; ++g)
                q.vec(C - 1, g) = V{carry(2 * g), carry(2 * g + 1)};
            if constexpr (FASTQ) {
                sdl[(C - 1) * ms] = db2;
                sil[(C - 1) * ms] = ib2;
            }
        }
    }

    // Column C is in registers (cur), column C-1 is read, and C-1 becomes
    // the carried column.
    __device__ __forceinline__ void step_q_carry(T cs, T sn)
    {
        if constexpr (FASTQ) {
            // q_C = da x, q_{C-1} = db y.  Form 1 (|cs| >= |sn|):
            //   x' = x + P y, y' = y - M x, da' = cs da, db' = cs db;
            // form 2 (|sn| > |cs|), columns exchange their roles:
            //   x' = y + M x, y' = x - P y, da' = sn db, db' = -sn da;
            // with t = sn/cs (form 1) or cs/sn (form 2), P = t db/da,
            // M = t da/db.  Either way Qt' diag(delta') = Qt diag(delta) G.
            T db = sdl[(C - 1) * ms], ib = sil[(C - 1) * ms];
            renorm_carried();
            renorm_mem(C - 1, db, ib);
            E nx[NE];
            q.load(C - 1, nx);
            const bool f1 = (__double_as_longlong(cs) & 0x7fffffffffffffffll) >=
                            (__double_as_longlong(sn) & 0x7fffffffffffffffll);
            const T rp = rcp_nr(f1 ? cs : sn);
            const T t = (f1 ? sn : cs) * rp;
            const T P = t * (db * ia), M = t * (da * ib);
            const T c1 = f1 ? P : M, c2 = f1 ? -M : -P;
#pragma unroll
            for (int j = 0; j < NE; ++j) {
                const E u = cur[j], v = nx[j];
                const E s1 = f1 ? v : u, s2 = f1 ? u : v;
                cur[j] = fma(c1, s1, s2);
                nx[j] = fma(c2, s2, s1);
            }
            const T da2 = (f1 ? cs : sn) * (f1 ? da : db);
            const T db2 = (f1 ? cs : -sn) * (f1 ? db : da);
            const T ia2 = (f1 ? ia : ib) * rp;
            const T ib2 = (f1 ? ib : -ia) * rp;
            q.store(C, cur);
            sdl[C * ms] = da2;
            sil[C * ms] = ia2;
            if (C - 1 > lo) {
#pragma unroll
                for (int j = 0; j < NE; ++j)
                    cur[j] = nx[j];
                da = db2;
                ia = ib2;
            } else {
                q.store(C - 1, nx);
                sdl[(C - 1) * ms] = db2;
                sil[(C - 1) * ms] = ib2;
            }
        } else if constexpr (WANTZ) {
            E nx[NE];
            q.load(C - 1, nx);
            const typename El<T>::R rr = El<T>::make(cs, sn);
#pragma unroll
            for (int j = 0; j < NE; ++j)
                El<T>::rot(cur[j], nx[j], rr);
            q.store(C, cur);
            if (C - 1 > lo) {
#pragma unroll
                for (int j = 0; j < NE; ++j)
                    cur[j] = nx[j];
            } else {
                q.store(C - 1, nx);
            }
        }
    }

    __device__ __forceinline__ void post_pass()
    {
        if constexpr (LOG)
            cnt += lpad;  // the identity entries written with the header
        if (task == TASK_2X2) {
            lo += 2;
            if (lo > le)
                close_block();
        }
        task = TASK_NONE;
        L = 0;
    }
};

// The whole solve of one lane's problem (load, the settle/chase loop under
// the chosen scheduler, the sorted store); dyn_kernel and the fused syev
// kernel both run it.
template <typename T, int NM, bool WANTZ, int SCHED>
__device__ __forceinline__ void dyn_body(const KParams &p)
{
    extern __shared__ uint4 smem_raw[];
    using LaneT = DynLane<T, NM, WANTZ>;
    const int tpb = blockDim.x;
    const long long b = (long long)blockIdx.x * tpb + threadIdx.x;
    const bool live = b < p.batch;

    LaneT L;
    L.ms = tpb;
    L.sd = reinterpret_cast<T *>(smem_raw) + threadIdx.x;
    L.se = L.sd + NM * tpb;
    L.sdl = L.se + NM * tpb;
    L.sil = L.sdl + NM * tpb;
    if constexpr (LaneT::DELTA_GLOBAL) {
        // the column scales after every block's Q scratch, per block 2 NM
        // arrays of tpb values
        T *dg = reinterpret_cast<T *>(reinterpret_cast<typename DynQ<T, NM>::V16 *>(p.qwork) +
                                      (long long)gridDim.x * NM * DynQ<T, NM>::G * tpb);
        L.sdl = dg + (long long)blockIdx.x * 2 * NM * tpb + threadIdx.x;
        L.sil = L.sdl + NM * tpb;
    }
    // The carried column above n = 64 (CARRY_SMEM): its own region after d
    // and e (and the column scales when they are in shared memory), NE
    // elements of the update's element type per thread, element j of thread
    // t at [j * tpb + t].  The region starts at a multiple of 8 bytes from
    // the shared base (sizes are whole NM * tpb arrays of T), so 8-byte
    // elements stay aligned.
    L.scr = reinterpret_cast<typename LaneT::E *>(
                reinterpret_cast<char *>(smem_raw) +
                size_t((LaneT::FASTQ && !LaneT::DELTA_GLOBAL) ? 4 : 2) * NM * tpb * sizeof(T)) +
            threadIdx.x;
    L.da = L.ia = T(1);
    L.pg = p.scheme == 1;
    if constexpr (WANTZ) {
        // Q scratch in global memory: per block NM columns x G vectors x tpb
        constexpr int G = DynQ<T, NM>::G;
        L.q.base = reinterpret_cast<typename DynQ<T, NM>::V16 *>(p.qwork) +
                   ((long long)blockIdx.x * NM * G * tpb + threadIdx.x);
        L.q.stride = tpb;
    }
    L.load(p, b, live);
    if constexpr (WANTZ) {
        const T *zb = reinterpret_cast<const T *>(p.Q) + b * (long long)L.n * L.n;
        const bool zvec = q_vector_ok<T>(p.Q, L.n);
        if (L.status == ST_RUN)
            for (int s = 0; s < NM; ++s) {
                // column phys(s) of the identity, or of the caller's basis
                // with back_transform
                if (p.back == 2 && s < L.n)  // fused syev: Q of the reduction
                    L.q.init_col_strided(s,
                                         reinterpret_cast<const T *>(p.sscr) +
                                             ((size_t)blockIdx.x * 2 + 1) * L.n * L.n * tpb + threadIdx.x +
                                             (size_t)L.phys(s) * L.n * tpb,
                                         tpb, L.n);
                else if (p.back && s < L.n)
                    L.q.init_col_from(s, zb + (long long)L.phys(s) * L.n, L.n, zvec);
                else
                    L.q.init_col(s, s < L.n ? L.phys(s) : s);
                if constexpr (LaneT::FASTQ) {
                    L.sdl[s * tpb] = T(1);
                    L.sil[s * tpb] = T(1);
                }
            }
    }

    if (SCHED == SCHED_FLAT) {
        for (;;) {
            // settle every lane without a task (one call settles it fully)
            if (L.status == ST_RUN && L.task == TASK_NONE)
                L.settle_step();
            const bool has = L.has_task();
            if (!__any_sync(FULL, has))
                break;
            L.begin_pass();
            const int steps = __reduce_max_sync(FULL, L.L);
            for (int k = 0; k < steps; ++k)
                if (k < L.L)
                    L.step(k);
            if (has)
                L.post_pass();
        }
    } else {
        while (L.status == ST_RUN) {
            if (L.task == TASK_NONE) {
                L.settle_step();
                continue;
            }
            L.begin_pass();
            for (int k = 0; k < L.L; ++k)
                L.step(k);
            L.post_pass();
        }
    }

    if (!live)
        return;
    const int n = L.n;
    T *dout = reinterpret_cast<T *>(p.d) + b * n;
    T *qout = WANTZ ? reinterpret_cast<T *>(p.Q) + b * (long long)n * n : nullptr;
    if (L.status == ST_BAD) {
        const T nan = T(__int_as_float(0x7fffffff));
        for (int i = 0; i < n; ++i)
            dout[i] = nan;
        if (WANTZ)
            for (int i = 0; i < n * n; ++i)
                qout[i] = nan;
        p.info[b] = -1;
        return;
    }
    const bool sorted = p.sort && L.status == ST_DONE;
    if constexpr (NM > 32) {
        // n > 32: rolled ranking and column copy, 16 bytes at a time, so no
        // per-entry arrays live in registers
        using Q_ = DynQ<T, NM>;
        constexpr int W = 16 / (int)sizeof(T);
        const bool vec = WANTZ && q_vector_ok<T>(p.Q, n);
        for (int s = 0; s < n; ++s) {
            const T ds = L.D(s);
            const int phs = L.phys(s);
            int pos = phs;
            if (sorted) {
                pos = 0;
                for (int t = 0; t < n; ++t) {
                    const T dt = L.D(t);
                    pos += (dt < ds || (dt == ds && L.phys(t) < phs)) ? 1 : 0;
                }
            }
            dout[pos] = ds;
            if constexpr (WANTZ) {
                T scale = T(1);
                if constexpr (LaneT::FASTQ)
                    scale = L.sdl[s * tpb];  // Q = Qt diag(delta)
                T *qc = qout + (long long)pos * n;
                for (int g = 0; g < Q_::G && g * W < n; ++g) {
                    const typename Q_::V16 v = L.q.vec(s, g);
                    T x[W];
                    El<T>::get(v.a, &x[0]);
                    El<T>::get(v.b, &x[Q_::RPE]);
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        x[k] = LaneT::FASTQ ? x[k] * scale : x[k];
                    if (vec) {
                        struct alignas(16) V {
                            T y[W];
                        } o;
#pragma unroll
                        for (int k = 0; k < W; ++k)
                            o.y[k] = x[k];
                        reinterpret_cast<V *>(qc)[g] = o;
                    } else {
#pragma unroll
                        for (int k = 0; k < W; ++k)
                            if (g * W + k < n)
                                qc[g * W + k] = x[k];
                    }
                }
            }
        }
        p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
        return;
    }
    // eigenvalues into registers for the ranking
    T dv[NM];
    int ph[NM], pos[NM];
#pragma unroll
    for (int s = 0; s < NM; ++s) {
        dv[s] = s < n ? L.D(s) : T(0);
        ph[s] = s < n ? L.phys(s) : s;
        pos[s] = sorted ? 0 : ph[s];
    }
    if (sorted) {
#pragma unroll
        for (int s = 0; s < NM; ++s) {
#pragma unroll
            for (int t = s + 1; t < NM; ++t) {
                if (t < n) {
                    const bool lt = (dv[t] < dv[s]) || (dv[t] == dv[s] && ph[t] < ph[s]);
                    pos[s] += lt ? 1 : 0;
                    pos[t] += lt ? 0 : 1;
                }
            }
        }
    }
#pragma unroll
    for (int s = 0; s < NM; ++s)
        if (s < n)
            dout[pos[s]] = dv[s];
    if constexpr (WANTZ) {
        using Q_ = DynQ<T, NM>;
        const bool vec = q_vector_ok<T>(p.Q, n);
        for (int s = 0; s < n; ++s) {
            typename Q_::E x[Q_::NE];
            L.q.load(s, x);
            T col[Q_::NR];
#pragma unroll
            for (int j = 0; j < Q_::NE; ++j)
                El<T>::get(x[j], &col[j * Q_::RPE]);
            int ps = 0;
#pragma unroll
            for (int t = 0; t < NM; ++t)
                ps = (t == s) ? pos[t] : ps;
            T scale = T(1);
            if constexpr (LaneT::FASTQ)
                scale = L.sdl[s * tpb];  // Q = Qt diag(delta)
            if constexpr (LaneT::FASTQ) {
#pragma unroll
                for (int r = 0; r < Q_::NR; ++r)
                    col[r] *= scale;
            }
            store_col(qout + (long long)ps * n, col, n, vec);
        }
    }
    p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
}

template <typename T, int NM, bool WANTZ, int SCHED>
__global__ void dyn_kernel(KParams p)
{
    dyn_body<T, NM, WANTZ, SCHED>(p);
}

}  // namespace bstq
