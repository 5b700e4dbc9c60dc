// Lane-per-problem steqr kernel for sm_103a.
//
// One CUDA thread owns one tridiagonal problem of size n <= NM.  d and e live
// in registers and every access uses a compile-time index: the bulge chase is
// unrolled over the static positions NM-1 .. 1 and the warp skips positions
// outside the union of its lanes' active ranges.  Dynamic positions (the
// start of a sweep, the deflation point) only occur in the settle step and
// are resolved with bit masks and select chains.
//
// QR runs as QL on the mirrored block (BatchLAS page "perf_steqr", section
// "CTA STEQR: chase micro-structure decisions"; page "algo_steqr", QL on
// reversed local indices).  A block's direction depends only on its own
// entries when it is opened, and those are the input values, so each block
// that would run QR is reversed once while loading; every block then runs QL
// and Q starts from the permutation matrix of that reversal, which puts the
// rows of Q back in the caller's order.
//
// Schedulers (page "perf_steqr", section "Lockstep flat solver"):
//   NESTED: each lane loops settle -> chase on its own; lanes of a warp
//           diverge and realign only where their loops do.
//   FLAT:   the warp settles every lane (advance past deflated eigenvalues,
//           prepare a 2x2 solve or a sweep), then all lanes with work chase
//           together in one pass over the static positions.
// Both apply the same per-problem operations in the same order.
#pragma once

#include "bstq_numerics.cuh"

namespace bstq {

enum { QS_REG = 1, QS_SMEM = 2, QS_GLOBAL = 3 };
enum { SCHED_FLAT = 1, SCHED_NESTED = 2 };
enum { ST_RUN = 0, ST_DONE = 1, ST_FAIL = 2, ST_BAD = 3, ST_DEAD = 4 };
enum { TASK_NONE = 0, TASK_SWEEP = 1, TASK_2X2 = 2 };

constexpr unsigned FULL = 0xffffffffu;

struct KParams {
    void *d;           // batch x n, in/out
    const void *e;     // batch x (n-1)
    void *Q;           // batch x n x n (column-major per problem), out
    int *info;         // batch
    void *qwork;       // scratch for QS_GLOBAL: gridDim.x * NM * G * blockDim.x vectors
    long long batch;
    int n;
    int budget;        // sweep budget per problem (max_sweeps_per_n * n)
    int sort;          // 1: ascending output
};

// ---------------------------------------------------------------------------
// Q storage policies.  All rotate the column pair (C, C-1) with
//   q_C <- cs q_C + sn q_{C-1},  q_{C-1} <- -sn q_C + cs q_{C-1}
// which is Q <- Q G for the similarity G^T T G of the chase.
// ---------------------------------------------------------------------------

template <typename T, int NM, int QS>
struct QStore;

// Whole Q in registers: q[col][row].
template <typename T, int NM>
struct QStore<T, NM, QS_REG> {
    T q[NM][NM];

    __device__ __forceinline__ void setup(void *, int) {}
    __device__ __forceinline__ void init_col(int s, int row_of_one)
    {
#pragma unroll
        for (int k = 0; k < NM; ++k) {
            if (k == s) {
#pragma unroll
                for (int r = 0; r < NM; ++r)
                    q[k][r] = (r == row_of_one) ? T(1) : T(0);
            }
        }
    }
    __device__ __forceinline__ void begin(int) {}
    __device__ __forceinline__ void end(int) {}
    template <int C>
    __device__ __forceinline__ void rot(T cs, T sn)
    {
#pragma unroll
        for (int r = 0; r < NM; ++r) {
            T x = q[C][r], y = q[C - 1][r];
            q[C][r] = fma(cs, x, sn * y);
            q[C - 1][r] = fma(cs, y, -sn * x);
        }
    }
    // Column s (static s in an unrolled loop) into out[].
    __device__ __forceinline__ void get_col(int s, T (&out)[NM])
    {
#pragma unroll
        for (int k = 0; k < NM; ++k)
            if (k == s) {
#pragma unroll
                for (int r = 0; r < NM; ++r)
                    out[r] = q[k][r];
            }
    }
};

template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
    using V = float4;
    static constexpr int W = 4;
    __device__ static __forceinline__ void unpack(const V &v, float *x)
    {
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static __forceinline__ V pack(const float *x) { return make_float4(x[0], x[1], x[2], x[3]); }
};
template <>
struct Vec16<double> {
    using V = double2;
    static constexpr int W = 2;
    __device__ static __forceinline__ void unpack(const V &v, double *x)
    {
        x[0] = v.x; x[1] = v.y;
    }
    __device__ static __forceinline__ V pack(const double *x) { return make_double2(x[0], x[1]); }
};

// Q in memory (shared or global), streamed one column at a time: the column
// shared by two successive rotations of a sweep stays in registers (page
// "perf_steqr": streaming rotation apply).  Layout in 16-byte vectors,
// element (column k, row group g, thread t) at base[(k*G + g)*stride + t]:
// the lanes of a warp touch consecutive vectors whatever columns they are
// on, so shared-memory accesses are free of bank conflicts.
template <typename T, int NM>
struct QStream {
    using VT = Vec16<T>;
    using V = typename VT::V;
    static constexpr int W = VT::W;
    static constexpr int G = (NM + W - 1) / W;
    static constexpr int NR = G * W;
    V *base;
    int stride;
    T cur[NR];

    __device__ __forceinline__ void setup(void *p, int s)
    {
        base = reinterpret_cast<V *>(p);
        stride = s;
    }
    __device__ __forceinline__ void load(int k, T (&x)[NR]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            V v = base[(k * G + g) * stride];
            VT::unpack(v, &x[g * W]);
        }
    }
    __device__ __forceinline__ void store(int k, const T (&x)[NR]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g)
            base[(k * G + g) * stride] = VT::pack(&x[g * W]);
    }
    __device__ __forceinline__ void init_col(int s, int row_of_one)
    {
        T x[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r)
            x[r] = (r == row_of_one) ? T(1) : T(0);
        store(s, x);
    }
    __device__ __forceinline__ void begin(int hi) { load(hi, cur); }
    __device__ __forceinline__ void end(int lo) { store(lo, cur); }
    template <int C>
    __device__ __forceinline__ void rot(T cs, T sn)
    {
        T nx[NR];
        load(C - 1, nx);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            T x = cur[r], y = nx[r];
            cur[r] = fma(cs, x, sn * y);
            nx[r] = fma(cs, y, -sn * x);
        }
        store(C, cur);
#pragma unroll
        for (int r = 0; r < NR; ++r)
            cur[r] = nx[r];
    }
    __device__ __forceinline__ void get_col(int s, T (&out)[NM])
    {
        T x[NR];
        load(s, x);
#pragma unroll
        for (int r = 0; r < NM; ++r)
            out[r] = x[r];
    }
};

template <typename T, int NM>
struct QStore<T, NM, QS_SMEM> : QStream<T, NM> {};
template <typename T, int NM>
struct QStore<T, NM, QS_GLOBAL> : QStream<T, NM> {};

// Empty store for eigenvalues only.
template <typename T, int NM>
struct QNone {
    __device__ __forceinline__ void setup(void *, int) {}
    __device__ __forceinline__ void init_col(int, int) {}
    __device__ __forceinline__ void begin(int) {}
    __device__ __forceinline__ void end(int) {}
    template <int C>
    __device__ __forceinline__ void rot(T, T) {}
    __device__ __forceinline__ void get_col(int, T (&)[NM]) {}
};

// ---------------------------------------------------------------------------
// Register-array helpers for dynamic positions.
// ---------------------------------------------------------------------------
template <typename T, int NM>
__device__ __forceinline__ T pick(const T (&a)[NM], int i)
{
    T x = a[0];
#pragma unroll
    for (int k = 1; k < NM; ++k)
        x = (i == k) ? a[k] : x;
    return x;
}

template <typename T, int NM>
__device__ __forceinline__ void put(T (&a)[NM], int i, T v)
{
#pragma unroll
    for (int k = 0; k < NM; ++k)
        if (i == k)
            a[k] = v;
}

// First block [lb, le] containing storage index s, from the boundary mask
// (bit i set when e_i is an exact zero or i >= n-1).
__device__ __forceinline__ int block_lo(unsigned zmask, int s)
{
    unsigned below = s > 0 ? (zmask & ((1u << s) - 1u)) : 0u;
    return below ? (32 - __clz(below)) : 0;
}
__device__ __forceinline__ int block_hi(unsigned zmask, int s)
{
    return s + __ffs(zmask >> s) - 1;
}

// ---------------------------------------------------------------------------
// One problem.
// ---------------------------------------------------------------------------
template <typename T, int NM>
struct Lane {
    using C_ = Consts<T>;
    T d[NM], e[NM];
    int n, status, info;
    unsigned zmask;    // block boundaries (input exact zeros, i >= n-1)
    unsigned revmask;  // bit lb: block starting at lb was mirrored
    unsigned dmask;    // deflation test results over [lo, le)
    bool dvalid, inblock;
    int bnext, lb, le, lo;
    int iscale;
    T pre, sc, aeff, anorm;
    int jtot, budget;
    int task, m;
    T f, g;                    // running pair of the chase
    T lam_lo, lam_hi, cs2, sn2;  // pending 2x2 solve

    // Storage index s -> caller's index.
    __device__ __forceinline__ int phys(int s) const
    {
        int a = block_lo(zmask, s), b = block_hi(zmask, s);
        return ((revmask >> a) & 1u) ? (a + b - s) : s;
    }

    // Scale factors of a block with norm an (page "algo_steqr", scaling):
    // ssfmax/an when an > ssfmax, ssfmin/an when 0 < an < ssfmin (a
    // subnormal norm is first lifted by an exact power of two).
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
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            if (i >= a && i <= b)
                an = fmax(an, dabs(d[i]));
            if (i >= a && i < b)
                an = fmax(an, dabs(e[i]));
        }
        return an;
    }

    // Load problem `b`, mirroring every block that would run QR.
    __device__ void load(const KParams &p, long long b, bool live)
    {
        n = p.n;
        budget = p.budget;
        jtot = 0;
        task = TASK_NONE;
        inblock = false;
        dvalid = false;
        bnext = 0;
        lb = le = lo = m = 0;
        info = 0;
        revmask = 0;
        iscale = 0;
        pre = sc = aeff = anorm = T(1);
        f = g = lam_lo = lam_hi = cs2 = sn2 = T(0);
        if (!live) {
            status = ST_DEAD;
            zmask = ~0u;
#pragma unroll
            for (int i = 0; i < NM; ++i)
                d[i] = e[i] = T(0);
            return;
        }
        const T *dg = reinterpret_cast<const T *>(p.d) + b * n;
        const T *eg = reinterpret_cast<const T *>(p.e) + b * (n - 1);
        bool bad = false;
        zmask = 0;
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            d[i] = i < n ? dg[i] : T(0);
            e[i] = i < n - 1 ? eg[i] : T(0);
            bad |= !isfinite(d[i]) || !isfinite(e[i]);
            if (i >= n - 1 || e[i] == T(0))
                zmask |= 1u << i;
        }
        if (NM < 32)
            zmask |= ~0u << NM;
        status = bad ? ST_BAD : ST_RUN;
        if (bad)
            return;
        // Direction of every block, decided on the scaled end values exactly
        // as a QL/QR solver that scales first would decide it.
        for (int a = 0; a < n;) {
            int z = block_hi(zmask, a);
            if (z > a) {
                T an = block_norm(a, z);
                if (an > T(0)) {
                    int isc;
                    T pr, s, ae;
                    scale_factors(an, isc, pr, s, ae);
                    T x = pick(d, a), y = pick(d, z);
                    if (isc) {
                        x = (x * pr) * s;
                        y = (y * pr) * s;
                    }
                    if (dabs(x) > dabs(y))
                        revmask |= 1u << a;
                }
            }
            a = z + 1;
        }
        if (revmask) {
#pragma unroll
            for (int s = 0; s < NM; ++s) {
                if (s < n) {
                    int ps = phys(s);
                    d[s] = dg[ps];
                    if (s < n - 1 && !((zmask >> s) & 1u)) {
                        int pn = phys(s + 1);
                        e[s] = eg[ps < pn ? ps : pn];
                    }
                }
            }
        }
    }

    __device__ __forceinline__ void scale_block(T f1, T f2)
    {
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            if (i >= lb && i <= le)
                d[i] = (d[i] * f1) * f2;
            if (i >= lb && i < le)
                e[i] = (e[i] * f1) * f2;
        }
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
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            if (i >= lb && i <= le)
                d[i] = (d[i] * us) * up;
            if (with_e && i >= lb && i < le)
                e[i] = (e[i] * us) * up;
        }
    }

    __device__ __forceinline__ void close_block()
    {
        unscale_block(false);
        inblock = false;
    }

    // Relative deflation test (page "algo_steqr"):
    // |e_i|^2 <= eps^2 |d_i| |d_{i+1}| + safmin, for i in [lo, le).
    __device__ __forceinline__ unsigned deflation_mask() const
    {
        unsigned mk = 0;
#pragma unroll
        for (int i = 0; i < NM - 1; ++i) {
            if (i >= lo && i < le) {
                T ae = dabs(e[i]);
                T tst = ae * ae;
                T thr = fma(C_::eps2 * dabs(d[i]), dabs(d[i + 1]), C_::safmin);
                if (tst <= thr)
                    mk |= 1u << i;
            }
        }
        return mk;
    }

    // One settle event.  Returns true while the lane has no chase task and is
    // still running.
    __device__ bool settle_step()
    {
        if (!inblock) {
            if (bnext >= n) {
                status = ST_DONE;
                return false;
            }
            lb = bnext;
            le = block_hi(zmask, lb);
            bnext = le + 1;
            if (le == lb)
                return true;  // 1x1 block: final
            anorm = block_norm(lb, le);
            if (anorm == T(0))
                return true;  // zero block: final
            scale_factors(anorm, iscale, pre, sc, aeff);
            if (iscale)
                scale_block(pre, sc);
            lo = lb;
            inblock = true;
            dvalid = false;
        }
        if (!dvalid) {
            dmask = deflation_mask();
            dvalid = true;
        }
        int mm = __ffs((dmask & (~0u << lo)) | (1u << le)) - 1;
        if (mm < le)
            put(e, mm, T(0));
        if (mm == lo) {  // eigenvalue at lo has converged
            ++lo;
            if (lo > le)
                close_block();
            return true;
        }
        if (mm == lo + 1) {  // 2x2 direct solve, executed in the next pass
            T a = pick(d, lo), bb = pick(e, lo), c2 = pick(d, lo + 1);
            solve2x2(a, bb, c2, lam_lo, lam_hi, cs2, sn2);
            task = TASK_2X2;
            m = lo + 1;
            return false;
        }
        if (jtot == budget) {  // sweep budget exhausted
            unscale_block(true);
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < NM - 1; ++i)
                if (i < n - 1 && e[i] != T(0))
                    ++cnt;
            info = cnt;
            status = ST_FAIL;
            return false;
        }
        ++jtot;
        T d1 = pick(d, lo), d2 = pick(d, lo + 1), e1 = pick(e, lo);
        T mu = wilkinson_shift(d1, d2, e1);
        f = pick(d, mm) - mu;
        g = pick(e, mm - 1);
        m = mm;
        task = TASK_SWEEP;
        return false;
    }

    __device__ __forceinline__ int task_hi() const { return m; }
    __device__ __forceinline__ int task_lo() const { return lo + 1; }

    // Rotation on the pair (C, C-1) of the current task, if C is in its range.
    template <int C, class QS>
    __device__ __forceinline__ void chase_at(QS &Q)
    {
        if (task == TASK_SWEEP && C <= m && C > lo) {
            T cs, sn, r;
            lartg(f, g, cs, sn, r);
            T a = d[C], b = e[C - 1], cc = d[C - 1];
            // T+ = G^T T G on rows/columns (C, C-1) (page "algo_steqr", EXP)
            T p1 = fma(cs, a, sn * b);
            T p2 = fma(cs, b, sn * cc);
            T dn = fma(cs, p1, sn * p2);
            T en = fma(cs, p2, -sn * p1);
            d[C] = dn;
            d[C - 1] = (a + cc) - dn;
            e[C - 1] = en;
            if (C < m)
                e[C] = r;
            if constexpr (C >= 2) {
                if (C - 1 > lo) {
                    T eo = e[C - 2];
                    g = sn * eo;  // new bulge
                    e[C - 2] = cs * eo;
                    f = en;
                }
            }
            Q.template rot<C>(cs, sn);
        } else if (task == TASK_2X2 && C == lo + 1) {
            d[C - 1] = lam_lo;
            d[C] = lam_hi;
            e[C - 1] = T(0);
            Q.template rot<C>(cs2, sn2);
        }
    }

    __device__ __forceinline__ void post_pass()
    {
        if (task == TASK_2X2) {
            lo += 2;
            if (lo > le)
                close_block();
        }
        task = TASK_NONE;
        dvalid = false;
    }
};

// ---------------------------------------------------------------------------
// Kernel.
// ---------------------------------------------------------------------------
template <typename T, int NM, bool WANTZ, int QS>
struct QFor {
    using type = QStore<T, NM, QS>;
};
template <typename T, int NM, int QS>
struct QFor<T, NM, false, QS> {
    using type = QNone<T, NM>;
};

// Compile-time loop over the chase positions C = top, top-1, ..., 1; the
// warp (or, nested, the lane) skips positions outside [rlo, rhi].
template <int C>
struct ChaseLoop {
    template <class LaneT, class QT>
    __device__ static __forceinline__ void run(LaneT &L, QT &Q, int rhi, int rlo)
    {
        if (!(C > rhi || C < rlo))
            L.template chase_at<C>(Q);
        ChaseLoop<C - 1>::run(L, Q, rhi, rlo);
    }
};
template <>
struct ChaseLoop<0> {
    template <class LaneT, class QT>
    __device__ static __forceinline__ void run(LaneT &, QT &, int, int) {}
};

template <int NM, class LaneT, class QT>
__device__ __forceinline__ void chase_pass(LaneT &L, QT &Q, int rhi, int rlo)
{
    ChaseLoop<NM - 1>::run(L, Q, rhi, rlo);
}

template <typename T, int NM, bool WANTZ, int QS, int SCHED>
__global__ void lane_kernel(KParams p)
{
    extern __shared__ uint4 smem_raw[];
    using QT = typename QFor<T, NM, WANTZ, QS>::type;
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = b < p.batch;

    Lane<T, NM> L;
    L.load(p, b, live);
    QT Q;
    if (WANTZ) {
        if (QS == QS_SMEM) {
            Q.setup(reinterpret_cast<char *>(smem_raw) + 16 * threadIdx.x, blockDim.x);
        } else if (QS == QS_GLOBAL) {
            constexpr int G = (NM * (int)sizeof(T) + 15) / 16;
            char *base = reinterpret_cast<char *>(p.qwork) +
                         16ll * ((long long)blockIdx.x * NM * G * blockDim.x + threadIdx.x);
            Q.setup(base, blockDim.x);
        }
        if (L.status == ST_RUN) {
#pragma unroll
            for (int s = 0; s < NM; ++s)
                Q.init_col(s, s < L.n ? L.phys(s) : s);
        }
    }

    if (SCHED == SCHED_FLAT) {
        for (;;) {
            bool need = (L.status == ST_RUN) && (L.task == TASK_NONE);
            while (__any_sync(FULL, need)) {
                if (need)
                    need = L.settle_step();
            }
            const bool has = (L.status == ST_RUN) && (L.task != TASK_NONE);
            if (!__any_sync(FULL, has))
                break;
            const int rhi = __reduce_max_sync(FULL, has ? L.task_hi() : -1);
            const int rlo = __reduce_min_sync(FULL, has ? L.task_lo() : NM);
            if (has)
                Q.begin(L.task_hi());
            chase_pass<NM>(L, Q, rhi, rlo);
            if (has) {
                Q.end(L.task_lo() - 1);
                L.post_pass();
            }
        }
    } else {
        while (L.status == ST_RUN) {
            if (L.task == TASK_NONE) {
                L.settle_step();
                continue;
            }
            const int rhi = L.task_hi(), rlo = L.task_lo();
            Q.begin(rhi);
            chase_pass<NM>(L, Q, rhi, rlo);
            Q.end(rlo - 1);
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
    // Output position of each storage index: its rank in ascending order
    // (equal values keep the caller's order), or the caller's index when the
    // output stays unsorted.
    const bool sorted = p.sort && L.status == ST_DONE;
    int ph[NM], pos[NM];
#pragma unroll
    for (int s = 0; s < NM; ++s) {
        ph[s] = s < n ? L.phys(s) : s;
        pos[s] = sorted ? 0 : ph[s];
    }
    if (sorted) {
#pragma unroll
        for (int s = 0; s < NM; ++s) {
#pragma unroll
            for (int t = s + 1; t < NM; ++t) {
                if (t < n) {
                    const bool lt = (L.d[t] < L.d[s]) || (L.d[t] == L.d[s] && ph[t] < ph[s]);
                    pos[s] += lt ? 1 : 0;
                    pos[t] += lt ? 0 : 1;
                }
            }
        }
    }
#pragma unroll
    for (int s = 0; s < NM; ++s)
        if (s < n)
            dout[pos[s]] = L.d[s];
    if (WANTZ) {
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            if (s < n) {
                T col[NM];
                Q.get_col(s, col);
                T *qc = qout + (long long)pos[s] * n;
#pragma unroll
                for (int r = 0; r < NM; ++r)
                    if (r < n)
                        qc[r] = col[r];
            }
        }
    }
    p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
}

}  // namespace bstq
