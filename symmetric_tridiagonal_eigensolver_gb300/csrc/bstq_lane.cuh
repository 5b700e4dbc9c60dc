// Lane-per-problem steqr kernel for sm_103a.
//
// One CUDA thread owns one tridiagonal problem of size n <= NM.  d and e live
// in registers and every access uses a compile-time index: a sweep is a pass
// over the static chase positions C = NM-1 .. 1, entered through a jump table
// at the group top at or above the warp's highest active position and left
// at a group boundary once no lane has work below.  Each position is
// straight-line code: lanes for which the position is outside their sweep
// apply the identity rotation (lartg of (1, 0)) and keep d and e through
// selects, so each group of positions is one basic block in which the
// eigenvector update of one position overlaps the dependency chain of the
// next.  Dynamic positions (start of a sweep, deflation point)
// only occur in the settle step and are resolved with bit masks and selects.
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

enum { QS_REG = 1, QS_SMEM = 2, QS_GLOBAL = 3, QS_HYBRID = 4, QS_SPLIT = 5, QS_LOG = 6 };
enum { SCHED_FLAT = 1, SCHED_NESTED = 2 };
enum { ST_RUN = 0, ST_DONE = 1, ST_FAIL = 2, ST_BAD = 3, ST_DEAD = 4 };
enum { TASK_NONE = 0, TASK_SWEEP = 1, TASK_2X2 = 2 };

constexpr unsigned FULL = 0xffffffffu;
constexpr int kHybridRegRows = 8;

struct KParams {
    void *d;           // batch x n, in/out
    const void *e;     // batch x (n-1)
    void *Q;           // batch x n x n (column-major per problem), out
    int *info;         // batch
    void *qwork;       // scratch for QS_GLOBAL
    long long batch;
    int n;
    int budget;        // sweep budget per problem (max_sweeps_per_n * n)
    int sort;          // 1: ascending output
    int ppb;           // problems per block (split-role kernel)
    int back;          // 1: Q holds the basis Z on entry (back_transform);
                       // 2: the basis is the fused syev's, in sscr
    int scheme;        // 0 EXP, 1 PG update (dynamic-position kernels)
    const void *A;     // fused syev: dense input, batch x n x n
    void *sscr;        // fused syev: the reduction's scratch
    long long lcap;    // record-and-apply kernels: rotation log entries per problem,
    int *lcnt;         // per problem log length (or a state code),
    unsigned char *lmap;  // per problem column maps (2 n bytes)
};

// ---------------------------------------------------------------------------
// Element arithmetic of the eigenvector update.  float rows are processed in
// packed pairs (one f32x2 instruction updates two rows), double rows singly.
// Every policy rotates the column pair (C, C-1) as
//   q_C <- cs q_C + sn q_{C-1},  q_{C-1} <- -sn q_C + cs q_{C-1}
// which is Q <- Q G for the similarity G^T T G of the chase.
// ---------------------------------------------------------------------------
template <typename T>
struct El;

template <>
struct El<float> {
    using E = uint64_t;  // two consecutive rows
    static constexpr int RPE = 2;
    struct R {
        uint64_t c, s, ns;
    };
    __device__ static __forceinline__ R make(float cs, float sn) { return {pk2(cs, cs), pk2(sn, sn), pk2(-sn, -sn)}; }
    __device__ static __forceinline__ void rot(E &x, E &y, const R &r)
    {
        const E xo = x;
        x = fma2(r.c, x, mul2(r.s, y));
        y = fma2(r.c, y, mul2(r.ns, xo));
    }
    __device__ static __forceinline__ E unit(int row, int base)
    {
        return pk2(row == base ? 1.0f : 0.0f, row == base + 1 ? 1.0f : 0.0f);
    }
    __device__ static __forceinline__ void get(E v, float *out) { upk2(v, out[0], out[1]); }
    __device__ static __forceinline__ E pack(const float *in) { return pk2(in[0], in[1]); }
};

template <>
struct El<double> {
    using E = double;
    static constexpr int RPE = 1;
    struct R {
        double c, s, ns;
    };
    __device__ static __forceinline__ R make(double cs, double sn) { return {cs, sn, -sn}; }
    __device__ static __forceinline__ void rot(E &x, E &y, const R &r)
    {
        const E xo = x;
        x = fma(r.c, x, r.s * y);
        y = fma(r.c, y, r.ns * xo);
    }
    __device__ static __forceinline__ E unit(int row, int base) { return row == base ? 1.0 : 0.0; }
    __device__ static __forceinline__ void get(E v, double *out) { out[0] = v; }
    __device__ static __forceinline__ E pack(const double *in) { return in[0]; }
};

// One column of Q (rows 0 .. n-1) to global memory at qc.  With vec set the
// column is written in 16-byte vectors: a lane owns a whole problem, so the
// 32 lanes of a warp store to 32 places far apart, and each store
// instruction costs the memory pipeline one request per lane whatever its
// width; 16-byte stores take a quarter of the requests of 4-byte ones (for
// float).  vec requires n * sizeof(T) to be a multiple of 16 and Q to start
// on a 16-byte boundary, so that every column does (q_vector_ok).
template <typename T, int R>
__device__ __forceinline__ void store_col(T *qc, const T (&col)[R], int n, bool vec)
{
    constexpr int W = 16 / (int)sizeof(T);
    if (vec) {
        struct alignas(16) V {
            T x[W];
        };
#pragma unroll
        for (int v = 0; v < R / W; ++v) {
            if (v * W < n) {
                V o;
#pragma unroll
                for (int k = 0; k < W; ++k)
                    o.x[k] = col[v * W + k];
                reinterpret_cast<V *>(qc)[v] = o;
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (r < n)
                qc[r] = col[r];
    }
}

// One column of the caller's basis Z (rows 0 .. n-1) from global memory into
// col[]; rows n .. R-1 are zero.  vec as for store_col.
template <typename T, int R>
__device__ __forceinline__ void load_col(const T *zc, T (&col)[R], int n, bool vec)
{
    constexpr int W = 16 / (int)sizeof(T);
    if (vec) {
        struct alignas(16) V {
            T x[W];
        };
#pragma unroll
        for (int v = 0; v < R / W; ++v) {
            V o;
            if (v * W < n)
                o = reinterpret_cast<const V *>(zc)[v];
#pragma unroll
            for (int k = 0; k < W; ++k)
                col[v * W + k] = v * W < n ? o.x[k] : T(0);
        }
#pragma unroll
        for (int r = (R / W) * W; r < R; ++r)
            col[r] = T(0);
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
            col[r] = r < n ? zc[r] : T(0);
    }
}

template <typename T>
__device__ __forceinline__ bool q_vector_ok(const void *Q, int n)
{
    return ((n * (int)sizeof(T)) % 16) == 0 && ((reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
}

// Q with rows [0, RR) in registers and rows [RR, RR + MR) in memory (shared
// or global), streamed one column at a time: the column shared by two
// successive rotations of a sweep stays in registers (page "perf_steqr":
// streaming rotation apply).  Memory layout in 16-byte vectors, vector g of
// column k of thread t at base[(k*G + g)*stride + t]: the lanes of a warp
// touch consecutive vectors whatever column they are on, so shared memory is
// accessed without bank conflicts and global memory is coalesced.  (A
// lane-major layout with an odd lane pitch, whose addresses are compile-time
// offsets, measured slower for the hybrid store.)  Loads are unconditional
// (every lane's region holds finite values).
// ST > 0 fixes the stride (in vectors) at compile time: the compiler then
// knows that the column a position loads is not the one the previous
// position stored, and can issue the load ahead of the store.
template <typename T, int NM, int RR, int MR, int ST = 0>
struct QMix {
    using Tr = El<T>;
    using E = typename Tr::E;
    static constexpr int RPE = Tr::RPE;
    static constexpr int NER = RR / RPE;  // register elements per column
    static constexpr int NEM = MR / RPE;  // memory elements per column
    static constexpr int G = NEM / 2;     // 16-byte vectors per column
    static_assert(RR % RPE == 0 && NEM % 2 == 0, "row split must match the vector width");
    struct V16 {
        E a, b;
    };

    E qr[NM][NER > 0 ? NER : 1];
    E cur[NEM > 0 ? NEM : 1];
    V16 *base;
    int stride;

    // bytes of the memory rows per thread
    static constexpr int MEM_BYTES = NM * G * 16;

    __device__ __forceinline__ void setup(void *p, int s)
    {
        base = reinterpret_cast<V16 *>(p);
        stride = s;
    }
    __device__ __forceinline__ int vidx(int k, int g) const { return (k * G + g) * (ST > 0 ? ST : stride); }
    __device__ __forceinline__ void load(int k, E (&x)[NEM > 0 ? NEM : 1]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const V16 v = base[vidx(k, g)];
            x[2 * g] = v.a;
            x[2 * g + 1] = v.b;
        }
    }
    __device__ __forceinline__ void store(int k, const E (&x)[NEM > 0 ? NEM : 1]) const
    {
#pragma unroll
        for (int g = 0; g < G; ++g)
            base[vidx(k, g)] = V16{x[2 * g], x[2 * g + 1]};
    }
    __device__ __forceinline__ void init_col(int s, int row_of_one)
    {
#pragma unroll
        for (int k = 0; k < NM; ++k)
            if (k == s) {
#pragma unroll
                for (int j = 0; j < NER; ++j)
                    qr[k][j] = Tr::unit(row_of_one, j * RPE);
            }
        if constexpr (NEM > 0) {
            E x[NEM];
#pragma unroll
            for (int j = 0; j < NEM; ++j)
                x[j] = Tr::unit(row_of_one, RR + j * RPE);
            store(s, x);
        }
    }
    // Column s (static s in an unrolled loop) from the caller's basis:
    // rows 0 .. n-1 of zc, zero below (back_transform).
    __device__ __forceinline__ void init_col_from(int s, const T *zc, int n, bool vec)
    {
        T col[RR + MR];
        load_col(zc, col, n, vec);
#pragma unroll
        for (int k = 0; k < NM; ++k)
            if (k == s) {
#pragma unroll
                for (int j = 0; j < NER; ++j)
                    qr[k][j] = Tr::pack(&col[j * RPE]);
            }
        if constexpr (NEM > 0) {
            E x[NEM];
#pragma unroll
            for (int j = 0; j < NEM; ++j)
                x[j] = Tr::pack(&col[RR + j * RPE]);
            store(s, x);
        }
    }
    __device__ __forceinline__ void begin(int hi)
    {
        if constexpr (NEM > 0)
            load(hi, cur);
    }
    __device__ __forceinline__ void end(int col, bool st)
    {
        if constexpr (NEM > 0)
            if (st)
                store(col, cur);
    }
    // The streamed column is written back unconditionally: a lane for which
    // the position is inactive rotates by the identity and stores the values
    // it loaded (up to the sign of a zero), and a predicated store would
    // split the position's straight-line code.
    template <int C>
    __device__ __forceinline__ void rot(T cs, T sn, bool)
    {
        const typename Tr::R r = Tr::make(cs, sn);
#pragma unroll
        for (int j = 0; j < NER; ++j)
            Tr::rot(qr[C][j], qr[C - 1][j], r);
        if constexpr (NEM > 0) {
            E nx[NEM];
            load(C - 1, nx);
#pragma unroll
            for (int j = 0; j < NEM; ++j)
                Tr::rot(cur[j], nx[j], r);
            store(C, cur);
#pragma unroll
            for (int j = 0; j < NEM; ++j)
                cur[j] = nx[j];
        }
    }
    // Column s (static s in an unrolled loop), all stored rows, into out[].
    __device__ __forceinline__ void get_col(int s, T (&out)[RR + MR])
    {
#pragma unroll
        for (int k = 0; k < NM; ++k)
            if (k == s) {
#pragma unroll
                for (int j = 0; j < NER; ++j)
                    Tr::get(qr[k][j], &out[j * RPE]);
            }
        if constexpr (NEM > 0) {
            E x[NEM];
            load(s, x);
#pragma unroll
            for (int j = 0; j < NEM; ++j)
                Tr::get(x[j], &out[RR + j * RPE]);
        }
    }
};

// Empty store for eigenvalues only.
template <typename T, int NM>
struct QNone {
    static constexpr int MEM_BYTES = 0;
    __device__ __forceinline__ void setup(void *, int) {}
    __device__ __forceinline__ void init_col(int, int) {}
    __device__ __forceinline__ void begin(int) {}
    __device__ __forceinline__ void end(int, bool) {}
    template <int C>
    __device__ __forceinline__ void rot(T, T, bool) {}
};

// Row split per storage policy.  Memory rows are padded to whole 16-byte
// vectors; padding rows stay zero.
template <typename T, int NM, int QS>
struct QLayout {
    static constexpr int W = 16 / (int)sizeof(T);
    static constexpr int RR = QS == QS_REG ? NM : (QS == QS_HYBRID ? kHybridRegRows : 0);
    static constexpr int MR = QS == QS_REG ? 0 : ((NM - RR + W - 1) / W) * W;
    using type = QMix<T, NM, RR, MR>;
    static constexpr int ROWS = RR + MR;
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
        a[k] = (i == k) ? v : a[k];
}

// Block [lb, le] containing storage index s, from the boundary mask (bit i
// set when e_i is an exact zero or i >= n-1).
__device__ __forceinline__ int block_lo(unsigned zmask, int s)
{
    unsigned below = s > 0 ? (zmask & ((1u << s) - 1u)) : 0u;
    return below ? (32 - __clz(below)) : 0;
}
__device__ __forceinline__ int block_hi(unsigned zmask, int s)
{
    return s + __ffs(zmask >> s) - 1;
}
// 64-bit forms for problems with more than 32 entries (dynamic kernels).
__device__ __forceinline__ int block_lo(unsigned long long zmask, int s)
{
    unsigned long long below = s > 0 ? (zmask & ((1ull << s) - 1ull)) : 0ull;
    return below ? (64 - __clzll((long long)below)) : 0;
}
__device__ __forceinline__ int block_hi(unsigned long long zmask, int s)
{
    return s + __ffsll((long long)(zmask >> s)) - 1;
}

// ---------------------------------------------------------------------------
// Pass entry.  A pass is left only at group boundaries (after positions
// C with (C - 1) % KEXIT == 0) and entered only at group tops (multiples of
// KEXIT, or NM - 1), so each group of KEXIT positions is a single basic
// block and the compiler can overlap the eigenvector update of one position
// with the dependency chain of the next.  Entering above the warp's highest
// active position costs a few identity rotations; for a block that reaches
// the end of the problem the highest position is NM - 1, already a top.
// ---------------------------------------------------------------------------
template <int NM, int KEXIT>
__device__ __forceinline__ int group_top(int rhi)
{
    const int t = (rhi + KEXIT - 1) / KEXIT * KEXIT;
    return t < NM - 1 ? t : NM - 1;
}
// switch value of a group top: NM - 1 enters at the head of the list
template <int NM>
__device__ __forceinline__ int group_case(int top)
{
    return top == NM - 1 ? 32 : top;
}

// Positions 31 .. 1 with case labels at the group tops only; S(C) expands
// to the (compile-time guarded) code of position C.
#define BSTQ_CASES_K4(S)                                                      \
    case 32:                                                                  \
        S(31) S(30) S(29)                                                     \
    case 28:                                                                  \
        S(28) S(27) S(26) S(25)                                               \
    case 24:                                                                  \
        S(24) S(23) S(22) S(21)                                               \
    case 20:                                                                  \
        S(20) S(19) S(18) S(17)                                               \
    case 16:                                                                  \
        S(16) S(15) S(14) S(13)                                               \
    case 12:                                                                  \
        S(12) S(11) S(10) S(9)                                                \
    case 8:                                                                   \
        S(8) S(7) S(6) S(5)                                                   \
    case 4:                                                                   \
        S(4) S(3) S(2) S(1)
#define BSTQ_CASES_K2(S)                                                      \
    case 32:                                                                  \
        S(31)                                                                 \
    case 30:                                                                  \
        S(30) S(29)                                                           \
    case 28:                                                                  \
        S(28) S(27)                                                           \
    case 26:                                                                  \
        S(26) S(25)                                                           \
    case 24:                                                                  \
        S(24) S(23)                                                           \
    case 22:                                                                  \
        S(22) S(21)                                                           \
    case 20:                                                                  \
        S(20) S(19)                                                           \
    case 18:                                                                  \
        S(18) S(17)                                                           \
    case 16:                                                                  \
        S(16) S(15)                                                           \
    case 14:                                                                  \
        S(14) S(13)                                                           \
    case 12:                                                                  \
        S(12) S(11)                                                           \
    case 10:                                                                  \
        S(10) S(9)                                                            \
    case 8:                                                                   \
        S(8) S(7)                                                             \
    case 6:                                                                   \
        S(6) S(5)                                                             \
    case 4:                                                                   \
        S(4) S(3)                                                             \
    case 2:                                                                   \
        S(2) S(1)
#define BSTQ_CASES_K8(S)                                                      \
    case 32:                                                                  \
        S(31) S(30) S(29) S(28) S(27) S(26) S(25)                             \
    case 24:                                                                  \
        S(24) S(23) S(22) S(21) S(20) S(19) S(18) S(17)                       \
    case 16:                                                                  \
        S(16) S(15) S(14) S(13) S(12) S(11) S(10) S(9)                        \
    case 8:                                                                   \
        S(8) S(7) S(6) S(5) S(4) S(3) S(2) S(1)
#define BSTQ_GROUPED_SWITCH(KX, SW, S)                                        \
    static_assert(KX == 2 || KX == 4 || KX == 8, "group size 2, 4 or 8");     \
    if constexpr (KX == 8) {                                                  \
        switch (SW) {                                                         \
            BSTQ_CASES_K8(S)                                                  \
        default:                                                              \
            break;                                                            \
        }                                                                     \
    } else if constexpr (KX == 4) {                                           \
        switch (SW) {                                                         \
            BSTQ_CASES_K4(S)                                                  \
        default:                                                              \
            break;                                                            \
        }                                                                     \
    } else {                                                                  \
        switch (SW) {                                                         \
            BSTQ_CASES_K2(S)                                                  \
        default:                                                              \
            break;                                                            \
        }                                                                     \
    }

// ---------------------------------------------------------------------------
// One problem.
// ---------------------------------------------------------------------------
template <typename T, int NM, int KEXIT>
struct Lane {
    using C_ = Consts<T>;
    T d[NM], e[NM];
    int n, status, info;
    unsigned zmask;    // block boundaries (input exact zeros, i >= n-1)
    unsigned revmask;  // bit lb: block starting at lb was mirrored
    unsigned tmask;    // deflation test result of every e_i, for the current values
    bool inblock;
    int bnext, lb, le, lo;
    int iscale;
    T pre, sc, aeff, anorm;
    int jtot, budget;
    int task, m;
    T f, g;        // running pair of the chase
    T rpend;       // r of the previous position, not yet stored (float)
    T f0, g0;      // seed of the current sweep, (d_m - mu, e_{m-1})
    T cs2, sn2;    // rotation of a pending 2x2 solve
    unsigned zeroed;  // off-diagonals set to zero by the deflation test
    // current pass: positions [lo_l, hi_l] are this lane's (hi_l < 0: none),
    // and the same as bit masks over C: in range, sweep rotation, 2x2
    // rotation, first rotation, "e_C <- r", columns this lane changes
    int hi_l, lo_l;
    unsigned m_in, m_act, m_22, m_first, m_er, m_touch;
    // shared-memory mirror of d and e for the settle step's dynamic reads,
    // per warp [entry][lane]: entry i of d at mir[i * 32], of e at
    // mir[(NM + i) * 32], mir = warp region + lane.  Static entries are
    // compile-time offsets from the lane's base, and dynamic reads hit one
    // bank per lane whatever entry each lane reads.
    static constexpr int MIRROR_WARP_ELEMS = 2 * NM * 32;
    T *mir;

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
        tmask = 0;
        bnext = 0;
        lb = le = lo = m = 0;
        info = 0;
        revmask = 0;
        iscale = 0;
        pre = sc = aeff = anorm = T(1);
        f = g = f0 = g0 = cs2 = sn2 = rpend = T(0);
        zeroed = 0;
        clear_pass();
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
    // |e_i|^2 <= eps^2 |d_i| |d_{i+1}| + safmin.
    __device__ __forceinline__ static bool negligible(T ei, T di, T dn)
    {
        const T ae = dabs(ei);
        const T tst = ae * ae;
        const T thr = fma(C_::eps2 * dabs(di), dabs(dn), C_::safmin);
        if constexpr (sizeof(T) == 8)  // non-negative doubles order as their bits
            return __double_as_longlong(tst) <= __double_as_longlong(thr);
        else
            return tst <= thr;
    }

    // Entry i's values are final for this pass: copy d_i and e_i to the
    // mirror and record the deflation test of e_i.  The chase calls this for
    // each position once that position's values are final, and for the two
    // entries below the last position when the pass ends, so the settle step
    // finds the mirror and the test bits of every entry current without
    // recomputing them.
    template <int I>
    __device__ __forceinline__ void settle_entry()
    {
        if constexpr (I >= 0 && I <= NM - 1) {
            mir[I * 32] = d[I];
            mir[(NM + I) * 32] = e[I];
            if constexpr (I <= NM - 2) {
                const bool ng = negligible(e[I], d[I], d[I + 1]);
                tmask = ng ? (tmask | (1u << I)) : (tmask & ~(1u << I));
            }
        }
    }

    // Every entry (after loading or scaling a block, and after a nested pass).
    __device__ __forceinline__ void refresh_all()
    {
        unsigned mk = 0;
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            mir[i * 32] = d[i];
            mir[(NM + i) * 32] = e[i];
        }
#pragma unroll
        for (int i = 0; i < NM - 1; ++i)
            mk |= negligible(e[i], d[i], d[i + 1]) ? (1u << i) : 0u;
        tmask = mk;
    }

    __device__ __forceinline__ T mir_d(int i) const { return mir[i * 32]; }
    __device__ __forceinline__ T mir_e(int i) const { return mir[(NM + i) * 32]; }

    // Settle the lane: advance past converged eigenvalues and blocks until
    // the lane has a task (2x2 solve or sweep), is done, or has exhausted
    // its sweep budget.  Consecutive deflations are handled in one call, so
    // a lockstep warp computes the shifts of all its lanes together.
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
                    continue;  // 1x1 block: final
                anorm = block_norm(lb, le);
                if (anorm == T(0))
                    continue;  // zero block: final
                scale_factors(anorm, iscale, pre, sc, aeff);
                if (iscale)
                    scale_block(pre, sc);
                lo = lb;
                inblock = true;
                refresh_all();
            }
            // negligible off-diagonals of the active range [lo, le); one
            // found negligible earlier counts as the exact zero it was set to
            unsigned dmask = (tmask | zeroed) & ((1u << le) - 1u) & (~0u << lo);
            // Eigenvalues lo, lo+1, ... have converged while e_lo, e_lo+1,
            // ... are negligible: skip that run of set bits in one step (bit
            // le stands for the block end; a run through it closes the
            // block).  Every negligible e_i passed over, and the first one
            // after the run, is set to zero.
            const unsigned long long x = (unsigned long long)(dmask | (1u << le)) >> lo;
            const int run = __ffsll((long long)~x) - 1;
            const unsigned below_le = (1u << le) - 1u;
            zeroed |= (unsigned)((((1ull << run) - 1ull) << lo)) & below_le;
            lo += run;
            if (lo > le) {
                close_block();
                continue;
            }
            dmask &= ~0u << lo;
            mm = __ffs(dmask | (1u << le)) - 1;  // > lo
            if (mm < le)
                zeroed |= 1u << mm;  // e_mm <- 0
            break;
        }
        // Shift and 2x2 rotation from one evaluation, without branches: the
        // lanes of a warp settling together need not split by task.
        const T d1 = mir_d(lo), d2 = mir_d(lo + 1), e1 = mir_e(lo);
        const T dm = mir_d(mm), gm = mir_e(mm - 1);
        T t, mu;
        shift_tangent(d1, d2, e1, t, mu);
        if constexpr (sizeof(T) == 8)
            rot_from_tangent(t, cs2, sn2);  // used by a 2x2 solve only
        const bool two = mm == lo + 1;  // 2x2 direct solve, applied in the next pass
        if (!two && jtot == budget) {  // sweep budget exhausted
            unscale_block(true);
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < NM - 1; ++i)
                if (i < n - 1 && e[i] != T(0) && !((zeroed >> i) & 1u))
                    ++cnt;
            info = cnt;
            status = ST_FAIL;
            return;
        }
        jtot += two ? 0 : 1;
        f0 = dm - mu;
        g0 = gm;
        if constexpr (sizeof(T) == 4) {
            // float: the 2x2 solve runs as a one-position sweep seeded with
            // the direction (1, t) of its rotation: lartg(1, t) is
            // (1, t) / sqrt(1 + t^2), the rotation with tangent t, so the
            // chase needs no separate 2x2 path and the settle step no
            // second square root; e_lo is set to zero through the mask when
            // the pass is done (post_pass)
            f0 = two ? T(1) : f0;
            g0 = two ? t : g0;
        }
        m = mm;
        task = two ? TASK_2X2 : TASK_SWEEP;
    }

    __device__ __forceinline__ bool has_task() const { return status == ST_RUN && task != TASK_NONE; }

    __device__ __forceinline__ void clear_pass()
    {
        hi_l = -1;
        lo_l = NM;
        m_in = m_act = m_22 = m_first = m_er = m_touch = 0u;
    }

    __device__ __forceinline__ void prepare_pass()
    {
        if (!has_task()) {
            clear_pass();
            return;
        }
        hi_l = m;
        lo_l = lo + 1;
        const unsigned upto = hi_l >= 31 ? ~0u : ((2u << hi_l) - 1u);  // bits 0..hi_l
        m_in = upto & (~0u << lo_l);
        m_touch = upto & (~0u << lo);
        if (task == TASK_2X2 && sizeof(T) == 8) {
            m_act = 0u;
            m_22 = m_in;
            m_first = 0u;
        } else {
            m_act = m_in;
            m_22 = 0u;
            m_first = 1u << hi_l;
        }
        m_er = m_act & ~(1u << hi_l);
    }

    // Position C of a pass: rotation on the pair (C, C-1) for lanes whose
    // task covers C, identity (lartg of (1, 0)) for the others.
    template <int C, bool DEFER, class QT>
    __device__ __forceinline__ void chase_at(QT &Q)
    {
        if constexpr (sizeof(T) == 4)
            chase_at_f32<C, DEFER>(Q);
        else
            chase_at_f64<C>(Q);
    }

    // The tail of position C: e_C takes r where the lane's sweep continues
    // below C, and entry C is final (mirror and deflation test).  In a
    // static pass (DEFER) the tail of C runs at the start of position C-1,
    // or when the pass ends: a pass may end at every group boundary, which
    // ends a basic block, and the tail's late operands would otherwise hold
    // up the next group's dependency chain.
    template <int C>
    __device__ __forceinline__ void finish_at()
    {
        if constexpr (sizeof(T) == 4 && C >= 1 && C <= NM - 1) {
            e[C] = ((m_er >> C) & 1u) ? rpend : e[C];
            settle_entry<C>();
        }
    }

    // float.  The rotation of position C comes from the running pair (f, g)
    // that position C+1 produced, and position C produces the pair of C-1:
    // that recurrence is the serial chain of a pass, so it is written to be
    // short.  With fs, gs the pair scaled so that max(|fs|, |gs|) is in
    // [1, 1.125] and r2 = fs^2 + gs^2 (c = fs/sqrt(r2), s = gs/sqrt(r2)), the
    // EXP update of the off-diagonal (page "algo_steqr") is
    //   e+ = (c^2 - s^2) e + c s (d' - d)
    //      = ((fs^2 - gs^2) e + fs gs (d' - d)) / r2,
    // so the next f needs 1/r2 (one Newton step on y0^2, y0 = rsqrt.approx
    // r2, the flush-to-zero form: its operand is normal, and it measured 19
    // cycles of latency against 40 for the form that accepts subnormals)
    // but neither c nor s; the next bulge is s e'' = (gs e'') y.
    // Everything else (d+, d'+, the eigenvector update, r) uses c and s.
    //   scale:  2^-k from the exponent field costs a mask and a subtract;
    //           subtracting the raw bits from those of 2^127 gives a factor
    //           within 1.125 of it in one integer subtract (the rotation is
    //           invariant to the scale, and r = f c + g s needs none);
    //   floor:  r2 gets 2^-100 added, which a normal pair (r2 >= 1) rounds
    //           away, so f = g = 0 yields a finite 1/r2;
    //   exact identity: where g = 0 (and for lanes without a rotation at C,
    //           which run lartg(1, 0)) c = 1, s = 0 are selected and e+ takes
    //           e through masks, so d, e and Q keep their values bit for bit.
    template <int C, bool DEFER, class QT>
    __device__ __forceinline__ void chase_at_f32(QT &Q)
    {
        if constexpr (DEFER)
            finish_at<C + 1>();
        const bool act = (m_act >> C) & 1u;
        const bool first = (m_first >> C) & 1u;
        // one select on the chain: the running pair, or the sweep's seed at
        // its first position, or (1, 0) where the lane has no rotation (a
        // 2x2 solve is a one-position sweep seeded with its rotation)
        const bool own = act && !first;
        const float fa = own ? f : (first ? f0 : 1.0f);
        const float ga = own ? g : (first ? g0 : 0.0f);
        const float mx = fmaxf(fabsf(fa), fabsf(ga));
        const float sc = __uint_as_float(0x7f000000u - __float_as_uint(mx));
        const float fs = fa * sc, gs = ga * sc;
        const float gg = fmaf(gs, gs, 0x1p-100f);
        const float r2 = fmaf(fs, fs, gg);
        float y0;
        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(r2));  // r2 >= 2^-100: normal
        const float z2 = y0 * y0;             // ~ 1/r2
        const float ee = fmaf(-r2, z2, 1.0f);  // 1 - r2 y0^2
        const float y = fmaf(0.5f * y0, ee, y0);  // 1/sqrt(r2), one Newton step
        const bool z = ga == 0.0f;
        float cs = fs * y;
        const float sn = gs * y;
        cs = z ? 1.0f : cs;
        const float a = d[C], b = e[C - 1], cc = d[C - 1];
        // e+ from 1/r2 (the chain), exactly e where g = 0
        const float d1 = fmaf(fs, fs, -gg);
        const float nn = fmaf(d1, z ? 0.0f : b, (fs * gs) * (cc - a));
        const float nz = nn * z2;
        const float en = fmaf(nz, ee, nz + (z ? b : 0.0f));
        // T+ = G^T T G on rows/columns (C, C-1) (page "algo_steqr", EXP):
        // d_C from its explicit formula, d_{C-1} from the trace
        const float p1 = fmaf(cs, a, sn * b);
        const float p2 = fmaf(cs, b, sn * cc);
        const float dn = fmaf(cs, p1, sn * p2);
        d[C] = dn;
        d[C - 1] = z ? cc : (a + cc) - dn;
        rpend = fmaf(fa, cs, ga * sn);
        e[C - 1] = en;
        if constexpr (C >= 2) {
            const float eo = e[C - 2];
            g = (gs * eo) * y;  // new bulge s e''
            e[C - 2] = cs * eo;
        }
        f = en;
        if constexpr (!DEFER)
            finish_at<C>();
        Q.template rot<C>(cs, sn, (m_touch >> C) & 1u);
    }

    template <int C, class QT>
    __device__ __forceinline__ void chase_at_f64(QT &Q)
    {
        const bool in = (m_in >> C) & 1u;
        const bool act = (m_act >> C) & 1u;
        const bool a22 = (m_22 >> C) & 1u;
        const bool first = (m_first >> C) & 1u;
        const T fa = first ? f0 : f;
        const T ga = first ? g0 : g;
        T cs, sn, r;
        lartg(act ? fa : T(1), act ? ga : T(0), cs, sn, r);
        cs = a22 ? cs2 : cs;
        sn = a22 ? sn2 : sn;
        const T a = d[C], b = e[C - 1], cc = d[C - 1];
        // T+ = G^T T G on rows/columns (C, C-1) (page "algo_steqr", EXP);
        // d_{C-1} from the trace identity and a select (the integer pipe is
        // idle next to FP64)
        const T p1 = fma(cs, a, sn * b);
        const T p2 = fma(cs, b, sn * cc);
        const T dn = fma(cs, p1, sn * p2);
        const T en = fma(cs, p2, -sn * p1);
        d[C] = in ? dn : a;
        d[C - 1] = in ? (a + cc) - dn : cc;
        e[C - 1] = a22 ? T(0) : en;
        e[C] = ((m_er >> C) & 1u) ? r : e[C];
        if constexpr (C >= 2) {
            const T eo = e[C - 2];
            g = sn * eo;  // new bulge
            e[C - 2] = cs * eo;
        }
        f = en;
        settle_entry<C>();
        Q.template rot<C>(cs, sn, (m_touch >> C) & 1u);
    }

    // One pass over positions top .. (group boundary <= rlo), where top is
    // the first group top at or above rhi; positions above rhi are inactive
    // in every lane (identity rotations).
    template <class QT>
    __device__ __forceinline__ void run_pass(QT &Q, int rhi, int rlo)
    {
        const int top = group_top<NM, KEXIT>(rhi);
        Q.begin(top);
        int last = 0;
#define BSTQ_POS(C)                                                          \
    if constexpr (C <= NM - 1) {                                             \
        chase_at<C, true>(Q);                                                \
        if constexpr (C > 1 && ((C - 1) % KEXIT) == 0) {                     \
            if (C - 1 < rlo) {                                               \
                last = C - 1;                                                \
                finish_at<C>();                                              \
                settle_entry<C - 1>();                                       \
                settle_entry<C - 2>();                                       \
                goto pass_done;                                              \
            }                                                                \
        }                                                                    \
    }
        BSTQ_GROUPED_SWITCH(KEXIT, group_case<NM>(top), BSTQ_POS)
#undef BSTQ_POS
        last = 0;
        finish_at<1>();
        settle_entry<0>();
    pass_done:
        Q.end(last, (m_touch >> last) & 1u);
    }

    // Nested form of a pass: the lane runs exactly its own positions.
    template <int C, class QT>
    __device__ __forceinline__ void own_positions(QT &Q)
    {
        if constexpr (C >= 1) {
            if (C <= hi_l && C >= lo_l)
                chase_at<C, false>(Q);
            own_positions<C - 1>(Q);
        }
    }
    template <class QT>
    __device__ __forceinline__ void run_pass_nested(QT &Q)
    {
        Q.begin(hi_l);
        own_positions<NM - 1>(Q);
        Q.end(lo_l - 1, true);
        refresh_all();
    }

    __device__ __forceinline__ void post_pass()
    {
        if (task == TASK_2X2) {
            zeroed |= 1u << lo;  // e_lo of the solved 2x2 block
            lo += 2;
            if (lo > le)
                close_block();
        }
        task = TASK_NONE;
        clear_pass();
    }
};

// ---------------------------------------------------------------------------
// Kernel.
// ---------------------------------------------------------------------------
template <typename T, int NM, bool WANTZ, int QS>
struct QFor {
    using type = typename QLayout<T, NM, QS>::type;
    static constexpr int ROWS = QLayout<T, NM, QS>::ROWS;
};
template <typename T, int NM, int QS>
struct QFor<T, NM, false, QS> {
    using type = QNone<T, NM>;
    static constexpr int ROWS = 1;
};

template <typename T, int NM, bool WANTZ, int QS, int SCHED>
__global__ void lane_kernel(KParams p)
{
    extern __shared__ uint4 smem_raw[];
    using QT = typename QFor<T, NM, WANTZ, QS>::type;
    constexpr int KEXIT = WANTZ ? 4 : 2;
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = b < p.batch;

    // dynamic shared memory: [memory rows of Q (shared / hybrid)] [mirror]
    constexpr bool kQShared = WANTZ && (QS == QS_SMEM || QS == QS_HYBRID);
    // (sizes as static_smem_per_thread() on the host side)
    constexpr size_t kQBytesPerLane = kQShared ? size_t(QT::MEM_BYTES) : 0;
    using LaneT = Lane<T, NM, KEXIT>;
    LaneT L;
    L.mir = reinterpret_cast<T *>(reinterpret_cast<char *>(smem_raw) + kQBytesPerLane * blockDim.x) +
            (threadIdx.x >> 5) * LaneT::MIRROR_WARP_ELEMS + (threadIdx.x & 31);
    L.load(p, b, live);
    QT Q;
    if constexpr (WANTZ) {
        if constexpr (kQShared) {
            Q.setup(reinterpret_cast<char *>(smem_raw) + 16 * threadIdx.x, blockDim.x);
        } else if constexpr (QS == QS_GLOBAL) {
            constexpr int G = QLayout<T, NM, QS>::MR * (int)sizeof(T) / 16;
            char *base = reinterpret_cast<char *>(p.qwork) +
                         16ll * ((long long)blockIdx.x * NM * G * blockDim.x + threadIdx.x);
            Q.setup(base, blockDim.x);
        }
        // every lane initialises its Q (dead and poisoned lanes too: the
        // memory rows are read unconditionally during the passes).  Column s
        // of the working Q is column phys(s) of the identity, or of the
        // caller's basis with back_transform (Z P, P the permutation of the
        // mirrored blocks).
        const bool from_z = p.back && L.status == ST_RUN;
        const T *zb = reinterpret_cast<const T *>(p.Q) + b * (long long)L.n * L.n;
        const bool zvec = q_vector_ok<T>(p.Q, L.n);
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            if (from_z && s < L.n)
                Q.init_col_from(s, zb + (long long)L.phys(s) * L.n, L.n, zvec);
            else
                Q.init_col(s, (L.status == ST_RUN && s < L.n) ? L.phys(s) : s);
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
            L.prepare_pass();
            const int rhi = __reduce_max_sync(FULL, L.hi_l);
            const int rlo = __reduce_min_sync(FULL, L.lo_l);
            L.run_pass(Q, rhi, rlo);
            if (has)
                L.post_pass();
        }
    } else {
        while (L.status == ST_RUN) {
            if (L.task == TASK_NONE) {
                L.settle_step();
                continue;
            }
            L.prepare_pass();
            L.run_pass_nested(Q);
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
    if constexpr (WANTZ) {
        const bool vec = q_vector_ok<T>(p.Q, n);
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            if (s < n) {
                T col[QFor<T, NM, WANTZ, QS>::ROWS];
                Q.get_col(s, col);
                store_col(qout + (long long)pos[s] * n, col, n, vec);
            }
        }
    }
    p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
}

}  // namespace bstq
