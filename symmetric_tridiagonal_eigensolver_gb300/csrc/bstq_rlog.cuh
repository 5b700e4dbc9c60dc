// Record-and-apply steqr (float, eigenvectors, 32 < n <= 128).
//
// Above n = 32 the lane-per-problem kernel of bstq_dyn.cuh rotates its
// problem's Q in global scratch at every rotation (one column read, one
// written), so its time follows the memory traffic of Q rather than the
// arithmetic.  The pages' path for sizes above one sub-group (BatchLAS page
// "algo_steqr", the steqr_wg paragraph) stores a sweep's rotations and
// applies them afterwards; here that idea spans the whole solve, in three
// launches:
//  1. rlog_chase_kernel (either scheduler; nested by default): lane b runs
//     the dynamic-position chase of problem b without Q and appends every
//     pass to the problem's rotation log in global memory: a header (top
//     position m, count L) and the rotations (cs, sn) of positions m, m-1,
//     ..., m-L+1, the last few of them identities that end the pass on a
//     multiple of kRlogGroup (bstq_dyn.cuh).  The log is cut into pages of
//     kRlogPage entries and a pass never crosses a page boundary: a pass
//     that does not fit in the rest of a page starts the next page, after
//     an end-of-page header (0, 0).  The lane writes the eigenvalues, info,
//     the log length and the problem's column maps (the initial row of each
//     column, from the mirrored blocks, and each column's sorted place).
//     A problem whose log runs out of room stops, leaves d untouched and is
//     marked for the third launch.
//  2. rlog_apply_kernel: one warp per problem (and per 32 rows above
//     n = 64): each lane holds rows of Q in registers (two rows for
//     n <= 64, so a warp covers 64 rows; one row above) and applies every
//     logged rotation in order.  The log pages come into shared memory by
//     asynchronous copies two pages ahead, and each position's rotation is
//     read two positions ahead.  Each column goes to its sorted place.
//  3. rlog_kernel, for the marked problems only (normally none): the same
//     chase from the untouched input with the log applied by the warp
//     whenever a lane's log is full (Q through global memory between such
//     rounds, unpermuted until the last one).
// Every row of Q sees the same rotations in the same order, with the same
// arithmetic, as in the dynamic-position kernel; only the order in which
// the rows are visited changes, so Q is the same to the last bit (the
// identity padding can only turn a -0 entry into +0).
#pragma once

#include <type_traits>

#include "bstq_dyn.cuh"
#include "bstq_plan.h"

namespace bstq {

template <int NM>
struct Rlog {
    // Rows of Q per lane: two for 32 < n_pad <= 64 (rows r0 + lane and
    // r0 + 32 + lane, two independent dependency chains), one otherwise.  Scalar FP32:
    // on GB300 a packed f32x2 rotation (mul, then fma into the other row)
    // measured 23 cycles of latency against 8.4 for the scalar pair, and
    // the update is bound by that chain.
    static constexpr int RPL = (NM > 32 && NM <= 64) ? 2 : 1;
    static constexpr int ROWS = 32 * RPL;  // rows of Q a warp holds at once
    static_assert(ROWS == rlog_rows(NM), "one rule for the rows per warp");
    // three page buffers per warp (pages k, k+1, k+2 in flight), each with
    // two entries of slack for the reads ahead
    static constexpr int BUF = kRlogPage + 2;
    static constexpr size_t WARP_BYTES = 3 * BUF * sizeof(float2);
};

// Shared memory of the finishing launch's blocks: d and e of every problem
// slot (2 NM floats each, [entry][slot]), the per-warp page buffers, and two
// byte maps per slot (the initial row of each column, and each column's
// output place).
__host__ __device__ inline size_t rlog_smem_bytes(int nm, int warps, int ppw)
{
    const size_t slots = size_t(warps) * ppw;
    const size_t per_warp = 3 * (kRlogPage + 2) * 8;
    return 2 * size_t(nm) * slots * 4 + size_t(warps) * per_warp + 2 * size_t(nm) * slots;
}

// Rotation of position C on the lane's rows: columns (C, C-1) as
//   q_C <- cs q_C + sn q_{C-1},  q_{C-1} <- -sn q_C + cs q_{C-1}
// (the arithmetic of bstq_lane.cuh's El<float>, one row at a time).
template <int C, int NM, int RPL>
__device__ __forceinline__ void rlog_rot(float (&q)[RPL][NM], const float2 r)
{
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
        const float x = q[j][C], y = q[j][C - 1];
        q[j][C] = fmaf(r.x, x, r.y * y);
        q[j][C - 1] = fmaf(r.x, y, -r.y * x);
    }
}

// One logged pass: positions m down to lo + 1, lo a multiple of
// kRlogGroup.  top points at the entry of position 0, so position C's
// rotation is top[-C].  The switch enters at m; the end test runs only at
// group boundaries.  An identity rotation leaves the rows as they were (up
// to the sign of a zero).  Rotations are read two positions ahead into
// three slots indexed by position mod 3 (compile-time indices, so the slots
// stay in registers); the reads past the pass's end land in the two slack
// entries of the page and are not used.
template <int NM, int RPL>
__device__ __forceinline__ void rlog_pass(float (&q)[RPL][NM], const float2 *top, int m, int lo)
{
    float2 sl[3];
    switch (m % 3) {
    case 0:
        sl[0] = top[-m];
        sl[2] = top[1 - m];
        break;
    case 1:
        sl[1] = top[-m];
        sl[0] = top[1 - m];
        break;
    default:
        sl[2] = top[-m];
        sl[1] = top[1 - m];
        break;
    }
#define BSTQ_RL(C)                                                            \
    case C:                                                                   \
        if constexpr ((C) <= NM - 1) {                                        \
            sl[((C) + 1) % 3] = top[2 - (C)];                                 \
            rlog_rot<(C), NM, RPL>(q, sl[(C) % 3]);                           \
            if constexpr (((C) - 1) % kRlogGroup == 0) {                      \
                if ((C) - 1 <= lo)                                            \
                    break;                                                    \
            }                                                                 \
        }
#define BSTQ_RL8(B)                                                           \
    BSTQ_RL(B + 7) BSTQ_RL(B + 6) BSTQ_RL(B + 5) BSTQ_RL(B + 4) BSTQ_RL(B + 3) \
    BSTQ_RL(B + 2) BSTQ_RL(B + 1) BSTQ_RL(B + 0)
    switch (m) {
        BSTQ_RL8(120) BSTQ_RL8(112) BSTQ_RL8(104) BSTQ_RL8(96) BSTQ_RL8(88) BSTQ_RL8(80)
        BSTQ_RL8(72) BSTQ_RL8(64) BSTQ_RL8(56) BSTQ_RL8(48) BSTQ_RL8(40) BSTQ_RL8(32)
        BSTQ_RL8(24) BSTQ_RL8(16) BSTQ_RL8(8)
        BSTQ_RL(7) BSTQ_RL(6) BSTQ_RL(5) BSTQ_RL(4) BSTQ_RL(3) BSTQ_RL(2) BSTQ_RL(1)
    default:
        break;
    }
#undef BSTQ_RL8
#undef BSTQ_RL
}

// 8-byte asynchronous copy global -> shared (completes at cp.async.wait_group)
__device__ __forceinline__ void rlog_cp8(void *dst, const void *src)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void rlog_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void rlog_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Status codes in the per-problem log length array (values >= 0 are
// lengths): the input was not finite, or the log ran out of room and the
// finishing launch solves the problem again.
constexpr int kRlogBad = -1;
constexpr int kRlogRedo = -2;
// info value of a problem the finishing launch solves again (replaced by
// that launch)
constexpr int kRlogRedoInfo = 0x7fffffff;

// One problem's Q, rows [r0, r0 + ROWS): initial columns from the column
// map (the identity's, or the basis Z's with back), every logged pass
// applied, each column stored at its place in the output (pos, or column s
// itself when pos is null).  phys[s * ms] and pos[s * ms] are column s's
// entries of the maps.  buf: the warp's three page buffers.  Lane l holds
// rows r0 + l (and r0 + 32 + l), so each column moves as whole 128-byte
// lines.
template <int NM>
__device__ __forceinline__ void rlog_apply_rows(const float2 *lq, int cq, float *Qb, int n, int r0, bool fresh,
                                                bool back, const unsigned char *phys, const unsigned char *pos,
                                                int ms, float2 *buf)
{
    using R = Rlog<NM>;
    constexpr int RPL = R::RPL;
    const int lane = threadIdx.x & 31;
    const int pages = (cq + kRlogPage - 1) / kRlogPage;
    auto issue = [&](int k) {
        if (k < pages) {
            const int len = cq - k * kRlogPage < kRlogPage ? cq - k * kRlogPage : kRlogPage;
            float2 *dst = buf + (k % 3) * R::BUF;
            const float2 *src = lq + (long long)k * kRlogPage;
            for (int j = lane; j < len; j += 32)
                rlog_cp8(dst + j, src + j);
        }
        rlog_commit();
    };
    issue(0);
    issue(1);
    float q[RPL][NM];
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
        const int row = r0 + 32 * j + lane;
        const bool in = row < n;
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            float v = 0.f;
            if (s < n) {
                if (fresh) {
                    const int ps = phys[s * ms];
                    if (back)
                        v = in ? Qb[(long long)ps * n + row] : 0.f;
                    else
                        v = ps == row ? 1.f : 0.f;
                } else {
                    v = in ? Qb[(long long)s * n + row] : 0.f;
                }
            }
            q[j][s] = v;
        }
    }
    for (int k = 0; k < pages; ++k) {
        rlog_wait<1>();  // page k has landed (this lane's part)
        __syncwarp();
        issue(k + 2);  // into the buffer of page k - 1, read by every lane
        const int plen = cq - k * kRlogPage < kRlogPage ? cq - k * kRlogPage : kRlogPage;
        const float2 *pg = buf + (k % 3) * R::BUF;
        int w = 0;
        while (w < plen) {
            const float2 h = pg[w];
            const int m = __float_as_int(h.x), ls = __float_as_int(h.y);
            // a pass is 1 <= ls <= m <= NM - 1 rotations ending on a group
            // boundary, whole inside the page; an end-of-page header has
            // ls = 0
            if (ls < 1 || ls > m || m >= NM || (m - ls) % kRlogGroup != 0 || w + 1 + ls > plen)
                break;
            rlog_pass<NM, RPL>(q, pg + w + 1 + m, m, m - ls);
            w += 1 + ls;
        }
        __syncwarp();
    }
    rlog_wait<0>();
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
        const int row = r0 + 32 * j + lane;
        if (row < n) {
#pragma unroll
            for (int s = 0; s < NM; ++s) {
                if (s < n) {
                    const int col = pos ? pos[s * ms] : s;
                    Qb[(long long)col * n + row] = q[j][s];
                }
            }
        }
    }
}

// Column maps of a problem in the lane's own smem slot or global array:
// the initial row of column s (phys) at mp[s * ms], its output place at
// mq[s * ms].
template <typename LaneT>
__device__ __forceinline__ void rlog_output(const KParams &p, LaneT &L, long long b, unsigned char *mq, int ms)
{
    const int n = L.n;
    float *dout = reinterpret_cast<float *>(p.d) + b * n;
    if (L.status == ST_BAD) {
        for (int i = 0; i < n; ++i)
            dout[i] = __int_as_float(0x7fffffff);
        p.info[b] = -1;
        return;
    }
    const bool sorted = p.sort && L.status == ST_DONE;
    for (int s = 0; s < n; ++s) {
        const float ds = L.D(s);
        const int phs = L.phys(s);
        int pos = phs;
        if (sorted) {
            pos = 0;
            for (int t = 0; t < n; ++t) {
                const float dt = L.D(t);
                pos += (dt < ds || (dt == ds && L.phys(t) < phs)) ? 1 : 0;
            }
        }
        dout[pos] = ds;
        mq[s * ms] = (unsigned char)pos;
    }
    p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
}

// Launch 1: the chase of every problem with its rotation log.
template <int NM, int SCHED>
__global__ void rlog_chase_kernel(KParams p)
{
    using LaneT = DynLane<float, NM, false, true>;
    extern __shared__ uint4 smem_raw[];
    const int tpb = blockDim.x;
    const long long b = (long long)blockIdx.x * tpb + threadIdx.x;
    const bool live = b < p.batch;
    const int n = p.n;
    const long long cap = p.lcap;  // a multiple of kRlogPage

    LaneT L;
    L.ms = tpb;
    L.sd = reinterpret_cast<float *>(smem_raw) + threadIdx.x;
    L.se = L.sd + NM * tpb;
    L.sdl = L.sil = nullptr;
    L.scr = nullptr;
    L.da = L.ia = 1.f;
    L.pg = p.scheme == 1;
    L.lg = reinterpret_cast<float2 *>(p.qwork) + (live ? b : 0) * cap;
    L.cnt = 0;
    L.lpad = 0;
    L.load(p, b, live);
    unsigned char *mp = p.lmap + (live ? b : 0) * 2 * n;
    if (live && L.status == ST_RUN)
        for (int s = 0; s < n; ++s)
            mp[s] = (unsigned char)L.phys(s);
    bool redo = false;
    // Room for the next pass: 1 + (m - lo) entries and the padding, inside
    // one page.  Without room the lane stops (the finishing launch takes
    // its problem); else an end-of-page header closes the page when needed.
    auto make_room = [&]() -> bool {
        const int need = 1 + L.m - (L.lo / kRlogGroup) * kRlogGroup;
        long long at = L.cnt;
        if ((at % kRlogPage) + need > kRlogPage)
            at = (at / kRlogPage + 1) * kRlogPage;
        if (at + need > cap) {
            redo = true;
            L.status = ST_DEAD;
            return false;
        }
        if ((L.cnt % kRlogPage) + need > kRlogPage) {
            L.lg[L.cnt] = make_float2(0.f, 0.f);  // end of this page
            L.cnt = (L.cnt / kRlogPage + 1) * kRlogPage;
        }
        return true;
    };
    if constexpr (SCHED == SCHED_NESTED) {
        // every lane runs its own loop: with no eigenvector work in the
        // chase, this measured faster than the lockstep form (f32 V n = 64
        // 3.71 against 3.81 ms, n = 128 10.16 against 10.75 ms)
        while (L.status == ST_RUN) {
            if (L.task == TASK_NONE) {
                L.settle_step();
                continue;
            }
            if (!make_room())
                break;
            L.begin_pass();
            for (int k = 0; k < L.L; ++k)
                L.step(k);
            L.post_pass();
        }
    } else {
        for (;;) {
            if (L.status == ST_RUN && L.task == TASK_NONE)
                L.settle_step();
            bool has = L.has_task();
            if (has && !make_room())
                has = false;
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
    }
    if (!live)
        return;
    if (redo) {
        p.lcnt[b] = kRlogRedo;
        p.info[b] = kRlogRedoInfo;
        return;
    }
    rlog_output(p, L, b, mp + n, 1);
    p.lcnt[b] = L.status == ST_BAD ? kRlogBad : L.cnt;
}

// Launch 2: one warp per problem and row chunk applies the problem's log.
template <int NM, int SCHED>
__global__ void __launch_bounds__(128, 3) rlog_apply_kernel(KParams p)
{
    using R = Rlog<NM>;
    extern __shared__ uint4 smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    const int chunks = (n + R::ROWS - 1) / R::ROWS;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
    const long long b = gw / chunks;
    const int r0 = (int)(gw % chunks) * R::ROWS;
    if (b >= p.batch)
        return;
    const int cq = p.lcnt[b];
    if (cq == kRlogRedo)
        return;  // solved again by the finishing launch
    float *Qb = reinterpret_cast<float *>(p.Q) + b * (long long)n * n;
    if (cq == kRlogBad) {
        // non-finite input: Q is NaN (this chunk's rows)
        for (int s = 0; s < n; ++s)
            for (int i = r0 + lane; i < n && i < r0 + R::ROWS; i += 32)
                Qb[(long long)s * n + i] = __int_as_float(0x7fffffff);
        return;
    }
    float2 *wb = reinterpret_cast<float2 *>(reinterpret_cast<char *>(smem_raw) + size_t(warp) * R::WARP_BYTES);
    const unsigned char *mp = p.lmap + b * 2 * n;
    rlog_apply_rows<NM>(reinterpret_cast<const float2 *>(p.qwork) + b * p.lcap, cq, Qb, n, r0, true, p.back != 0,
                        mp, mp + n, 1, wb);
}

// Launch 3: the chase with the apply rounds inside, for the problems whose
// log ran out of room in launch 1 (info == kRlogRedoInfo on entry); every
// other lane is idle.  ppw problems per warp; their maps in shared memory.
template <int NM, int SCHED>
__global__ void __launch_bounds__(256, 1) rlog_kernel(KParams p)
{
    static_assert(SCHED == SCHED_FLAT, "the record-and-apply kernels run the flat scheduler");
    using R = Rlog<NM>;
    using LaneT = DynLane<float, NM, false, true>;
    extern __shared__ uint4 smem_raw[];
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ppw = p.ppb;
    const int S = nw * ppw;         // problem slots of the block
    const int slot0 = warp * ppw;   // first slot of this warp
    const long long b0 = (long long)blockIdx.x * S + slot0;  // first problem of this warp
    const bool mine = lane < ppw;
    const long long b = b0 + lane;
    const bool live = mine && b < p.batch && p.info[b] == kRlogRedoInfo;
    if (!__any_sync(FULL, live))
        return;
    const int n = p.n;
    const long long cap = p.lcap;

    char *sm = reinterpret_cast<char *>(smem_raw);
    float *smf = reinterpret_cast<float *>(sm);
    char *wbuf = sm + size_t(2) * NM * S * sizeof(float) + size_t(warp) * R::WARP_BYTES;
    unsigned char *sphys =
        reinterpret_cast<unsigned char *>(sm + size_t(2) * NM * S * sizeof(float) + size_t(nw) * R::WARP_BYTES);
    unsigned char *spos = sphys + NM * S;
    float2 *pbuf = reinterpret_cast<float2 *>(wbuf);

    LaneT L;
    const int slot = slot0 + (mine ? lane : 0);  // lanes without a problem never touch their slot
    L.ms = S;
    L.sd = smf + slot;
    L.se = L.sd + NM * S;
    L.sdl = L.sil = nullptr;
    L.scr = nullptr;
    L.da = L.ia = 1.f;
    L.pg = p.scheme == 1;
    L.lg = reinterpret_cast<float2 *>(p.qwork) + (live ? b : 0) * cap;
    L.cnt = 0;
    L.lpad = 0;
    L.load(p, b, live);
    if (live && L.status == ST_RUN)
        for (int s = 0; s < n; ++s)
            sphys[s * S + slot] = (unsigned char)L.phys(s);
    bool fresh = true;  // Q of this lane's problem not yet written by a round

    // One round: the warp applies the logs of its problems (fin: the last
    // round, every problem with the columns at their sorted places).
    auto apply_round = [&](bool fin) {
        __syncwarp();  // the logs and the maps written by the lanes
        for (int qq = 0; qq < ppw; ++qq) {
            const long long bq = b0 + qq;
            if (bq >= p.batch)
                break;
            const int st = __shfl_sync(FULL, L.status, qq);
            const int cq = __shfl_sync(FULL, L.cnt, qq);
            const bool fr = __shfl_sync(FULL, fresh ? 1 : 0, qq) != 0;
            if (st == ST_DEAD)
                continue;  // not this launch's problem
            float *Qb = reinterpret_cast<float *>(p.Q) + bq * (long long)n * n;
            if (st == ST_BAD) {
                if (fin)
                    for (long long i = lane; i < (long long)n * n; i += 32)
                        Qb[i] = __int_as_float(0x7fffffff);
                continue;
            }
            if (!fin && cq == 0)
                continue;
            for (int r0 = 0; r0 < n; r0 += R::ROWS)
                rlog_apply_rows<NM>(reinterpret_cast<const float2 *>(p.qwork) + bq * cap, cq, Qb, n, r0, fr,
                                    p.back != 0, sphys + slot0 + qq, fin ? spos + slot0 + qq : nullptr, S, pbuf);
        }
        __syncwarp();
        if (L.cnt > 0 || fin)
            fresh = false;
        L.cnt = 0;
    };

    for (;;) {
        if (L.status == ST_RUN && L.task == TASK_NONE)
            L.settle_step();
        const bool has = L.has_task();
        if (!__any_sync(FULL, has))
            break;
        // apply the logs first when one of the warp's lanes has no room left
        // for its pass
        const int need = 1 + L.m - (L.lo / kRlogGroup) * kRlogGroup;
        long long at = L.cnt;
        if (has && (at % kRlogPage) + need > kRlogPage)
            at = (at / kRlogPage + 1) * kRlogPage;
        const bool full = has && at + need > cap;
        if (__any_sync(FULL, full))
            apply_round(false);
        if (has && (L.cnt % kRlogPage) + need > kRlogPage) {
            L.lg[L.cnt] = make_float2(0.f, 0.f);  // end of this page
            L.cnt = (L.cnt / kRlogPage + 1) * kRlogPage;
        }
        L.begin_pass();
        const int steps = __reduce_max_sync(FULL, L.L);
        for (int k = 0; k < steps; ++k)
            if (k < L.L)
                L.step(k);
        if (has)
            L.post_pass();
    }
    if (live)
        rlog_output(p, L, b, spos + slot, S);
    apply_round(true);
}

}  // namespace bstq
