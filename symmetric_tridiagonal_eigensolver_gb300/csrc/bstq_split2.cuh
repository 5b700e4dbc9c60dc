// Split-role steqr kernel with the eigenvector rows spread over several Q
// warps (float, eigenvectors, 16 < n <= 32).
//
// Above n = 16 one lane cannot hold a useful part of its problem's Q (n^2
// floats, 4 KB at n = 32) in registers, and the one-lane kernel that keeps
// the rest in shared memory spends most of each chase position on the
// eigenvector update in the chase's own instruction stream.  Here each
// group of warps serves 32 problems: one chase warp runs the chase of its
// 32 problems exactly as bstq_lane.cuh does and records each pass's
// rotations in shared memory (as bstq_split.cuh's chase warps do); QW Q
// warps each keep RR + MR rows of those problems' Q (RR rows in registers,
// MR rows streamed from shared memory one column at a time) and apply the
// recorded rotations one pass behind.  Lane j of Q warp q holds rows
// [q (RR + MR), (q + 1) (RR + MR)) of problem j.  The chase warp and its Q
// warps meet once per pass on a named barrier (bar.sync, 32 (1 + QW)
// threads); all of them make the same number of barrier calls.
//
// The arithmetic applied to each problem is the same as in the static-
// position kernel (BatchLAS pages "algo_steqr" and "perf_steqr").
#pragma once

#include "bstq_split.cuh"

namespace bstq {

template <int NM, int QW, int G, int RR, int MR>
struct Split2Shape {
    static constexpr int RQ = RR + MR;          // rows per Q warp
    static constexpr int WARPS = G * (1 + QW);  // chase warps, then Q warps
    static constexpr int THREADS = 32 * WARPS;
    static_assert(QW * RQ >= NM, "the Q warps must cover every row");
    static_assert(THREADS <= 1024, "one block holds at most 1024 threads");
    static_assert(G <= 15, "one named barrier per group");
    // shared memory: mirror | rot | ctrl | hand | qmem
    static constexpr size_t mirror = 2ull * NM * sizeof(float) * 32 * G;
    static constexpr size_t rot = size_t(G) * 2 * NM * 32 * sizeof(float2);
    static constexpr size_t ctrl = size_t(G) * 2 * sizeof(int2);
    static constexpr size_t hand = size_t(G) * 32 * (4 * sizeof(int) + NM);
    static constexpr size_t qmem = size_t(G) * QW * 32 * NM * MR * sizeof(float);
    static constexpr size_t off_rot = mirror;
    static constexpr size_t off_ctrl = off_rot + rot;
    static constexpr size_t off_hand = off_ctrl + ctrl;
    static constexpr size_t off_qmem = (off_hand + hand + 15) / 16 * 16;
    static constexpr size_t total = off_qmem + qmem;
};

// Launch shapes by compile-time size (n in (16, 24] and (24, 32]), from
// measurement on GB300 (batch 32,768, float V): n = 24 with four groups of
// one chase and three Q warps per block (512 threads, 226 KB of shared
// memory) 0.287 ms against 0.368 ms with three groups; n = 32 with two
// groups of one chase and four Q warps (320 threads), the most that the
// shared memory and the register file hold at four register rows.
template <int NM>
struct Split2Cfg;
template <>
struct Split2Cfg<24> {
    static constexpr int QW = 3, G = 4, RR = 4, MR = 4;
};
template <>
struct Split2Cfg<32> {
    static constexpr int QW = 4, G = 2, RR = 4, MR = 4;
};

template <int NM>
using Split2ShapeOf = Split2Shape<NM, Split2Cfg<NM>::QW, Split2Cfg<NM>::G, Split2Cfg<NM>::RR, Split2Cfg<NM>::MR>;

template <int NM, int SCHED>
__global__ void __launch_bounds__(Split2ShapeOf<NM>::THREADS, 1) split2_kernel(KParams p)
{
    static_assert(SCHED == SCHED_FLAT, "the split kernels pair warps per pass");
    using Cfg = Split2Cfg<NM>;
    constexpr int QW = Cfg::QW, G = Cfg::G, RR = Cfg::RR, MR = Cfg::MR;
    using SH = Split2ShapeOf<NM>;
    constexpr int RQ = SH::RQ;
    constexpr int KEXIT = 4;
    extern __shared__ uint4 smem_raw[];
    char *sm = reinterpret_cast<char *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool chase = warp < G;
    const int grp = chase ? warp : (warp - G) / QW;
    const int qi = chase ? 0 : (warp - G) % QW;  // this Q warp's row block
    const int slot = grp * 32 + lane;           // problem within the block
    const long long b = (long long)blockIdx.x * p.ppb + slot;
    const bool live = slot < p.ppb && b < p.batch;
    if (grp * 32 >= p.ppb)
        return;  // no problems for this group: all of its warps leave
    float2 *rot = reinterpret_cast<float2 *>(sm + SH::off_rot) + (size_t)grp * 2 * NM * 32 + lane;
    int2 *ctrl = reinterpret_cast<int2 *>(sm + SH::off_ctrl) + grp * 2;
    int *hand = reinterpret_cast<int *>(sm + SH::off_hand);  // [4][32 G] ints
    unsigned char *hpos = reinterpret_cast<unsigned char *>(hand + 4 * 32 * G) + slot;  // [NM][32 G]
    const int bar = 1 + grp;
    const int nbar = 32 * (1 + QW);
    auto group_barrier = [&]() {
        __syncwarp();
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nbar) : "memory");
    };

    if (chase) {
        Lane<float, NM, KEXIT> L;
        L.mir = reinterpret_cast<float *>(sm) + grp * Lane<float, NM, KEXIT>::MIRROR_WARP_ELEMS + lane;
        L.load(p, b, live);
        hand[0 * 32 * G + slot] = (int)L.zmask;
        hand[1 * 32 * G + slot] = (int)L.revmask;
        hand[2 * 32 * G + slot] = L.status;
        group_barrier();  // start
        QRecorder<NM> Q;
        int parity = 0;
        for (;;) {
            if (L.status == ST_RUN && L.task == TASK_NONE)
                L.settle_step();
            const bool has = L.has_task();
            const bool any = __any_sync(FULL, has);
            int rhi = -1, rlo = NM;
            if (any) {
                L.prepare_pass();
                rhi = __reduce_max_sync(FULL, L.hi_l);
                rlo = __reduce_min_sync(FULL, L.lo_l);
                Q.buf = rot + parity * NM * 32;
                L.run_pass(Q, rhi, rlo);
                if (has)
                    L.post_pass();
            }
            if (lane == 0)
                ctrl[parity] = make_int2(rhi, rlo);
            group_barrier();  // pass recorded (or: no more passes)
            if (!any)
                break;
            parity ^= 1;
        }
        // eigenvalues, info and the output permutation
        const int n = L.n;
        if (live) {
            float *dout = reinterpret_cast<float *>(p.d) + b * n;
            if (L.status == ST_BAD) {
                for (int i = 0; i < n; ++i)
                    dout[i] = __int_as_float(0x7fffffff);
                p.info[b] = -1;
            } else {
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
                for (int s = 0; s < NM; ++s) {
                    if (s < n)
                        dout[pos[s]] = L.d[s];
                    hpos[s * 32 * G] = (unsigned char)pos[s];
                }
                p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
            }
        }
        hand[2 * 32 * G + slot] = L.status;
        group_barrier();  // output permutation ready
    } else {
        group_barrier();  // start
        const unsigned zmask = (unsigned)hand[0 * 32 * G + slot];
        const unsigned revmask = (unsigned)hand[1 * 32 * G + slot];
        const int status0 = hand[2 * 32 * G + slot];
        const int n = p.n;
        const int r0 = qi * RQ;  // first row of Q this warp keeps
        QApplier<NM, KEXIT, QMix<float, NM, RR, MR, 32 * G * QW>> A;
        // Q lane index t = (grp QW + qi) 32 + lane, compile-time stride
        A.Q.setup(sm + SH::off_qmem + 16 * ((grp * QW + qi) * 32 + lane), 0);
        const bool zvec = q_vector_ok<float>(p.Q, n) && (r0 * 4) % 16 == 0;
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            int row = s;
            if (status0 == ST_RUN && s < n) {
                const int a = block_lo(zmask, s), bb = block_hi(zmask, s);
                row = ((revmask >> a) & 1u) ? (a + bb - s) : s;
            }
            if (p.back && status0 == ST_RUN && s < n)
                A.Q.init_col_from(s,
                                  reinterpret_cast<const float *>(p.Q) + b * (long long)n * n + (long long)row * n + r0,
                                  n - r0, zvec);
            else
                A.Q.init_col(s, row - r0);
        }
        int parity = 0;
        for (;;) {
            group_barrier();  // pass recorded
            const int2 c = ctrl[parity];
            if (c.x < 0)
                break;
            A.buf = rot + parity * NM * 32;
            A.pass(c.x, c.y);
            parity ^= 1;
        }
        group_barrier();  // output permutation ready
        const int cnt = n - r0 < RQ ? n - r0 : RQ;  // rows of this block inside the problem
        if (live && cnt > 0) {
            const int status = hand[2 * 32 * G + slot];
            float *qout = reinterpret_cast<float *>(p.Q) + b * (long long)n * n + r0;
            if (status == ST_BAD) {
                for (int s = 0; s < n; ++s)
                    for (int i = 0; i < cnt; ++i)
                        qout[(long long)s * n + i] = __int_as_float(0x7fffffff);
            } else {
                // this warp's rows of each column, as 16-byte vectors when
                // the columns are aligned and the block is whole
                const bool vec = zvec && cnt == RQ;
#pragma unroll
                for (int s = 0; s < NM; ++s) {
                    if (s < n) {
                        float col[RQ];
                        A.Q.get_col(s, col);
                        store_col(qout + (long long)hpos[s * 32 * G] * n, col, cnt, vec);
                    }
                }
            }
        }
    }
}

}  // namespace bstq
