// Split-role steqr kernel (float, eigenvectors): chase warps and Q warps.
//
// The static-position kernel runs the bulge chase and the eigenvector update
// of a problem in the same thread, so the long dependency chain of the chase
// and the wide, independent eigenvector FMAs share one in-order instruction
// stream and one register budget.  Here every block holds 8 pairs of warps
// as four warpgroups: warpgroups 0-1 are chase warps, 2-3 their Q partners.
// The block is launched with 128 registers per thread (the whole register
// file for 512 threads); the chase warpgroups then give registers back
// (setmaxnreg.dec to kSplitChaseRegs) and the Q warpgroups take them
// (setmaxnreg.inc to kSplitQRegs), so a Q lane holds 8 rows of its problem's
// Q in registers without spilling while the chase keeps what it needs.  The
// host launches this kernel only after checking that the compiled kernel
// uses exactly those 128 registers, so the increase always finds its
// registers.  At most kSplitLivePairs pairs carry problems (shared memory
// holds seven pairs' state); the eighth pair exits right after the register
// hand-over.
// Lane j of chase warp w runs the chase of problem (block, w, j) exactly as
// bstq_lane.cuh does, but instead of rotating Q it records the pass's
// rotations (cs, sn) per position in shared memory.  Lane j of the partner Q
// warp keeps that problem's whole Q in registers and applies the recorded
// rotations one pass behind, while the chase warp already computes the next
// pass (double-buffered).  The two warps meet once per pass on a named
// barrier (bar.sync with 64 threads); both execute exactly the same number
// of barrier calls: one to start, one per pass including the final empty
// one that announces the end, and one before the output.
//
// The arithmetic applied to each problem is the same as in the static-
// position kernel (BatchLAS pages "algo_steqr" and "perf_steqr").
#pragma once

#include "bstq_lane.cuh"

namespace bstq {

constexpr int kSplitPairs = 8;      // 8 chase + 8 Q warps: four warpgroups, 512 threads
constexpr int kSplitLivePairs = 7;  // pairs that carry problems: up to 224 per block
constexpr int kSplitLaunchRegs = 128;
constexpr int kSplitChaseRegs = 96;
constexpr int kSplitQRegs = 160;
static_assert(4 * 32 * (2 * kSplitChaseRegs + 2 * kSplitQRegs) <= 32 * kSplitPairs * 2 * kSplitLaunchRegs,
              "register hand-over must fit the launch allocation");

__device__ __forceinline__ void pair_barrier(int id)
{
    __syncwarp();
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// Q policy of the chase warp: record (cs, sn) of position C.
template <int NM>
struct QRecorder {
    float2 *buf;  // this lane's slot of the current pass buffer
    __device__ __forceinline__ void init_col(int, int) {}
    __device__ __forceinline__ void begin(int) {}
    __device__ __forceinline__ void end(int, bool) {}
    template <int C>
    __device__ __forceinline__ void rot(float cs, float sn, bool)
    {
        buf[C * 32] = make_float2(cs, sn);
    }
};

// Rows of Q the Q warp keeps in registers (8 rows: 128 registers of the
// kSplitQRegs); the rest (a multiple of 4) is streamed from shared memory
// like the hybrid store.
template <int NM>
constexpr int split_reg_rows()
{
    return NM <= 8 ? NM : 8;
}

// Q warp: applies one recorded pass to Q (registers + shared rows).
// The shared rows use the block's fixed lane stride (32 lanes per live pair),
// and each position's rotation is read one position ahead, before the
// position's store, so neither shared-memory read waits behind a store.
template <int NM, int KEXIT,
          class QM = QMix<float, NM, split_reg_rows<NM>(), NM - split_reg_rows<NM>(), 32 * kSplitLivePairs>>
struct QApplier {
    QM Q;
    const float2 *buf;
    float2 rn;  // rotation of the next position

    template <int C>
    __device__ __forceinline__ void apply_at()
    {
        const float2 r = rn;
        if constexpr (C >= 2)
            rn = buf[(C - 1) * 32];
        Q.template rot<C>(r.x, r.y, true);
    }

    // same entry and group exits as Lane::run_pass, so exactly the recorded
    // positions are read; identity rotations leave a column unchanged (up to
    // the sign of a zero), so every streamed column is written back
    __device__ __forceinline__ void pass(int rhi, int rlo)
    {
        const int top = group_top<NM, KEXIT>(rhi);
        rn = buf[top * 32];
        Q.begin(top);
        int last = 0;
#define BSTQ_APOS(C)                                                         \
    if constexpr (C <= NM - 1) {                                             \
        apply_at<C>();                                                       \
        if constexpr (C > 1 && ((C - 1) % KEXIT) == 0) {                     \
            if (C - 1 < rlo) {                                               \
                last = C - 1;                                                \
                goto applied;                                                \
            }                                                                \
        }                                                                    \
    }
        BSTQ_GROUPED_SWITCH(KEXIT, group_case<NM>(top), BSTQ_APOS)
#undef BSTQ_APOS
        last = 0;
    applied:
        Q.end(last, true);
    }
};

// Shared-memory layout of one block (P = kSplitLivePairs pairs, 32 lanes
// each):
//   mirror   : 2 * NM floats per chase lane, per warp [entry][lane]
//   rot      : [pair][parity][NM][32] float2             (recorded passes)
//   ctrl     : [pair][parity] int2 (rhi, rlo); rhi < 0 ends the loop
//   handoff  : per chase lane: zmask, revmask, status, n and pos[NM] bytes
template <int NM>
struct SplitSmem {
    static constexpr int P = kSplitLivePairs;
    static constexpr size_t mirror = 2ull * NM * sizeof(float) * 32 * P;
    static constexpr size_t rot = size_t(P) * 2 * NM * 32 * sizeof(float2);
    static constexpr size_t ctrl = size_t(P) * 2 * sizeof(int2);
    static constexpr size_t hand = size_t(P) * 32 * (4 * sizeof(int) + NM);
    static constexpr size_t qmem = size_t(P) * 32 * NM * (NM - split_reg_rows<NM>()) * sizeof(float);
    static constexpr size_t off_rot = mirror;
    static constexpr size_t off_ctrl = off_rot + rot;
    static constexpr size_t off_hand = off_ctrl + ctrl;
    static constexpr size_t off_qmem = (off_hand + hand + 15) / 16 * 16;
    static constexpr size_t total = off_qmem + qmem;
};
static_assert(SplitSmem<16>::total <= 232448, "split-role shared memory exceeds the per-block maximum");

template <int NM, int SCHED>
__global__ void __launch_bounds__(32 * 2 * kSplitPairs, 1) split_kernel(KParams p)
{
    static_assert(SCHED == SCHED_FLAT, "the split kernel pairs warps per pass");
    extern __shared__ uint4 smem_raw[];
    using SM = SplitSmem<NM>;
    constexpr int P = kSplitLivePairs;  // stride of the per-lane shared arrays
    constexpr int KEXIT = 4;
    char *sm = reinterpret_cast<char *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool chase = warp < kSplitPairs;
    const int pair = chase ? warp : warp - kSplitPairs;
    // no problems for this pair: both of its warps leave right after the
    // register hand-over (which every warp of a warpgroup executes)
    const bool idle = pair >= kSplitLivePairs || pair * 32 >= p.ppb;
    const int slot = pair * 32 + lane;  // chase-lane index within the block
    const long long b = (long long)blockIdx.x * p.ppb + slot;
    const bool live = slot < p.ppb && b < p.batch;
    float2 *rot = reinterpret_cast<float2 *>(sm + SM::off_rot) + (size_t)pair * 2 * NM * 32 + lane;
    int2 *ctrl = reinterpret_cast<int2 *>(sm + SM::off_ctrl) + pair * 2;
    int *hand = reinterpret_cast<int *>(sm + SM::off_hand);  // [4][32 P] ints
    unsigned char *hpos = reinterpret_cast<unsigned char *>(hand + 4 * 32 * P) + slot;  // [NM][32 P]
    const int bar = 1 + pair;

    // Each role changes its register budget inside its own branch, so the
    // compiler allocates each role's code under that role's budget.
    if (chase) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kSplitChaseRegs) : "memory");
        if (idle)
            return;
        Lane<float, NM, KEXIT> L;
        L.mir = reinterpret_cast<float *>(sm) + pair * Lane<float, NM, KEXIT>::MIRROR_WARP_ELEMS + lane;
        L.load(p, b, live);
        hand[0 * 32 * P + slot] = (int)L.zmask;
        hand[1 * 32 * P + slot] = (int)L.revmask;
        hand[2 * 32 * P + slot] = L.status;
        pair_barrier(bar);  // start
        QRecorder<NM> Q;
        int parity = 0;
        for (;;) {
            // settle every lane without a task (one call settles it fully)
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
            pair_barrier(bar);  // pass recorded (or: no more passes)
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
                    hpos[s * 32 * P] = (unsigned char)pos[s];
                }
                p.info[b] = (L.status == ST_FAIL) ? L.info : 0;
            }
        }
        hand[2 * 32 * P + slot] = L.status;
        pair_barrier(bar);  // output permutation ready
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kSplitQRegs) : "memory");
        if (idle)
            return;
        pair_barrier(bar);  // start
        const unsigned zmask = (unsigned)hand[0 * 32 * P + slot];
        const unsigned revmask = (unsigned)hand[1 * 32 * P + slot];
        const int status0 = hand[2 * 32 * P + slot];
        const int n = p.n;
        QApplier<NM, KEXIT> A;
        A.Q.setup(sm + SM::off_qmem + 16 * slot, 32 * P);
#pragma unroll
        for (int s = 0; s < NM; ++s) {
            int row = s;
            if (status0 == ST_RUN && s < n) {
                const int a = block_lo(zmask, s), bb = block_hi(zmask, s);
                row = ((revmask >> a) & 1u) ? (a + bb - s) : s;
            }
            // column `row` of the identity, or of the caller's basis with
            // back_transform
            if (p.back && status0 == ST_RUN && s < n)
                A.Q.init_col_from(s, reinterpret_cast<const float *>(p.Q) + b * (long long)n * n + (long long)row * n,
                                  n, q_vector_ok<float>(p.Q, n));
            else
                A.Q.init_col(s, row);
        }
        int parity = 0;
        for (;;) {
            pair_barrier(bar);  // pass recorded
            const int2 c = ctrl[parity];
            if (c.x < 0)
                break;
            A.buf = rot + parity * NM * 32;
            A.pass(c.x, c.y);
            parity ^= 1;
        }
        pair_barrier(bar);  // output permutation ready
        if (live) {
            const int status = hand[2 * 32 * P + slot];
            float *qout = reinterpret_cast<float *>(p.Q) + b * (long long)n * n;
            if (status == ST_BAD) {
                for (int i = 0; i < n * n; ++i)
                    qout[i] = __int_as_float(0x7fffffff);
            } else {
                const bool vec = q_vector_ok<float>(p.Q, n);
#pragma unroll
                for (int s = 0; s < NM; ++s) {
                    if (s < n) {
                        float col[NM];
                        A.Q.get_col(s, col);
                        store_col(qout + (long long)hpos[s * 32 * P] * n, col, n, vec);
                    }
                }
            }
        }
    }
}

}  // namespace bstq
