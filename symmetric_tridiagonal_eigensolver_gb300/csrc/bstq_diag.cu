// Diagnostic kernels: one building block of the solve at a time, on a table
// of inputs, so that each block can be checked on its own against exact or
// higher-precision arithmetic (the unit layer under the end-to-end parity
// tests).  They call the very device functions and lane structures the
// solver kernels use: the reciprocal / quotient / square-root refinements,
// lartg, the shift with its 2x2 rotation (BatchLAS page "algo_steqr": Givens
// rotation, copysign shift, 2x2 solve), one pass of the bulge chase with the
// EXP or PG update in both kernel families (page "algo_steqr": implicit step,
// update schemes), and the factored double eigenvector update with its scale
// guard.
#include <cuda_runtime.h>

#include <stdint.h>

#include "../../include/bstq.h"
#include "bstq_diag.h"
#include "bstq_dyn.cuh"

namespace bstq {
namespace {

constexpr int kDiagNM = 16;  // compile-time size of the pass diagnostics
constexpr int kDiagTpb = 64;
// one pass: record and result sizes, in elements of the dtype
constexpr int kPassIn = 10 + 2 * kDiagNM;
constexpr int kPassOut = 2 * kDiagNM + kDiagNM * kDiagNM;

template <typename T>
__global__ void diag_scalar(int op, long long count, const T *in, T *out)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count)
        return;
    switch (op) {
    case BSTQ_DIAG_RCP:
        out[i] = rcp_nr(in[i]);
        break;
    case BSTQ_DIAG_DIV:
        out[i] = div_nr(in[2 * i], in[2 * i + 1]);
        break;
    case BSTQ_DIAG_SQRT:
        out[i] = sqrt_nr(in[i]);
        break;
    case BSTQ_DIAG_RSQRT:
        out[i] = rsqrt_nr(in[i]);
        break;
    case BSTQ_DIAG_HYP1:
        out[i] = hyp1(in[i]);
        break;
    case BSTQ_DIAG_LARTG:
    case BSTQ_DIAG_LARTG_FAST: {
        T c, s, r;
        if constexpr (sizeof(T) == 8) {
            if (op == BSTQ_DIAG_LARTG_FAST)
                lartg_fast(in[2 * i], in[2 * i + 1], c, s, r);
            else
                lartg(in[2 * i], in[2 * i + 1], c, s, r);
        } else {
            lartg(in[2 * i], in[2 * i + 1], c, s, r);
        }
        out[3 * i] = c;
        out[3 * i + 1] = s;
        out[3 * i + 2] = r;
        break;
    }
    case BSTQ_DIAG_SHIFT: {
        T t, mu, cs, sn;
        shift_tangent(in[3 * i], in[3 * i + 1], in[3 * i + 2], t, mu);
        rot_from_tangent(t, cs, sn);
        out[4 * i] = t;
        out[4 * i + 1] = mu;
        out[4 * i + 2] = cs;
        out[4 * i + 3] = sn;
        break;
    }
    default:
        break;
    }
}

// Record of one pass (elements of T): n, lo, m, task (1 sweep, 2 2x2 solve),
// rhi, rlo (the warp's union of positions, containing [lo+1, m]), f0, g0
// (the sweep's seed), cs2, sn2 (the 2x2 rotation), d[16], e[16].
// Result: d[16], e[16], then Q (16 x 16, column-major): the product of the
// pass's rotations, i.e. T_after = Q^T T_before Q.
template <typename T>
struct PassRec {
    int n, lo, m, task, rhi, rlo;
    T f0, g0, cs2, sn2;
    __device__ PassRec(const T *r)
    {
        n = (int)r[0];
        lo = (int)r[1];
        m = (int)r[2];
        task = (int)r[3];
        rhi = (int)r[4];
        rlo = (int)r[5];
        f0 = r[6];
        g0 = r[7];
        cs2 = r[8];
        sn2 = r[9];
    }
};

// Static-position family: Lane<T, 16> with Q in registers.
template <typename T>
__global__ void diag_pass_static(long long count, const T *in, T *out)
{
    extern __shared__ uint4 smem_raw[];
    constexpr int NM = kDiagNM;
    using LaneT = Lane<T, NM, 4>;
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= count)
        return;
    const T *rec = in + b * kPassIn;
    const PassRec<T> pr(rec);
    LaneT L;
    L.mir = reinterpret_cast<T *>(smem_raw) + (threadIdx.x >> 5) * LaneT::MIRROR_WARP_ELEMS + (threadIdx.x & 31);
#pragma unroll
    for (int i = 0; i < NM; ++i) {
        L.d[i] = rec[10 + i];
        L.e[i] = rec[10 + NM + i];
    }
    // the state settle_step leaves behind for this task
    L.n = pr.n;
    L.status = ST_RUN;
    L.info = 0;
    L.zmask = 0;
    L.revmask = 0;
    L.tmask = 0;
    L.zeroed = 0;
    L.inblock = true;
    L.lb = 0;
    L.le = pr.n - 1;
    L.bnext = pr.n;
    L.iscale = 0;
    L.jtot = 0;
    L.budget = 1;
    L.lo = pr.lo;
    L.m = pr.m;
    L.task = pr.task;
    L.f = L.g = L.rpend = T(0);
    L.f0 = pr.f0;
    L.g0 = pr.g0;
    L.cs2 = pr.cs2;
    L.sn2 = pr.sn2;
    if (sizeof(T) == 4 && pr.task == TASK_2X2) {
        // as settle_step leaves it: the float 2x2 solve is a one-position
        // sweep seeded with its rotation
        L.f0 = pr.cs2;
        L.g0 = pr.sn2;
    }
    L.prepare_pass();
    QMix<T, NM, NM, 0> Q;
#pragma unroll
    for (int s = 0; s < NM; ++s)
        Q.init_col(s, s);
    L.run_pass(Q, pr.rhi, pr.rlo);
    L.post_pass();
    T *o = out + b * kPassOut;
    // entries the pass set to zero through the mask read as zero
#pragma unroll
    for (int i = 0; i < NM; ++i) {
        o[i] = L.d[i];
        o[NM + i] = ((L.zeroed >> i) & 1u) ? T(0) : L.e[i];
    }
#pragma unroll
    for (int s = 0; s < NM; ++s) {
        T col[NM];
        Q.get_col(s, col);
#pragma unroll
        for (int r = 0; r < NM; ++r)
            o[2 * NM + s * NM + r] = col[r];
    }
}

// Dynamic-position family: DynLane<T, 16> (d, e in shared memory, Q in the
// work buffer), EXP or PG update.
template <typename T>
__global__ void diag_pass_dyn(long long count, int pg, const T *in, T *out, void *qwork)
{
    extern __shared__ uint4 smem_raw[];
    constexpr int NM = kDiagNM;
    using LaneT = DynLane<T, NM, true>;
    using Q_ = DynQ<T, NM>;
    const int tpb = blockDim.x;
    const long long b = (long long)blockIdx.x * tpb + threadIdx.x;
    if (b >= count)
        return;
    const T *rec = in + b * kPassIn;
    const PassRec<T> pr(rec);
    LaneT L;
    L.ms = tpb;
    L.sd = reinterpret_cast<T *>(smem_raw) + threadIdx.x;
    L.se = L.sd + NM * tpb;
    L.sdl = L.se + NM * tpb;
    L.sil = L.sdl + NM * tpb;
    L.q.base = reinterpret_cast<typename Q_::V16 *>(qwork) + ((long long)blockIdx.x * NM * Q_::G * tpb + threadIdx.x);
    L.q.stride = tpb;
    for (int i = 0; i < NM; ++i) {
        L.setD(i, rec[10 + i]);
        L.setE(i, rec[10 + NM + i]);
        L.q.init_col(i, i);
        L.sdl[i * tpb] = T(1);
        L.sil[i * tpb] = T(1);
    }
    L.da = L.ia = T(1);
    L.n = pr.n;
    L.status = ST_RUN;
    L.info = 0;
    L.zmask = 0;
    L.revmask = 0;
    L.inblock = true;
    L.lb = 0;
    L.le = pr.n - 1;
    L.bnext = pr.n;
    L.iscale = 0;
    L.jtot = 0;
    L.budget = 1;
    L.lo = pr.lo;
    L.m = pr.m;
    L.task = pr.task;
    L.f = pr.f0;
    L.g = pr.g0;
    L.cs2 = pr.cs2;
    L.sn2 = pr.sn2;
    L.pg = pg != 0;
    L.begin_pass();
    for (int k = 0; k < L.L; ++k)
        L.step(k);
    T *o = out + b * kPassOut;
    for (int i = 0; i < NM; ++i) {
        o[i] = L.D(i);
        o[NM + i] = L.Ev(i);
    }
    for (int s = 0; s < NM; ++s) {
        typename Q_::E x[Q_::NE];
        L.q.load(s, x);
        T col[Q_::NR];
#pragma unroll
        for (int j = 0; j < Q_::NE; ++j)
            El<T>::get(x[j], &col[j * Q_::RPE]);
        const T sc = LaneT::FASTQ ? L.sdl[s * tpb] : T(1);
        for (int r = 0; r < NM; ++r)
            o[2 * NM + s * NM + r] = col[r] * sc;
    }
}

// The factored double eigenvector update alone: K sweeps over the whole
// 16 x 16 Q (positions 15 .. 1, the column of each step carried to the
// next, as in a pass), rotation (c, s) of sweep k, step j at
// in[((b * K + k) * 15 + j) * 2].  Result: Q = Qt diag(delta), 256 values.
__global__ void diag_fastq(long long count, int K, const double *in, double *out, void *qwork)
{
    extern __shared__ uint4 smem_raw[];
    constexpr int NM = kDiagNM;
    using LaneT = DynLane<double, NM, true>;
    using Q_ = DynQ<double, NM>;
    const int tpb = blockDim.x;
    const long long b = (long long)blockIdx.x * tpb + threadIdx.x;
    if (b >= count)
        return;
    LaneT L;
    L.ms = tpb;
    L.sd = reinterpret_cast<double *>(smem_raw) + threadIdx.x;
    L.se = L.sd + NM * tpb;
    L.sdl = L.se + NM * tpb;
    L.sil = L.sdl + NM * tpb;
    L.q.base = reinterpret_cast<typename Q_::V16 *>(qwork) + ((long long)blockIdx.x * NM * Q_::G * tpb + threadIdx.x);
    L.q.stride = tpb;
    for (int i = 0; i < NM; ++i) {
        L.q.init_col(i, i);
        L.sdl[i * tpb] = 1.0;
        L.sil[i * tpb] = 1.0;
    }
    L.n = NM;
    L.lo = 0;
    const double *rot = in + b * (long long)K * (NM - 1) * 2;
    for (int k = 0; k < K; ++k) {
        L.C = NM - 1;
        L.q.load(L.C, L.cur);
        L.da = L.sdl[L.C * tpb];
        L.ia = L.sil[L.C * tpb];
        for (int j = 0; j < NM - 1; ++j) {
            L.step_q(rot[2 * j], rot[2 * j + 1]);
            --L.C;
        }
        rot += 2 * (NM - 1);
    }
    double *o = out + b * NM * NM;
    for (int s = 0; s < NM; ++s) {
        double x[Q_::NE];
        L.q.load(s, x);
        const double sc = L.sdl[s * tpb];
        for (int r = 0; r < NM; ++r)
            o[s * NM + r] = x[r] * sc;
    }
}

int op_shape(int op, int dtype, int &in_per, int &out_per)
{
    switch (op) {
    case BSTQ_DIAG_RCP:
    case BSTQ_DIAG_SQRT:
    case BSTQ_DIAG_RSQRT:
    case BSTQ_DIAG_HYP1:
        in_per = 1;
        out_per = 1;
        return 0;
    case BSTQ_DIAG_DIV:
        in_per = 2;
        out_per = 1;
        return 0;
    case BSTQ_DIAG_LARTG:
        in_per = 2;
        out_per = 3;
        return 0;
    case BSTQ_DIAG_LARTG_FAST:
        in_per = 2;
        out_per = 3;
        return dtype == BSTQ_F64 ? 0 : -1;
    case BSTQ_DIAG_SHIFT:
        in_per = 3;
        out_per = 4;
        return 0;
    case BSTQ_DIAG_PASS_STATIC:
    case BSTQ_DIAG_PASS_DYN_EXP:
    case BSTQ_DIAG_PASS_DYN_PG:
        in_per = kPassIn;
        out_per = kPassOut;
        return 0;
    case BSTQ_DIAG_FASTQ:
        in_per = 0;  // 30 K values per problem
        out_per = kDiagNM * kDiagNM;
        return dtype == BSTQ_F64 ? 0 : -1;
    default:
        return -1;
    }
}

}  // namespace

bool diag_uses_work(int op)
{
    return op == BSTQ_DIAG_PASS_DYN_EXP || op == BSTQ_DIAG_PASS_DYN_PG || op == BSTQ_DIAG_FASTQ;
}

int diag_check_op(int op, int f64)
{
    int ip, opp;
    return op_shape(op, f64 ? BSTQ_F64 : BSTQ_F32, ip, opp);
}

size_t diag_work_bytes(int op, int f64, long long count)
{
    if (!diag_uses_work(op))
        return 16;
    const long long blocks = (count + kDiagTpb - 1) / kDiagTpb;
    const size_t elem = f64 ? 8 : 4;
    // DynQ: NM columns of NM rows (padded to 16-byte vectors) per thread
    const size_t rows = ((kDiagNM * elem + 15) / 16) * 16 / elem;
    const size_t w = (size_t)blocks * kDiagTpb * kDiagNM * rows * elem;
    return w ? w : 16;
}

cudaError_t launch_diag(int op, int f64, long long count, int arg, const void *in, void *out, void *work,
                        cudaStream_t st)
{
    const long long blocks = (count + kDiagTpb - 1) / kDiagTpb;
    const dim3 grid((unsigned)blocks), block(kDiagTpb);
    const size_t elem = f64 ? 8 : 4;
    switch (op) {
    case BSTQ_DIAG_PASS_STATIC: {
        const size_t smem = (size_t)(kDiagTpb / 32) * 2 * kDiagNM * 32 * elem;
        if (f64)
            diag_pass_static<double><<<grid, block, smem, st>>>(count, (const double *)in, (double *)out);
        else
            diag_pass_static<float><<<grid, block, smem, st>>>(count, (const float *)in, (float *)out);
        break;
    }
    case BSTQ_DIAG_PASS_DYN_EXP:
    case BSTQ_DIAG_PASS_DYN_PG: {
        const size_t smem = 4 * (size_t)kDiagNM * kDiagTpb * elem;
        const int pg = op == BSTQ_DIAG_PASS_DYN_PG;
        if (f64)
            diag_pass_dyn<double><<<grid, block, smem, st>>>(count, pg, (const double *)in, (double *)out, work);
        else
            diag_pass_dyn<float><<<grid, block, smem, st>>>(count, pg, (const float *)in, (float *)out, work);
        break;
    }
    case BSTQ_DIAG_FASTQ: {
        const size_t smem = 4 * (size_t)kDiagNM * kDiagTpb * 8;
        diag_fastq<<<grid, block, smem, st>>>(count, arg, (const double *)in, (double *)out, work);
        break;
    }
    default:
        if (f64)
            diag_scalar<double><<<grid, block, 0, st>>>(op, count, (const double *)in, (double *)out);
        else
            diag_scalar<float><<<grid, block, 0, st>>>(op, count, (const float *)in, (float *)out);
        break;
    }
    return cudaGetLastError();
}

}  // namespace bstq
