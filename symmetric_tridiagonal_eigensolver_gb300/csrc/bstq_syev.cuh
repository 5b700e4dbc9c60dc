// Fused small-n dense symmetric eigensolver ("syev"), one problem per lane.
//
// The BatchLAS pages describe a fused small-n syev kernel (page "perf_steqr":
// the device solve of steqr_cta also runs inside it; the reduction to
// tridiagonal form, the steqr solve and the back-transform share one kernel,
// so the dense matrix is read once and the eigenvectors written once).  They
// give no formulas for the reduction; this is the plain unblocked Householder
// reduction of the lower triangle:
//   for i = 0 .. n-2: the reflector H_i = I - tau v v^T (v_{i+1} = 1,
//   v_k = 0 for k <= i) annihilates A[i+2:n, i]; with p = tau A22 v and
//   w = p - (tau/2)(p^T v) v the trailing block becomes A22 - v w^T - w v^T;
//   d_i = A[i,i], e_i = the new A[i+1,i].
// Then T = Q^T A Q with Q = H_0 H_1 ... H_{n-2}, and the eigenvectors of A are
// Q times those of T: the kernel forms Q and hands it to the dynamic-position
// solve as its basis (back_transform), so the eigenvector update runs on Q.
//
// Each lane keeps its copy of the lower triangle in global scratch,
// interleaved across the block (element (r, c) of lane t at
// S[(r + c n) * blockDim + t]), so the lanes of a warp, which walk the same
// (r, c) together, touch consecutive words.
#pragma once

#include "bstq_dyn.cuh"

namespace bstq {

// Z (if WANTZ) is written interleaved like S: element (r, c) at
// Z[(r + c n) * st].
template <typename T, int NM, bool WANTZ>
__device__ void sytd2_lane(int n, const T *A, T *S, int st, T *d, T *e, T *Z)
{
    auto s_at = [&](int r, int c) -> T & { return S[(size_t)(r + c * n) * st]; };
    auto z_at = [&](int r, int c) -> T & { return Z[(size_t)(r + c * n) * st]; };
    bool bad = false;
    for (int c = 0; c < n; ++c)
        for (int r = c; r < n; ++r) {
            const T a = A[r + (size_t)c * n];
            bad |= !isfinite(a);
            s_at(r, c) = a;
        }
    if (bad) {
        // a non-finite entry poisons the problem: the solve sees a NaN
        // diagonal and returns NaN eigenpairs with info -1
        for (int i = 0; i < n; ++i)
            d[i] = T(__int_as_float(0x7fffffff));
        for (int i = 0; i + 1 < n; ++i)
            e[i] = T(0);
        return;
    }
    T tau[NM], v[NM], w[NM];
    for (int i = 0; i + 1 < n; ++i) {
        T alpha = s_at(i + 1, i);
        // norm of A[i+2:n, i], scaled by its largest entry
        T sc = T(0);
        for (int k = i + 2; k < n; ++k)
            sc = fmax(sc, dabs(s_at(k, i)));
        T xnorm = T(0);
        if (sc > T(0)) {
            T ss = T(0);
            for (int k = i + 2; k < n; ++k) {
                const T y = s_at(k, i) / sc;
                ss = fma(y, y, ss);
            }
            xnorm = sc * sqrt(ss);
        }
        T t = T(0);
        if (xnorm != T(0)) {
            const T beta = -copysign(hypot(alpha, xnorm), alpha);
            t = (beta - alpha) / beta;
            const T scal = T(1) / (alpha - beta);
            for (int k = i + 2; k < n; ++k)
                s_at(k, i) = s_at(k, i) * scal;
            alpha = beta;
        }
        e[i] = alpha;
        tau[i] = t;
        if (t != T(0)) {
            v[i + 1] = T(1);
            for (int k = i + 2; k < n; ++k)
                v[k] = s_at(k, i);
            // p = tau A22 v (symmetric A22, lower triangle stored)
            for (int r = i + 1; r < n; ++r) {
                T acc = T(0);
                for (int c = i + 1; c < n; ++c)
                    acc = fma(r >= c ? s_at(r, c) : s_at(c, r), v[c], acc);
                w[r] = t * acc;
            }
            T pv = T(0);
            for (int r = i + 1; r < n; ++r)
                pv = fma(w[r], v[r], pv);
            const T a2 = T(-0.5) * t * pv;
            for (int r = i + 1; r < n; ++r)
                w[r] = fma(a2, v[r], w[r]);
            for (int c = i + 1; c < n; ++c)
                for (int r = c; r < n; ++r)
                    s_at(r, c) = s_at(r, c) - fma(v[r], w[c], w[r] * v[c]);
        }
        d[i] = s_at(i, i);
    }
    d[n - 1] = s_at(n - 1, n - 1);
    if constexpr (WANTZ) {
        // Q = H_0 (H_1 (... H_{n-2})): the identity, then the reflectors
        // left-applied last to first; H_i changes rows and columns i+1..
        for (int c = 0; c < n; ++c)
            for (int r = 0; r < n; ++r)
                z_at(r, c) = r == c ? T(1) : T(0);
        for (int i = n - 2; i >= 0; --i) {
            if (tau[i] == T(0))
                continue;
            v[i + 1] = T(1);
            for (int k = i + 2; k < n; ++k)
                v[k] = s_at(k, i);
            for (int c = i + 1; c < n; ++c) {
                T sum = T(0);
                for (int r = i + 1; r < n; ++r)
                    sum = fma(v[r], z_at(r, c), sum);
                sum = sum * tau[i];
                for (int r = i + 1; r < n; ++r)
                    z_at(r, c) = fma(-sum, v[r], z_at(r, c));
            }
        }
    }
}

// p.A: batch x n x n dense input (column-major per problem, lower triangle
// read); p.d: the eigenvalues out; p.e: batch x (n-1) scratch for the
// off-diagonal; p.Q: the eigenvectors out (jobz V); p.sscr: per block
// 2 n^2 x blockDim elements, the reduction's copy of A, then Q of the
// reduction (both interleaved), which the solve takes as its basis.
template <typename T, int NM, bool WANTZ, int SCHED>
__global__ void syev_kernel(KParams p)
{
    const int tpb = blockDim.x;
    const long long b = (long long)blockIdx.x * tpb + threadIdx.x;
    const int n = p.n;
    if (b < p.batch) {
        T *S = reinterpret_cast<T *>(p.sscr) + (size_t)blockIdx.x * 2 * n * n * tpb + threadIdx.x;
        sytd2_lane<T, NM, WANTZ>(n, reinterpret_cast<const T *>(p.A) + b * (long long)n * n, S, tpb,
                                 reinterpret_cast<T *>(p.d) + b * n,
                                 reinterpret_cast<T *>(const_cast<void *>(p.e)) + b * (n - 1),
                                 S + (size_t)n * n * tpb);
    }
    KParams q = p;
    q.back = WANTZ ? 2 : 0;  // basis from the interleaved scratch
    dyn_body<T, NM, WANTZ, SCHED>(q);
}

}  // namespace bstq
