// Leaf solve of divide and conquer (BatchLAS pages "algo_steqr": the leaf
// solve of stedc, and "perf_steqr": steqr_cta also runs at the stedc leaves).
//
// A size-n problem is cut into consecutive leaves of `leaf` rows (the
// remainder, if any, is a last and shorter leaf).  At every boundary between
// rows r-1 | r the off-diagonal beta = e[r-1] is torn off as a rank-one term:
// T = diag(T_1, T_2) + |beta| v v^T, v = e_{r-1} + sign(beta) e_r, so each
// leaf is T's diagonal block with |beta| subtracted from the two diagonal
// entries next to the boundary (left boundary first, then right, in the
// problem's precision).  The leaves are then solved as ordinary batched
// problems by the steqr kernels of this library.
//
// This file holds the two memory-bound kernels around those solves:
//   tear   d, e (batch x n, batch x (n-1))  ->  leaf d', e' grouped by leaf
//          size (all full leaves problem-major, then all tail leaves), the
//          layout the batched solve reads;
//   gather leaf eigenvalues back to each leaf's rows of d, and the solves'
//          per-leaf status to info[batch][leaves].
// Both are one thread per row of d in a grid-stride loop: coalesced reads of
// d and e, contiguous writes per problem.
#include <cuda_runtime.h>

#include <stdint.h>

#include "bstq_leaves.h"

namespace bstq {
namespace {

__device__ __forceinline__ float absv(float x) { return fabsf(x); }
__device__ __forceinline__ double absv(double x) { return fabs(x); }

struct LeafShape {
    long long batch;
    int n, L, nfull, t;
};

// Row g of the batch -> (problem b, row i).  I is the index type: 32-bit
// unsigned where batch * n fits (its division is a short sequence; the
// 64-bit one is a long software routine that dominated these kernels).
template <typename T, typename I>
__global__ void tear_kernel(LeafShape s, const T *__restrict__ d, const T *__restrict__ e, T *__restrict__ dfull,
                            T *__restrict__ efull, T *__restrict__ dtail, T *__restrict__ etail)
{
    const I total = (I)(s.batch * s.n);
    const I step = (I)gridDim.x * blockDim.x;
    const I nn = (I)s.n;
    for (I g = (I)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += step) {
        const long long b = (long long)(g / nn);
        const int i = (int)(g - (I)b * nn);
        const int k = i / s.L;
        const int j = i - k * s.L;
        const bool full = k < s.nfull;
        const int nk = full ? s.L : s.t;
        const T *eb = e + b * (s.n - 1);
        T x = d[(long long)g];
        if (j == 0 && i > 0)
            x = x - absv(eb[i - 1]);
        if (j == nk - 1 && i < s.n - 1)
            x = x - absv(eb[i]);
        if (full) {
            const long long leaf = b * s.nfull + k;
            dfull[leaf * s.L + j] = x;
            if (j < s.L - 1)
                efull[leaf * (s.L - 1) + j] = eb[i];
        } else {
            dtail[b * s.t + j] = x;
            if (j < s.t - 1)
                etail[b * (s.t - 1) + j] = eb[i];
        }
    }
}

template <typename T, typename I>
__global__ void gather_kernel(LeafShape s, T *__restrict__ d, const T *__restrict__ dfull,
                              const T *__restrict__ dtail, const int *__restrict__ info_full,
                              const int *__restrict__ info_tail, int *__restrict__ info)
{
    const I total = (I)(s.batch * s.n);
    const I step = (I)gridDim.x * blockDim.x;
    const I nn = (I)s.n;
    const int leaves = s.nfull + (s.t > 0 ? 1 : 0);
    for (I g = (I)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += step) {
        const long long b = (long long)(g / nn);
        const int i = (int)(g - (I)b * nn);
        const int k = i / s.L;
        const int j = i - k * s.L;
        if (k < s.nfull) {
            const long long leaf = b * s.nfull + k;
            d[(long long)g] = dfull[leaf * s.L + j];
            if (j == 0)
                info[b * leaves + k] = info_full[leaf];
        } else {
            d[(long long)g] = dtail[b * s.t + j];
            if (j == 0)
                info[b * leaves + k] = info_tail[b];
        }
    }
}

constexpr int kLeafThreads = 256;

// 32-bit indexing needs total rows plus one grid stride below 2^32.
bool fits32(long long total, long long grid)
{
    return total + grid * kLeafThreads < (1LL << 32);
}

long long leaf_grid(long long total, int sms)
{
    // enough blocks to fill every SM a few times over, no more than the rows
    const long long want = (long long)(sms > 0 ? sms : 152) * 8;
    const long long need = (total + kLeafThreads - 1) / kLeafThreads;
    return need < want ? need : want;
}

}  // namespace

cudaError_t launch_leaf_tear(int f64, long long batch, int n, int L, const void *d, const void *e, void *dfull,
                             void *efull, void *dtail, void *etail, int sms, cudaStream_t st)
{
    LeafShape s{batch, n, L, n / L, n % L};
    const long long grid = leaf_grid(batch * n, sms);
    if (grid <= 0)
        return cudaSuccess;
    const bool w32 = fits32(batch * n, grid);
    if (f64 && w32)
        tear_kernel<double, unsigned><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (const double *)d, (const double *)e, (double *)dfull, (double *)efull, (double *)dtail,
            (double *)etail);
    else if (f64)
        tear_kernel<double, unsigned long long><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (const double *)d, (const double *)e, (double *)dfull, (double *)efull, (double *)dtail,
            (double *)etail);
    else if (w32)
        tear_kernel<float, unsigned><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (const float *)d, (const float *)e, (float *)dfull, (float *)efull, (float *)dtail,
            (float *)etail);
    else
        tear_kernel<float, unsigned long long><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (const float *)d, (const float *)e, (float *)dfull, (float *)efull, (float *)dtail,
            (float *)etail);
    return cudaGetLastError();
}

cudaError_t launch_leaf_gather(int f64, long long batch, int n, int L, void *d, const void *dfull,
                               const void *dtail, const int *info_full, const int *info_tail, int *info, int sms,
                               cudaStream_t st)
{
    LeafShape s{batch, n, L, n / L, n % L};
    const long long grid = leaf_grid(batch * n, sms);
    if (grid <= 0)
        return cudaSuccess;
    const bool w32 = fits32(batch * n, grid);
    if (f64 && w32)
        gather_kernel<double, unsigned><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (double *)d, (const double *)dfull, (const double *)dtail, info_full, info_tail, info);
    else if (f64)
        gather_kernel<double, unsigned long long><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (double *)d, (const double *)dfull, (const double *)dtail, info_full, info_tail, info);
    else if (w32)
        gather_kernel<float, unsigned><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (float *)d, (const float *)dfull, (const float *)dtail, info_full, info_tail, info);
    else
        gather_kernel<float, unsigned long long><<<(unsigned)grid, kLeafThreads, 0, st>>>(
            s, (float *)d, (const float *)dfull, (const float *)dtail, info_full, info_tail, info);
    return cudaGetLastError();
}

}  // namespace bstq
