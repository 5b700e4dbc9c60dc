// Device building blocks of the steqr iteration: machine constants, the
// reciprocal square root, lartg, the copysign shift and the 2x2 direct solve.
//
// Sources: BatchLAS page "algo_steqr" (deflation criterion, scaling, shift,
// Givens rotation, EXP update, 2x2 solve) and BatchLAS page "perf_steqr",
// section "CTA STEQR: chase micro-structure decisions" (rsqrt + one Newton
// step, range guard, g = 0 select).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bstq {

// Machine constants (LAPACK convention; the pages name but do not define
// them): eps = unit roundoff, safmin = smallest normal, ssfmax =
// sqrt(1/safmin)/3, ssfmin = sqrt(safmin)/eps^2.  The lartg fast path is
// valid while max(|f|,|g|) lies in (sqrt(safmin), sqrt(safmax/2)).
template <typename T>
struct Consts;

template <>
struct Consts<float> {
    static constexpr float eps = 0x1p-24f;
    static constexpr float eps2 = 0x1p-48f;
    static constexpr float safmin = 0x1p-126f;
    static constexpr float ssfmax = 0x1p63f / 3.0f;
    static constexpr float ssfmin = 0x1p-15f;
    static constexpr float prescale = 0x1p24f;
    static constexpr float rt_lo = 0x1p-63f;
    static constexpr float rt_hi = 6.5219089e18f;  // just below 2^62.5
};

template <>
struct Consts<double> {
    static constexpr double eps = 0x1p-53;
    static constexpr double eps2 = 0x1p-106;
    static constexpr double safmin = 0x1p-1022;
    static constexpr double ssfmax = 0x1p511 / 3.0;
    static constexpr double ssfmin = 0x1p-405;
    static constexpr double prescale = 0x1p53;
    static constexpr double rt_lo = 0x1p-511;
    static constexpr double rt_hi = 4.7403759540545887e153;  // just below 2^510.5
};

__device__ __forceinline__ float dabs(float x) { return fabsf(x); }
__device__ __forceinline__ double dabs(double x) { return fabs(x); }

// 1/sqrt(x) for a normal, finite x > 0.
// float: hardware approximation (rel. error < 2^-22) plus one Newton-Raphson
// step y <- y + y (1 - x y^2) / 2, as perf_steqr describes.
__device__ __forceinline__ float rsqrt_nr(float x)
{
    float y;
    asm("rsqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    float h = x * y;
    float u = fmaf(-h, y, 1.0f);  // 1 - x y^2
    return fmaf(0.5f * y, u, y);
}

// double: hardware approximation refined by one third-order step of the
// series (1 - u)^(-1/2) = 1 + u/2 + 3u^2/8 + ..., u = 1 - x y^2
// (Householder's method of order 3 for f(y) = y^-2 - x), which triples the
// number of correct bits.
__device__ __forceinline__ double rsqrt_nr(double x)
{
    double y;
    asm("rsqrt.approx.ftz.f64 %0, %1;" : "=d"(y) : "d"(x));
    double h = x * y;
    double u = fma(-h, y, 1.0);
    double w = fma(0.375, u, 0.5);
    double v = u * w;
    return fma(y, v, y);
}

// sqrt(1 + x^2) without overflow for large |x|.
template <typename T>
__device__ __forceinline__ T hyp1(T x)
{
    T ax = dabs(x);
    if (ax <= T(1))
        return sqrt(T(1) + ax * ax);
    T y = T(1) / ax;
    return ax * sqrt(T(1) + y * y);
}

// lartg: G(c,s) = [[c,-s],[s,c]] with G^T [f; g] = [r; 0].
// g == 0 gives (1, 0, f) through a final select (no early return).
// In-range inputs use r2 = f^2 + g^2, y = rsqrt(r2): c = f y, s = g y,
// r = r2 y.  Anything else (including NaN) takes the max-scaled formula.
template <typename T>
__device__ __forceinline__ void lartg(T f, T g, T &c, T &s, T &r)
{
    T w = fmax(dabs(f), dabs(g));
    T r2 = fma(f, f, g * g);
    T y = rsqrt_nr(r2);
    c = f * y;
    s = g * y;
    r = r2 * y;
    if (!(w > Consts<T>::rt_lo && w < Consts<T>::rt_hi)) {
        T z = fmin(dabs(f), dabs(g)) / w;
        T h = w * sqrt(T(1) + z * z);
        c = f / h;
        s = g / h;
        r = h;
    }
    if (g == T(0)) {
        c = T(1);
        s = T(0);
        r = f;
    }
}

// Copysign shift from the 2x2 block (d1, e1; e1, d2) at the converging end:
// g = (d2 - d1) / (2 e1), r = sqrt(g^2 + 1), mu = d1 - e1 / (g + copysign(r, g)).
template <typename T>
__device__ __forceinline__ T wilkinson_shift(T d1, T d2, T e1)
{
    T g = (d2 - d1) / (T(2) * e1);
    T r = hyp1(g);
    return d1 - e1 / (g + copysign(r, g));
}

// Direct solve of the 2x2 block [[a, b], [b, c2]] (b != 0): the rotation
// with tangent t, the smaller root of t^2 + 2 tau t - 1 = 0,
// tau = (c2 - a) / (2 b), diagonalises it; the eigenvalues are a - t b and
// c2 + t b.  Returns them with (cs, sn) of that rotation written in the
// chase's column convention for the pair (k + 1, k):
//   q_{k+1} <- cs q_{k+1} + sn q_k,  q_k <- -sn q_{k+1} + cs q_k.
template <typename T>
__device__ __forceinline__ void solve2x2(T a, T b, T c2, T &lam_lo, T &lam_hi, T &cs, T &sn)
{
    T tau = (c2 - a) / (T(2) * b);
    T sgn = tau < T(0) ? T(-1) : T(1);
    T t = sgn / (dabs(tau) + hyp1(tau));
    T cq = T(1) / hyp1(t);
    lam_lo = a - t * b;
    lam_hi = c2 + t * b;
    cs = cq;
    sn = t * cq;
}

}  // namespace bstq
