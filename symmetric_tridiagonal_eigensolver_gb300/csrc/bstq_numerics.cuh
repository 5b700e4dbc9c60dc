// Device building blocks of the steqr iteration: machine constants, Newton-
// Raphson reciprocal / square-root kernels, lartg, and the copysign shift
// together with the 2x2 direct solve.
//
// Sources: BatchLAS page "algo_steqr" (deflation criterion, scaling, shift,
// Givens rotation, EXP update, 2x2 solve) and BatchLAS page "perf_steqr",
// section "CTA STEQR: chase micro-structure decisions" (hardware reciprocal
// square root plus one Newton step; the g = 0 case returns (1, 0, f) through
// a final select so identity rotations do not diverge).
//
// The division, reciprocal and square-root helpers here are our own
// Newton-Raphson refinements of the hardware approximations (rcp.approx,
// rsqrt.approx); the solver only needs them to be accurate to about an ulp
// and deterministic, not correctly rounded.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bstq {

// Machine constants (LAPACK convention; the pages name but do not define
// them): eps = unit roundoff, safmin = smallest normal, ssfmax =
// sqrt(1/safmin)/3, ssfmin = sqrt(safmin)/eps^2.
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
};

template <>
struct Consts<double> {
    static constexpr double eps = 0x1p-53;
    static constexpr double eps2 = 0x1p-106;
    static constexpr double safmin = 0x1p-1022;
    static constexpr double ssfmax = 0x1p511 / 3.0;
    static constexpr double ssfmin = 0x1p-405;
    static constexpr double prescale = 0x1p53;
};

__device__ __forceinline__ float dabs(float x) { return fabsf(x); }
__device__ __forceinline__ double dabs(double x) { return fabs(x); }

// ---------------------------------------------------------------------------
// Reciprocal square root of a normal, finite x > 0.
// float: hardware approximation (relative error below 2^-22) and one
// Newton-Raphson step y <- y + y (1 - x y^2) / 2.  Every caller passes a
// normal number, so the flush-to-zero form serves (19 cycles of latency on
// GB300 against 40 for the form that accepts subnormal operands).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float rsqrt_nr(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// Reciprocal of a normal x: hardware approximation, then Newton-Raphson
// y <- y (2 - x y) (float) or the third-order step y <- y (1 + e + e^2),
// e = 1 - x y (double).
__device__ __forceinline__ float rcp_nr(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    float e = fmaf(-x, y, 1.0f);
    return fmaf(y, e, y);
}
__device__ __forceinline__ double rcp_nr(double x)
{
    double y;
    asm("rcp.approx.ftz.f64 %0, %1;" : "=d"(y) : "d"(x));
    double e = fma(-x, y, 1.0);
    double e2 = fma(e, e, e);
    return fma(y, e2, y);
}

// a / b: quotient from the reciprocal plus one residual correction
// q + (a - b q) / b.
template <typename T>
__device__ __forceinline__ T div_nr(T a, T b)
{
    T y = rcp_nr(b);
    T q = a * y;
    T r = fma(-b, q, a);
    return fma(r, y, q);
}

// sqrt(x) for a normal, finite x > 0: s = x rsqrt(x) with one correction
// s + (x - s^2) / (2 s).
template <typename T>
__device__ __forceinline__ T sqrt_nr(T x)
{
    T y = rsqrt_nr(x);
    T s = x * y;
    T r = fma(-s, s, x);
    return fma(T(0.5) * y, r, s);
}

// sqrt(1 + x^2) without overflow, branch free: with w = max(1, |x|) and
// v = min(1, |x|), it equals w sqrt(1 + (v/w)^2).
template <typename T>
__device__ __forceinline__ T hyp1(T x)
{
    T ax = dabs(x);
    T w = fmax(T(1), ax);
    T v = fmin(T(1), ax);
    T q = div_nr(v, w);
    return w * sqrt_nr(fma(q, q, T(1)));
}

// ---------------------------------------------------------------------------
// lartg: G(c,s) = [[c,-s],[s,c]] with G^T [f; g] = [r; 0], r = hypot(f, g);
// g == 0 returns (1, 0, f) through a final select (page "perf_steqr":
// identity rotations must not diverge).
//
// float: branch free.  f and g are multiplied by the power of two 2^-k that
// brings max(|f|, |g|) into [1, 2) (k read from the exponent field on the
// integer pipe), so the sum of squares can neither overflow nor underflow;
// c and s follow from one reciprocal square root, and r = f c + g s (which
// equals (f^2 + g^2) / r) needs no scale-back.  A guarded fast path with a
// rare scaled branch measured slower here: the branch splits the unrolled
// chase into one basic block per position, so the eigenvector update of one
// position can no longer overlap the dependency chain of the next.
// double: the exponent arithmetic likewise runs on the integer pipe, which
// is idle next to the FP64 pipe.
// ---------------------------------------------------------------------------
// Requires max(|f|, |g|) < 2^126 (entries of a scaled block are below
// 2^65).
__device__ __forceinline__ void lartg(float f, float g, float &c, float &s, float &r)
{
    // exponent field of max(|f|, |g|, 2^-126) in place
    const float mx = fmaxf(fmaxf(fabsf(f), fabsf(g)), 0x1p-126f);
    const unsigned eb = __float_as_uint(mx) & 0x7f800000u;
    const float sc = __uint_as_float(0x7f000000u - eb);  // 2^(127 - exponent)
    const float fs = f * sc, gs = g * sc;
    const float r2 = fmaf(fs, fs, gs * gs);
    const float y = rsqrt_nr(r2);
    c = fs * y;
    s = gs * y;
    r = fmaf(f, c, g * s);
    const bool z = g == 0.0f;
    c = z ? 1.0f : c;
    s = z ? 0.0f : s;
    r = z ? f : r;
}

// double, FP64-lean: r2 = f^2 + g^2 directly while its exponent (read on the
// integer pipe) is comfortably inside the normal range, else (a rare,
// divergent branch) the scaled form below.
__device__ __forceinline__ void lartg_scaled(double f, double g, double &c, double &s, double &r);

__device__ __forceinline__ void lartg_fast(double f, double g, double &c, double &s, double &r)
{
    const double r2 = fma(f, f, g * g);
    const int ex = (__double2hiint(r2) >> 20) & 0x7ff;
    const double y = rsqrt_nr(r2);
    c = f * y;
    s = g * y;
    r = r2 * y;
    if (ex < 64 || ex > 1983)
        lartg_scaled(f, g, c, s, r);
    const bool z = (((unsigned)__double2hiint(g) & 0x7fffffffu) | (unsigned)__double2loint(g)) == 0u;
    c = z ? 1.0 : c;
    s = z ? 0.0 : s;
    r = z ? f : r;
}

__device__ __forceinline__ void lartg(double f, double g, double &c, double &s, double &r)
{
    lartg_scaled(f, g, c, s, r);
}

__device__ __forceinline__ void lartg_scaled(double f, double g, double &c, double &s, double &r)
{
    const unsigned fh = (unsigned)__double2hiint(f) & 0x7fffffffu;
    const unsigned gh = (unsigned)__double2hiint(g) & 0x7fffffffu;
    int ew = (int)(max(fh, gh) >> 20);
    ew = min(max(ew, 1), 2045);
    const double sc = __hiloint2double((2046 - ew) << 20, 0);  // 2^(1023-ew)
    const double isc = __hiloint2double(ew << 20, 0);          // 2^(ew-1023)
    const double fs = f * sc, gs = g * sc;
    const double r2 = fma(fs, fs, gs * gs);
    const double y = rsqrt_nr(r2);
    c = fs * y;
    s = gs * y;
    r = (r2 * y) * isc;
    const bool z = (gh | (unsigned)__double2loint(g)) == 0u;
    c = z ? 1.0 : c;
    s = z ? 0.0 : s;
    r = z ? f : r;
}

// The leading 2x2 block (d1, e1; e1, d2) of the active block (e1 != 0, not
// negligible) gives both the copysign shift of a sweep and the rotation of a
// direct 2x2 solve (page "algo_steqr"):
//   shift:  g = (d2 - d1) / (2 e1), r = sqrt(g^2 + 1),
//           mu = d1 - e1 / (g + copysign(r, g));
//   solve:  tau = (d2 - d1) / (2 e1) = g, t = the smaller root of
//           t^2 + 2 tau t - 1 = 0, i.e. t = sgn(tau) / (|tau| + sqrt(tau^2 + 1));
//           the rotation with tangent t diagonalises the block (eigenvalues
//           d1 - t e1 and d2 + t e1).
// Both follow from delta = (d2 - d1) / 2, h = sqrt(delta^2 + e1^2) and
// q = 1 / (|delta| + h):
//   t = sgn(tau) |e1| q,   mu = d1 - e1 t = d1 - sgn(delta) e1^2 q,
// i.e. the shift is the eigenvalue of the 2x2 block nearer to d1 (multiply
// the fractions above by |e1| / |e1|).  At delta = 0 exactly, sgn(tau) is
// taken as sgn(e1) (tau = 0 / e1 carries e1's sign), so mu = d1 - |e1| as the
// copysign form gives; t = +-1 both diagonalise the block.  One square root
// and one reciprocal instead of the four of the two formulas evaluated
// separately.  e1^2 > safmin in a scaled block, so delta^2 + e1^2 is a
// normal number that does not overflow.
template <typename T>
__device__ __forceinline__ void shift_tangent(T d1, T d2, T e1, T &t, T &mu)
{
    const T dl = T(0.5) * (d2 - d1);
    const T ae = dabs(e1);
    const T h = sqrt_nr(fma(dl, dl, ae * ae));
    const T q = rcp_nr(dabs(dl) + h);
    const T at = ae * q;
    t = ((dl < T(0)) != (e1 < T(0))) ? -at : at;
    mu = fma(-e1, t, d1);
}

// (cs, sn) of the 2x2 solve from its tangent t (|t| <= 1), in the chase's
// column convention for the pair (k + 1, k), k the block's first index:
//   q_{k+1} <- cs q_{k+1} + sn q_k,  q_k <- -sn q_{k+1} + cs q_k.
template <typename T>
__device__ __forceinline__ void rot_from_tangent(T t, T &cs, T &sn)
{
    cs = rsqrt_nr(fma(t, t, T(1)));
    sn = t * cs;
}

// ---------------------------------------------------------------------------
// Packed float pairs (f32x2): two FP32 lanes per instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk2(float a, float b)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

}  // namespace bstq
