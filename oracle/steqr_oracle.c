/*
 * CPU oracle for the batched symmetric tridiagonal eigensolver.
 *
 * TEST INFRASTRUCTURE ONLY: this file is built into liboracle.so and is
 * loaded by the tests, by the package entry's smoke check and by the
 * benchmark's CPU-baseline leg.  No product code path links or calls it.
 * It shares no source with the CUDA library.
 *
 * The algorithm (one problem per call, plain loops) lives in
 * steqr_oracle_impl.h and is instantiated here in float and in double; each
 * precision runs in its own arithmetic, as the BatchLAS pages run steqr in
 * the problem's type.  Build with -O2 -ffp-contract=off (no FMA contraction).
 *
 * Machine constants (the pages name eps, safmin, ssfmax and ssfmin without
 * defining them; LAPACK convention):
 *   eps    = unit roundoff (2^-24, 2^-53)
 *   safmin = smallest normal number (2^-126, 2^-1022), safmax = 1 / safmin
 *   ssfmax = sqrt(safmax) / 3,  ssfmin = sqrt(safmin) / eps^2
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>

/* Largest problem size (the buffers of one problem live on the stack). */
#define ORACLE_MAX_N 128

#define R_PRESCALE_F32 16777216.0f             /* 2^24 */
#define R_PRESCALE_F64 9007199254740992.0      /* 2^53 */

/* ---------------- float ---------------- */
#define real_t float
#define FN(x) x##_f32
#define R_ABS fabsf
#define R_SQRT sqrtf
#define R_COPYSIGN copysignf
#define R_EPS 0x1p-24f
#define R_SAFMIN 0x1p-126f
#define R_SSFMAX (0x1p63f / 3.0f)
#define R_SSFMIN 0x1p-15f
#define R_PRESCALE R_PRESCALE_F32
#include "steqr_oracle_impl.h"
#undef real_t
#undef FN
#undef R_ABS
#undef R_SQRT
#undef R_COPYSIGN
#undef R_EPS
#undef R_SAFMIN
#undef R_SSFMAX
#undef R_SSFMIN
#undef R_PRESCALE

/* ---------------- double ---------------- */
#define real_t double
#define FN(x) x##_f64
#define R_ABS fabs
#define R_SQRT sqrt
#define R_COPYSIGN copysign
#define R_EPS 0x1p-53
#define R_SAFMIN 0x1p-1022
#define R_SSFMAX (0x1p511 / 3.0)
#define R_SSFMIN 0x1p-405
#define R_PRESCALE R_PRESCALE_F64
#include "steqr_oracle_impl.h"
#undef real_t
#undef FN
#undef R_ABS
#undef R_SQRT
#undef R_COPYSIGN
#undef R_EPS
#undef R_SAFMIN
#undef R_SSFMAX
#undef R_SSFMIN
#undef R_PRESCALE

/* Constants as used above, exported so tests can check them against their
 * definitions. index: 0 eps, 1 safmin, 2 ssfmax, 3 ssfmin */
double oracle_constant(int dtype, int which)
{
    if (dtype == 0) {
        const float v[4] = {0x1p-24f, 0x1p-126f, 0x1p63f / 3.0f, 0x1p-15f};
        return (which >= 0 && which < 4) ? (double)v[which] : NAN;
    }
    const double v[4] = {0x1p-53, 0x1p-1022, 0x1p511 / 3.0, 0x1p-405};
    return (which >= 0 && which < 4) ? v[which] : NAN;
}
