/*
 * bstq — batched symmetric tridiagonal eigensolver for one NVIDIA GB300
 * (sm_103a).  C ABI.
 *
 * The operation (BatchLAS page "algo_steqr", problem statement): for each of
 * `batch` independent matrices T = tridiag(e_1..e_{n-1}; d_1..d_n) compute
 * T = Q Lambda Q^T with Lambda = diag(lambda_1 <= ... <= lambda_n) and, when
 * eigenvectors are requested, the orthogonal Q.  The method is implicit
 * shifted QL/QR with a Givens bulge chase ("steqr"): relative deflation
 * |e_i|^2 <= eps^2 |d_i||d_{i+1}| + safmin, per-block infinity-norm scaling
 * against ssfmax/ssfmin, the copysign 2x2 shift, lartg rotations with the
 * explicit (EXP) similarity update, direct 2x2 solves and a final ascending
 * sort (all on the "algo_steqr" page; the lane/warp scheduling choices follow
 * the BatchLAS page "perf_steqr").
 *
 * Layout (all arrays dense, row-major over the batch):
 *   d : batch x n        d[b*n + i]            = d_{i+1} of problem b
 *   e : batch x (n-1)    e[b*(n-1) + i]        = e_{i+1} of problem b
 *   Q : batch x n x n    Q[b*n*n + j*n + i]    = Q_{ij}  (column-major per
 *                        problem; column j is the eigenvector of lambda_j)
 *
 * Memory and streams: every pointer of bstq_solve / bstq_solve_ex is caller-
 * owned DEVICE memory.  The library allocates nothing, never synchronises and
 * only enqueues work on the given stream; calls are thread-safe.  All
 * results are valid once the stream reaches them.
 *
 * Errors: functions return 0 on success; -k when argument k (1-based) is
 * invalid; BSTQ_ERR_CUDA (> 0) when a CUDA launch or copy failed (the CUDA
 * error text is then available from bstq_last_error); BSTQ_ERR_NODEVICE when no
 * usable sm_103 device is current.  No C++ exception crosses the ABI.
 * batch == 0 is a no-op returning 0.
 *
 * Per-problem status (int32 info[b], first bytes of `work`):
 *    0  converged;
 *   k>0 the sweep budget (max_sweeps_per_n * n implicit steps) ran out with
 *       k off-diagonal entries still nonzero; d and Q hold the current,
 *       unsorted state of that problem;
 *   -1  the input had a NaN or Inf; every lambda and every Q entry of that
 *       problem is NaN.
 */
#ifndef BSTQ_H
#define BSTQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { BSTQ_F32 = 0, BSTQ_F64 = 1 } bstq_dtype;
typedef enum { BSTQ_JOBZ_N = 0, BSTQ_JOBZ_V = 1 } bstq_jobz;

/* Sweep scheduler within a warp (BatchLAS "perf_steqr", sections "Lockstep
 * flat solver" and "What ships").  NESTED: each problem runs its own loop
 * nest.  FLAT: all problems of a warp settle, then chase together.  Both run
 * the same per-problem operation sequence, so results are equal. */
typedef enum {
    BSTQ_SCHED_AUTO = 0,
    BSTQ_SCHED_FLAT = 1,
    BSTQ_SCHED_NESTED = 2
} bstq_scheduler;

/* Where the working copy of Q lives while rotations accumulate. */
typedef enum {
    BSTQ_QSTORE_AUTO = 0,
    BSTQ_QSTORE_REGISTERS = 1, /* whole Q in registers (small n)         */
    BSTQ_QSTORE_SHARED = 2,    /* per-lane columns in shared memory      */
    BSTQ_QSTORE_GLOBAL = 3,    /* per-lane columns in `work` (L1/L2)     */
    BSTQ_QSTORE_HYBRID = 4,    /* 8 rows in registers, rest in shared    */
    BSTQ_QSTORE_SPLIT = 5,     /* float, n <= 32: separate warps apply the
                                  rotations to Q held in their registers */
    BSTQ_QSTORE_LOG = 6        /* float, n > 32, flat scheduler (the
                                  default there): each lane logs its
                                  problem's rotations in `work`; the warp
                                  then applies each log to Q rows held in
                                  registers (record and apply) */
} bstq_qstore;

/* Options; an all-zero struct means the defaults. */
typedef struct {
    int no_sort;           /* 0: ascending lambda, Q columns permuted (default)
                              1: leave eigenpairs in converged order        */
    int max_sweeps_per_n;  /* 0 -> 30: budget = value * n implicit steps     */
    int scheduler;         /* bstq_scheduler                                 */
    int qstore;            /* bstq_qstore                                    */
    int threads_per_block; /* 0 = chosen by the library; else a multiple of
                              32 in [32, 1024]                               */
    int kernel;            /* bstq_kernel: 0 = chosen per (dtype, jobz, n)   */
    int back_transform;    /* 0 (default): Q starts as the identity.
                              1 (jobz == V only): Q is in/out.  On entry it
                              holds a basis Z per problem (same layout as the
                              output, Q[b*n*n + j*n + i] = Z_ij); the
                              rotations are right-applied to it, so on exit
                              it holds Z times the eigenvectors of T, sorted
                              with lambda (BatchLAS page "algo_steqr",
                              eigenvector accumulation: back_transform).     */
    int update_scheme;     /* bstq_update_scheme: 0 (default) EXP, 1 PG.    */
    int log_entries;       /* BSTQ_QSTORE_LOG only: rotation log entries per
                              problem (8 bytes each, in `work`), rounded up
                              to whole pages of 256; 0 = 1.5 n^2 + 8n, which
                              holds a typical solve in one apply round.  A
                              smaller log needs less workspace and costs
                              more rounds (Q goes through global memory once
                              per round); negative values return -10.       */
} bstq_params;

/* Form of the implicit step (BatchLAS page "algo_steqr", update schemes).
 * EXP writes each local similarity G^T T G out; PG propagates the scalars
 * (g, p, c, s) across the sweep.  Both perform the same implicit step.  PG
 * runs in the dynamic-position kernels: with kernel = AUTO it selects them,
 * with kernel = STATIC it returns -10. */
typedef enum {
    BSTQ_UPDATE_EXP = 0,
    BSTQ_UPDATE_PG = 1
} bstq_update_scheme;

/* Kernel family.  STATIC: d and e in registers, the chase unrolled over
 * compile-time positions (Q in registers, shared or global memory per
 * qstore).  DYNAMIC: d and e in shared memory, each lane chases its own
 * positions in a rolled loop, Q in global scratch (qstore ignored). */
typedef enum {
    BSTQ_KERNEL_AUTO = 0,
    BSTQ_KERNEL_STATIC = 1,
    BSTQ_KERNEL_DYNAMIC = 2
} bstq_kernel;

#define BSTQ_ERR_CUDA 1
#define BSTQ_ERR_NODEVICE 2
#define BSTQ_MAX_N 128

/* Bytes of device workspace bstq_solve needs for (dtype, jobz, n, batch)
 * with default parameters: int32 info[batch] at offset 0, then any scratch
 * the chosen kernel uses (aligned to 256 bytes).  Returns 0 for invalid
 * arguments. */
size_t bstq_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch);

/* Same, for explicit parameters (p may be NULL). */
size_t bstq_work_size_ex(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                         const bstq_params *p);

/*
 * Solve `batch` problems of size n (1 <= n <= 128; above 32 the dynamic-position
 * kernels run, the static family being built up to 32) on `stream`
 * (a cudaStream_t; NULL = legacy default stream).
 *   d     in/out  batch*n values of dtype; on exit the eigenvalues.
 *   e     in      batch*(n-1) values; may be NULL when n == 1.
 *   Q     out     batch*n*n values when jobz == BSTQ_JOBZ_V; ignored (may be
 *                 NULL) when jobz == BSTQ_JOBZ_N.  In/out with
 *                 p->back_transform (the basis Z on entry).
 *   work  in/out  at least bstq_work_size(...) bytes, 16-byte aligned;
 *                 receives int32 info[batch].
 * d, e and Q must be aligned to their element size.
 * Argument numbers for -k: 1 dtype, 2 jobz, 3 n, 4 batch, 5 d, 6 e, 7 Q,
 * 8 work, 10 params.
 */
int bstq_solve(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
               void *d, const void *e, void *Q, void *work, void *stream);

int bstq_solve_ex(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                  void *d, const void *e, void *Q, void *work, void *stream,
                  const bstq_params *p);

/*
 * End-to-end variant on HOST buffers: copies h_d and h_e (and h_Q with
 * p->back_transform) to the device workspace `dev`, solves there and copies
 * lambda (into h_d), Q (into h_Q, when jobz == V) and info (into h_info)
 * back, all enqueued on `stream`.
 * The host buffers are read/written asynchronously when they are pinned
 * (cudaHostAlloc / cudaHostRegister); the caller synchronises the stream
 * before reading them.  `dev` must hold bstq_host_work_size(...) bytes of
 * device memory (256-byte aligned).
 * Argument numbers for -k: 1 dtype, 2 jobz, 3 n, 4 batch, 5 h_d, 6 h_e,
 * 7 h_Q, 8 h_info, 9 dev, 11 params.
 */
size_t bstq_host_work_size(bstq_dtype dtype, bstq_jobz jobz, int n,
                           int64_t batch, const bstq_params *p);

int bstq_solve_host(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                    void *h_d, const void *h_e, void *h_Q, int32_t *h_info,
                    void *dev, void *stream, const bstq_params *p);

/*
 * Allocation-free variant of bstq_solve_ex for jobz == BSTQ_JOBZ_V (the
 * BatchLAS pages have no counterpart; this is a library convenience).
 *
 * For callers that cannot allocate device memory when they solve: code that
 * runs while a CUDA graph is being captured, inside an allocator callback, in
 * a plugin handed fixed buffers by its host framework, or in a real-time loop
 * that must never call cudaMalloc.  Instead of a caller-sized `work` buffer,
 * the eigenvector scratch lives in a 64 MiB array compiled into the library;
 * every GPU that loads the library reserves it until the process exits.
 * The call itself allocates nothing and calls no allocating routine.
 *   d, e, Q   as for bstq_solve (device memory); Q is required.
 *   info      device int32[batch], receives the per-problem status.
 *   p         optional parameters; p->qstore is ignored.  With p->kernel
 *             left at BSTQ_KERNEL_AUTO, sizes whose static-position kernel
 *             keeps Q in registers (float n <= 12, double n <= 8) run the
 *             dynamic-position kernel, which keeps Q in the scratch array;
 *             p->kernel = BSTQ_KERNEL_STATIC for those sizes returns -10.
 * Returns 0; -2 when jobz is not BSTQ_JOBZ_V; -4 when the problems need more
 * scratch than the array holds (n_pad^2 * sizeof(element) bytes per problem
 * slot, n_pad = n rounded up to 4, 8, 12, 16, 24, 32, 48, 64, 96 or 128, slots = batch rounded up to
 * the block size; e.g. about 58,000 double problems of n <= 12 fit, or 16,000
 * float problems of n <= 32); other codes as bstq_solve_ex.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * The address is kept per device ordinal for the rest of the process: it
 * belongs to the device's primary context, the one the CUDA runtime uses.
 * A caller that makes another context current on the device, or resets the
 * device (cudaDeviceReset) after the first call, must not call this entry
 * point afterwards.
 * All calls share the one array and the kernel overwrites the part it uses
 * before reading it, so nothing needs clearing between calls; calls that can
 * overlap on the GPU (different streams, or graphs replayed concurrently)
 * race on the array and must be serialised by the caller.
 */
int bstq_solve_noalloc(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                       void *d, const void *e, void *Q, int32_t *info,
                       void *stream, const bstq_params *p);

/*
 * Fused small-n dense symmetric eigensolver (BatchLAS page "perf_steqr": the
 * fused syev kernel runs the reduction to tridiagonal form, the steqr solve
 * and the back-transform in one launch).  One lane per problem: the lower
 * triangle of A is reduced by Householder reflectors (T = Q^T A Q), T is
 * solved with Q as the basis (as back_transform), so the eigenvectors come
 * out as those of A.  1 <= n <= 32.
 *   A     in      batch*n*n values, column-major per problem
 *                 (A[b*n*n + j*n + i] = A_ij); only i >= j is read.
 *   W     out     batch*n eigenvalues, ascending per problem.
 *   V     out     batch*n*n values when jobz == V (column j the eigenvector
 *                 of W[j]); ignored (may be NULL) for jobz == N.
 *   work  in/out  bstq_syev_work_size(...) bytes, 256-byte aligned; int32
 *                 info[batch] at offset 0 (0, k > 0 budget exhausted, -1 a
 *                 non-finite entry in the lower triangle).
 *   p     optional: no_sort, max_sweeps_per_n, scheduler, update_scheme and
 *                 threads_per_block apply; back_transform, qstore or a kernel
 *                 other than DYNAMIC return -10.
 * Returns 0 or -k as bstq_solve_ex (-5 A, -6 W, -7 V, -8 work, -3 n > 32).
 */
size_t bstq_syev_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                           const bstq_params *p);

int bstq_syev(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, const void *A,
              void *W, void *V, void *work, void *stream, const bstq_params *p);

/*
 * Leaf solve of divide and conquer (BatchLAS page "algo_steqr": the leaf
 * solve of stedc; page "perf_steqr": steqr_cta also runs at the stedc
 * leaves).  Each of `batch` size-n problems is cut into consecutive leaves
 * of `leaf` rows from the top (the remainder n % leaf, if any, is a last,
 * shorter leaf; leaf >= n gives one leaf).  At every leaf boundary r-1 | r
 * the coupling beta = e_r is torn off as the rank-one term |beta| v v^T,
 * v = unit_{r-1} + sign(beta) unit_r: |beta| is subtracted from the two
 * diagonal entries next to the boundary (the upper boundary of a leaf
 * first).  Every leaf is then solved as a steqr problem of its own (from
 * the identity, ascending), all leaves of the batch in one batched solve
 * (two when a shorter last leaf exists).  n >= 1, 1 <= leaf <= 128.
 *   d     in/out  batch*n values; on exit each leaf's eigenvalues, ascending
 *                 within the leaf, at the leaf's rows.
 *   e     in      batch*(n-1) values (may be NULL when n == 1).
 *   Q     out     jobz == V: the leaves' eigenvectors grouped by leaf size.
 *                 With L = min(leaf, n), F = n / L full leaves and the last
 *                 leaf of t = n % L rows: first batch*F blocks of L x L, block
 *                 (b*F + k) for leaf k of problem b, then batch blocks of
 *                 t x t, block b for problem b's last leaf; every block is
 *                 column-major (column j the eigenvector of the leaf's j-th
 *                 eigenvalue).  batch*(F*L*L + t*t) values in all.  Ignored
 *                 (may be NULL) for jobz == N.
 *   info  out     device int32[batch * leaves], leaves = F + (t > 0):
 *                 info[b*leaves + k] is leaf k's status as for bstq_solve.
 *                 A non-finite coupling beta poisons both leaves next to it.
 *   work  scratch bstq_stedc_leaves_work_size(...) bytes, 256-byte aligned.
 *   p     optional; applies to the leaf solves as in bstq_solve_ex except
 *         back_transform, which returns -10.
 * Returns 0; -1 dtype, -2 jobz, -3 n or leaf out of range, -4 batch, -5 d,
 * -6 e, -7 Q, -8 info or work NULL or misaligned, -10 parameters that no
 * leaf solve accepts; BSTQ_ERR_CUDA / BSTQ_ERR_NODEVICE as elsewhere.
 * Like every entry point it allocates nothing and only enqueues work.
 */
size_t bstq_stedc_leaves_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int leaf,
                                   int64_t batch, const bstq_params *p);

int bstq_stedc_leaves(bstq_dtype dtype, bstq_jobz jobz, int n, int leaf, int64_t batch,
                      void *d, const void *e, void *Q, int32_t *info, void *work,
                      void *stream, const bstq_params *p);

/* Description of the kernel the library would launch (for tests and
 * benchmarks): fills up to `len` bytes of `buf` with a NUL-terminated string
 * such as "lane<f32,16,V,shared,flat> tpb=224 grid=147" and returns 0, or
 * returns -k for invalid arguments as bstq_solve_ex would. */
int bstq_describe(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                  const bstq_params *p, char *buf, size_t len);

/*
 * Diagnostics: one building block of the solve, run on a table of inputs so
 * that it can be checked on its own (the tests' unit layer).  Each op calls
 * the same device code the solver kernels run.  The BatchLAS pages define
 * the blocks (page "algo_steqr": Givens rotation, copysign shift, 2x2 solve,
 * EXP and PG update schemes, eigenvector accumulation); this entry point
 * itself has no counterpart there.
 *
 * `in` and `out` are device arrays of the dtype; `count` records are
 * processed, record k at in + k * (values in) and out + k * (values out):
 *   RCP, SQRT, RSQRT, HYP1  1 -> 1   1/x, sqrt x, 1/sqrt x (x normal, > 0),
 *                                    sqrt(1 + x^2)
 *   DIV                     2 -> 1   a / b (b normal)
 *   LARTG                   2 -> 3   (f, g) -> (c, s, r), G^T [f; g] = [r; 0]
 *   LARTG_FAST (f64 only)   2 -> 3   the chase's fast double form
 *   SHIFT                   3 -> 4   (d1, d2, e1) -> (t, mu, cs, sn): the 2x2
 *                                    tangent, the copysign shift and the 2x2
 *                                    rotation of the leading block
 *   PASS_STATIC, PASS_DYN_EXP, PASS_DYN_PG    42 -> 288
 *       one pass of the chase at compile-time size 16 in the static- or
 *       dynamic-position family.  Record: n, lo, m, task (1 sweep over
 *       positions m .. lo+1, 2 the 2x2 solve at lo+1), rhi, rlo (the warp's
 *       union of positions, containing [lo+1, m]), f0, g0 (the sweep's
 *       seed: d_m - mu, e_{m-1}), cs2, sn2 (the 2x2 rotation), d[16], e[16]
 *       (integers stored as values of the dtype).  Result: d[16], e[16]
 *       after the pass, then the 16 x 16 column-major product of the pass's
 *       rotations Q, so that T_after = Q^T T_before Q.
 *   FASTQ (f64 only)        30 K -> 256
 *       the factored double eigenvector update alone: K = arg sweeps over
 *       positions 15 .. 1 of a 16 x 16 Q starting at the identity, the
 *       rotation (c, s) of sweep k, step j at values (k * 15 + j) * 2.
 *       Result: Q, column-major.
 * `work` (device, 16-byte aligned) holds bstq_diag_work_size(...) bytes for
 * PASS_DYN_* and FASTQ and may be NULL otherwise.  Returns 0; -1 unknown op
 * for the dtype, -2 dtype, -3 count, -4 arg, -5 in, -6 out, -7 work;
 * BSTQ_ERR_CUDA / BSTQ_ERR_NODEVICE as elsewhere.  Allocates nothing.
 */
typedef enum {
    BSTQ_DIAG_RCP = 1,
    BSTQ_DIAG_DIV = 2,
    BSTQ_DIAG_SQRT = 3,
    BSTQ_DIAG_RSQRT = 4,
    BSTQ_DIAG_HYP1 = 5,
    BSTQ_DIAG_LARTG = 6,
    BSTQ_DIAG_LARTG_FAST = 7,
    BSTQ_DIAG_SHIFT = 8,
    BSTQ_DIAG_PASS_STATIC = 20,
    BSTQ_DIAG_PASS_DYN_EXP = 21,
    BSTQ_DIAG_PASS_DYN_PG = 22,
    BSTQ_DIAG_FASTQ = 30
} bstq_diag_op;

size_t bstq_diag_work_size(int op, bstq_dtype dtype, int64_t count);

int bstq_diag(int op, bstq_dtype dtype, int64_t count, int arg, const void *in, void *out, void *work,
              void *stream);

/* Human-readable text for a return code. */
const char *bstq_status_string(int code);

/* Library version, e.g. "bstq 0.1.0 sm_103a". */
const char *bstq_version(void);

/* Text of the last CUDA error a bstq call on this thread returned
 * BSTQ_ERR_CUDA for ("" if none).  The pointer stays valid until the next
 * failing call on the same thread. */
const char *bstq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* BSTQ_H */
