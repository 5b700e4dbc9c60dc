// C ABI of the batched tridiagonal eigensolver: argument checks, the launch
// plan (kernel variant, block size, grid, workspace) and the launches.
#include <cuda_runtime.h>

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/bstq.h"
#include "bstq_rlog.cuh"
#include "bstq_split2.cuh"
#include "bstq_diag.h"
#include "bstq_leaves.h"
#include "bstq_plan.h"
#include "bstq_registry.h"

namespace bstq {
namespace {

struct Plan {
    const KernelEntry *k = nullptr;
    int tpb = 0;
    long long grid = 0;
    size_t smem = 0;
    size_t qwork_bytes = 0;
    size_t work_bytes = 0;
    int ppb = 0;  // problems per block (split-role kernel) or per warp (record-and-apply)
    // record-and-apply: log entries per problem, the apply and finishing
    // launches, and the offsets of the log lengths, maps and logs in work
    long long lcap = 0;
    int tpb2 = 0, tpb3 = 0;
    long long grid2 = 0, grid3 = 0;
    size_t smem2 = 0, smem3 = 0;
    size_t off_cnt = 0, off_map = 0, off_log = 0;
};

constexpr int kNmList[] = {4, 8, 12, 16, 24, 32, 48, 64, 96, 128};
constexpr int kSyevMaxN = 32;  // the fused syev kernels are built up to n = 32

thread_local char g_last_error[256] = "";

int cuda_fail(cudaError_t err, const char *what)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorString(err),
             cudaGetErrorName(err));
    return BSTQ_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct DevInfo {
    int sms = 0;
    int max_smem_block = 0;
    int max_regs_sm = 0;
    int max_threads_sm = 0;
    int major = 0, minor = 0;
};

// Device properties of the current device, cached per device ordinal.
bool dev_info(DevInfo &out)
{
    static std::mutex mu;
    static DevInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DevInfo di;
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        cache[dev] = di;
        have[dev] = true;
    }
    out = cache[dev];
    return true;
}

const KernelEntry *find_entry(int dtype, int jobz, int nm, int qs, int sched, int family)
{
    typedef const KernelEntry *(*Lister)(int *);
#define BSTQ_LISTER(name) entries_##name,
    static const Lister lists[] = {BSTQ_FOR_EACH_UNIT(BSTQ_LISTER)};
#undef BSTQ_LISTER
    for (Lister l : lists) {
        int cnt = 0;
        const KernelEntry *t = l(&cnt);
        for (int i = 0; i < cnt; ++i)
            if (t[i].dtype == dtype && t[i].jobz == jobz && t[i].nm == nm &&
                t[i].qs == (jobz ? qs : 0) && t[i].sched == sched && t[i].family == family)
                return &t[i];
    }
    return nullptr;
}

// Default Q storage, from measurement on GB300 (batch 32768, one wave):
//   float n <= 8: whole Q in registers;
//   float 9 <= n <= 16, flat scheduler: split roles (chase warps record the
//     rotations, Q warps apply them; n=16 V 0.131 vs 0.138 ms hybrid, n=12 V
//     0.072 vs 0.077 ms registers);
//   float 17 <= n <= 32, flat scheduler: split roles with each problem's Q
//     rows spread over several Q warps (bstq_split2.cuh; n = 17 V 0.219 vs
//     0.362 ms hybrid, n = 24 V 0.287 vs 0.487, n = 27 V 0.775 vs 1.70,
//     n = 32 V 0.813 vs 1.98);
//   float n <= 12 otherwise: registers; float n >= 16 otherwise: 8 rows of Q
//     in registers, the rest streamed from shared memory (one wave of 32768
//     problems stays resident);
//   double: registers for n <= 8, else global scratch (its FP64 pipe, not
//     L1/L2, bounds it);
//   float n > 32: the record-and-apply kernels (bstq_rlog.cuh; f32 V n = 64
//     3.8 against 16.9 ms with Q in global scratch, n = 128 10.7 against
//     87 ms at batch 8192).
int default_qstore(int dtype, int nm, int sched)
{
    (void)sched;
    if (dtype == 0) {
        if (nm > 32)
            return QS_LOG;
        if (nm <= 8)
            return QS_REG;
        if (nm <= 32 && sched == SCHED_FLAT)
            return QS_SPLIT;
        return nm <= 12 ? QS_REG : QS_HYBRID;
    }
    return nm <= 8 ? QS_REG : QS_GLOBAL;
}

// Rows of Q held in memory per lane (registers hold the rest), padded to
// whole 16-byte vectors.
int memory_rows(int dtype, int nm, int qs)
{
    const int w = dtype ? 2 : 4;
    const int rr = qs == QS_REG ? nm : (qs == QS_HYBRID ? kHybridRegRows : 0);
    return qs == QS_REG ? 0 : ((nm - rr + w - 1) / w) * w;
}

// Default scheduler per (dtype, jobz, compile-time size), chosen from
// measurement as the BatchLAS page "perf_steqr" (section "Lockstep flat
// solver") chooses it per (dtype, chunk).  GB300, batch 65,536 for n <= 8
// and 32,768 above, L2 flushed, medians of five interleaved rounds of 15
// steps (ms, flat against nested on the default family):
//   float n <= 4, V and N: nested (n = 3 V 0.0123 / 0.0143, n = 4 V
//     0.0164 / 0.0172, n = 4 N 0.0151 / 0.0168);
//   float 5 <= n <= 8, N: nested (n = 6 0.0246 / 0.0266; n = 5 and 8
//     equal);  V: flat (n = 5 0.0373 / 0.0389, n = 6 0.0529 / 0.0492,
//     n = 8 equal);
//   double n <= 4, V: nested, on the static-position family (n = 3 0.1024
//     against 0.1168 for the dynamic family either way, n = 4 0.1751 against
//     0.2103);
//   float n > 32, V (the record-and-apply chase, which carries no
//     eigenvector work): nested (n = 64 3.71 / 3.81 ms, n = 128 at batch
//     8192 10.16 / 10.75 ms, n = 64 at batch 4096 1.63 / 1.84 ms);
//   all other sizes: flat (float n = 12 V 0.053 / 0.062, n = 16 V
//     0.109 / 0.117, n = 32 V 1.95 / 3.39; double within 0.5 %).
int default_sched(int dtype, int jobz, int nm)
{
    if (dtype == BSTQ_F32)
        return (nm <= 4 || (nm <= 8 && !jobz) || (nm > 32 && jobz)) ? SCHED_NESTED : SCHED_FLAT;
    return (nm <= 4 && jobz) ? SCHED_NESTED : SCHED_FLAT;
}

// Default kernel family (static positions in registers, or dynamic
// positions with d and e in shared memory), per (dtype, jobz, n) from
// measurement on GB300 (batch 32768, one wave):
//   float: static at every n (n=16 V 0.137 vs 0.30 ms, n=24 V 0.58 vs
//          0.65 ms, n=32 V 2.26 vs 2.46 ms, n=32 N 0.21 vs 0.39 ms);
//   double: dynamic at every n (n=4 V 0.111 vs 0.112 ms, n=8 V 0.44 vs
//          0.53 ms, n=12 V 0.98 vs 1.31 ms, n=12 N 0.49 vs 0.51 ms):
//          FP64-bound, and the dynamic kernel has no union of position
//          ranges and a factored Q update;
//   n > 32: dynamic (the static family is built up to n = 32).
//   double n <= 4, V, under the nested scheduler: static (n = 4 V 0.175
//          against 0.210 ms; flat: 0.202 against 0.211).
int default_family(int dtype, int jobz, int nm, int sched)
{
    if (nm > 32)
        return FAMILY_DYNAMIC;  // the only family built above n = 32
    if (dtype == BSTQ_F64 && jobz && nm <= 4 && sched == SCHED_NESTED)
        return FAMILY_STATIC;
    return dtype == 0 ? FAMILY_STATIC : FAMILY_DYNAMIC;
}

int check_args(int dtype, int jobz, int n, long long batch, const bstq_params *p)
{
    if (dtype != BSTQ_F32 && dtype != BSTQ_F64)
        return -1;
    if (jobz != BSTQ_JOBZ_N && jobz != BSTQ_JOBZ_V)
        return -2;
    if (n < 1 || n > BSTQ_MAX_N)
        return -3;
    if (batch < 0)
        return -4;
    if (p) {
        if (p->no_sort != 0 && p->no_sort != 1)
            return -10;
        if (p->max_sweeps_per_n < 0 || p->max_sweeps_per_n > 1000000)
            return -10;
        if (p->scheduler < 0 || p->scheduler > 2)
            return -10;
        if (p->qstore < 0 || p->qstore > 6)
            return -10;
        if (p->log_entries < 0)
            return -10;
        if (p->kernel < 0 || p->kernel > 2)
            return -10;
        if (p->back_transform != 0 && p->back_transform != 1)
            return -10;
        if (p->update_scheme != 0 && p->update_scheme != 1)
            return -10;
        if (p->threads_per_block != 0 &&
            (p->threads_per_block < 32 || p->threads_per_block > 1024 || p->threads_per_block % 32))
            return -10;
    }
    return 0;
}

// Build the launch plan.  Returns 0, -10 for parameters no kernel supports,
// or BSTQ_ERR_NODEVICE.
int make_plan(int dtype, int jobz, int n, long long batch, const bstq_params *p, Plan &pl, int force_family = 0)
{
    DevInfo di;
    if (!dev_info(di))
        return BSTQ_ERR_NODEVICE;
    int nm = 0;
    for (int v : kNmList)
        if (v >= n) {
            nm = v;
            break;
        }
    const bool pg = p && p->update_scheme == 1;
    const int sched = (p && p->scheduler) ? p->scheduler : default_sched(dtype, jobz, nm);
    const int family = force_family ? force_family
                       : (p && p->kernel) ? p->kernel
                                          : (pg ? FAMILY_DYNAMIC : default_family(dtype, jobz, nm, sched));
    if (pg && family == FAMILY_STATIC)
        return -10;  // the PG step runs in the dynamic-position kernels only
    int qs = jobz ? ((p && p->qstore) ? p->qstore : default_qstore(dtype, nm, sched)) : 0;
    if (family != FAMILY_STATIC && jobz && qs != QS_LOG)
        qs = QS_GLOBAL;  // the dynamic kernels keep Q in global scratch
    pl.k = find_entry(dtype, jobz, nm, qs, sched, family);
    if (!pl.k)
        return -10;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pl.k->fn) != cudaSuccess) {
        cudaGetLastError();
        return BSTQ_ERR_NODEVICE;
    }
    if (qs == QS_LOG) {
        // record-and-apply (bstq_rlog.cuh), three launches:
        //  chase: one problem per thread, d and e in shared memory, blocks
        //    as the dynamic-position kernel's (threads_per_block applies);
        //  apply: one warp per problem and row chunk, four warps per block;
        //  finish: two warps of 32 problem slots per block, for the
        //    problems whose log ran out of room (normally none).
        // The log holds whole pages (a pass never crosses a page).
        const RlogLayout lay = rlog_layout(batch, n, nm, p ? p->log_entries : 0);
        const size_t per_thread = 2 * size_t(nm) * 4;
        const int regs = fa.numRegs > 0 ? fa.numRegs : 1;
        int cap = di.max_regs_sm / (((regs + 7) / 8) * 8);
        cap = cap / 32 * 32;
        if (cap > di.max_threads_sm)
            cap = di.max_threads_sm;
        const int by_smem = (int)((size_t)di.max_smem_block / per_thread) / 32 * 32;
        if (by_smem < cap)
            cap = by_smem;
        if (cap > fa.maxThreadsPerBlock)
            cap = fa.maxThreadsPerBlock / 32 * 32;
        if (cap > 1024)
            cap = 1024;
        if (cap < 32)
            return -10;
        int tpb;
        if (p && p->threads_per_block) {
            tpb = p->threads_per_block;
            if (tpb > cap)
                return -10;
        } else {
            tpb = choose_block_size(batch, di.sms, cap, false);
        }
        pl.tpb = tpb;
        pl.grid = batch > 0 ? (batch + tpb - 1) / tpb : 0;
        pl.smem = per_thread * tpb;
        constexpr int kApplyWarps = 4;
        pl.tpb2 = 32 * kApplyWarps;
        pl.smem2 = size_t(kApplyWarps) * Rlog<64>::WARP_BYTES;
        pl.grid2 = (lay.apply_warps + kApplyWarps - 1) / kApplyWarps;
        pl.tpb3 = 64;
        pl.ppb = 32;
        pl.smem3 = rlog_smem_bytes(nm, 2, 32);
        pl.grid3 = batch > 0 ? (batch + 63) / 64 : 0;
        if (pl.smem2 > (size_t)di.max_smem_block || pl.smem3 > (size_t)di.max_smem_block)
            return -10;
        pl.lcap = lay.lcap;
        pl.off_cnt = lay.off_cnt;
        pl.off_map = lay.off_map;
        pl.off_log = lay.off_log;
        pl.qwork_bytes = lay.total - lay.off_log;
        pl.work_bytes = lay.total;
        return 0;
    }
    if (qs == QS_SPLIT && (nm == 24 || nm == 32)) {
        // several Q warps per chase warp (bstq_split2.cuh): fixed block
        // shape, 32 problems per group of warps, as many blocks as the
        // batch needs (one block per SM at a time)
        const int threads = nm == 24 ? Split2ShapeOf<24>::THREADS : Split2ShapeOf<32>::THREADS;
        const int per_block = 32 * (nm == 24 ? Split2Cfg<24>::G : Split2Cfg<32>::G);
        pl.smem = nm == 24 ? Split2ShapeOf<24>::total : Split2ShapeOf<32>::total;
        pl.tpb = threads;
        if (p && p->threads_per_block && p->threads_per_block != pl.tpb)
            return -10;
        if (fa.maxThreadsPerBlock < pl.tpb || pl.smem > (size_t)di.max_smem_block)
            return -10;
        // spread the problems evenly over the SMs when one wave holds them
        long long ppb = batch > 0 ? (batch + di.sms - 1) / di.sms : 1;
        if (ppb > per_block)
            ppb = per_block;
        pl.ppb = (int)ppb;
        pl.grid = batch > 0 ? (batch + ppb - 1) / ppb : 0;
        pl.qwork_bytes = 0;
        pl.work_bytes = align256(size_t(batch) * 4);
        if (pl.work_bytes == 0)
            pl.work_bytes = 256;
        return 0;
    }
    if (qs == QS_SPLIT) {
        // fixed shape: kSplitPairs chase warps + kSplitPairs Q warps per block
        // (four warpgroups), up to 32 * kSplitLivePairs problems per block,
        // spread evenly over the SMs; shared memory as SplitSmem<nm>
        const int P = kSplitLivePairs;
        if (nm != 12 && nm != 16)
            return -10;
        pl.smem = nm == 12 ? SplitSmem<12>::total : SplitSmem<16>::total;
        pl.tpb = 64 * kSplitPairs;
        if (p && p->threads_per_block && p->threads_per_block != pl.tpb)
            return -10;
        if (fa.maxThreadsPerBlock < pl.tpb || pl.smem > (size_t)di.max_smem_block)
            return -10;
        // the register hand-over (setmaxnreg) draws on the block's launch
        // allocation: launch only if the compiled kernel holds all of it
        if ((long long)fa.numRegs * pl.tpb < 4LL * 32 * (2 * kSplitChaseRegs + 2 * kSplitQRegs))
            return -10;
        long long ppb = batch > 0 ? (batch + di.sms - 1) / di.sms : 1;
        if (ppb > 32LL * P)
            ppb = 32LL * P;
        pl.ppb = (int)ppb;
        pl.grid = batch > 0 ? (batch + ppb - 1) / ppb : 0;
        pl.qwork_bytes = 0;
        pl.work_bytes = align256(size_t(batch) * 4);
        if (pl.work_bytes == 0)
            pl.work_bytes = 256;
        return 0;
    }
    const size_t elem = dtype ? 8 : 4;
    const size_t mem_per_thread = jobz ? size_t(nm) * memory_rows(dtype, nm, qs) * elem : 0;
    size_t smem_per_thread;
    if (family == FAMILY_STATIC) {
        // the shared rows of Q (shared / hybrid), then the mirror of d and e
        // the settle step reads at dynamic positions, 2 nm elements per lane
        // (tpb is a multiple of 32: whole warps)
        smem_per_thread = ((qs == QS_SMEM || qs == QS_HYBRID) && jobz ? mem_per_thread : 0) +
                          2 * size_t(nm) * elem;
    } else {
        // d and e in shared memory, plus the column scales of the factored
        // double eigenvector update
        smem_per_thread = 2 * size_t(nm) * elem + ((dtype == BSTQ_F64 && jobz && nm < 48) ? 2 * size_t(nm) * elem : 0);
        // the carried eigenvector column above n = 64
        if (jobz && nm > 64)
            smem_per_thread += size_t(nm) * elem;
    }
    // Threads an SM can hold for this kernel.
    const int regs = fa.numRegs > 0 ? fa.numRegs : 1;
    int cap = di.max_regs_sm / (((regs + 7) / 8) * 8);
    cap = cap / 32 * 32;
    if (cap > di.max_threads_sm)
        cap = di.max_threads_sm;
    if (smem_per_thread) {
        const int by_smem = (int)((size_t)di.max_smem_block / smem_per_thread) / 32 * 32;
        if (by_smem < cap)
            cap = by_smem;
    }
    if (cap > fa.maxThreadsPerBlock)
        cap = fa.maxThreadsPerBlock / 32 * 32;
    if (cap > 1024)
        cap = 1024;
    if (cap < 32)
        return -10;
    int tpb;
    if (p && p->threads_per_block) {
        tpb = p->threads_per_block;
        if (tpb > cap)
            return -10;
    } else {
        // bstq_plan.h: one wave of one block per SM when the batch fits;
        // beyond, even waves for double (at n = 12 V, batch 131072,
        // 128-thread blocks left a quarter-full last wave and took 1.18x the
        // per-problem time of batch 32768, even waves 0.98x), 128-thread
        // blocks for float (n = 8 V, batch 65536: 0.057 against 0.059 ms)
        tpb = choose_block_size(batch, di.sms, cap, dtype == BSTQ_F64);
    }
    pl.tpb = tpb;
    pl.grid = batch > 0 ? (batch + tpb - 1) / tpb : 0;
    pl.smem = smem_per_thread * tpb;
    pl.qwork_bytes = (qs == QS_GLOBAL) ? size_t(pl.grid) * mem_per_thread * tpb : 0;
    // from n = 48 on, the double column scales follow Q in the scratch
    if (family != FAMILY_STATIC && dtype == BSTQ_F64 && jobz && nm >= 48)
        pl.qwork_bytes += size_t(pl.grid) * tpb * 2 * nm * elem;
    pl.work_bytes = align256(size_t(batch) * 4) + pl.qwork_bytes;
    if (pl.work_bytes == 0)
        pl.work_bytes = 256;
    return 0;
}

const char *qs_name(int qs)
{
    switch (qs) {
    case QS_REG: return "registers";
    case QS_SMEM: return "shared";
    case QS_GLOBAL: return "global";
    case QS_HYBRID: return "hybrid";
    case QS_SPLIT: return "split";
    case QS_LOG: return "log";
    default: return "none";
    }
}

int launch(const Plan &pl, int n, long long batch, int dtype, void *d, const void *e, void *Q,
           void *work, cudaStream_t st, const bstq_params *p)
{
    KParams kp{};
    kp.d = d;
    kp.e = e;
    kp.Q = Q;
    kp.info = reinterpret_cast<int *>(work);
    kp.qwork = pl.qwork_bytes ? reinterpret_cast<char *>(work) + align256(size_t(batch) * 4) : nullptr;
    kp.batch = batch;
    kp.n = n;
    const int per_n = (p && p->max_sweeps_per_n) ? p->max_sweeps_per_n : 30;
    kp.budget = per_n * n;
    kp.sort = (p && p->no_sort) ? 0 : 1;
    kp.ppb = pl.ppb;
    kp.back = (Q && p && p->back_transform) ? 1 : 0;
    kp.scheme = (p && p->update_scheme) ? 1 : 0;
    (void)dtype;
    void *args[] = {&kp};
    if (pl.k->qs == QS_LOG) {
        // record-and-apply: chase, apply, finish
        char *w = reinterpret_cast<char *>(work);
        kp.lcnt = reinterpret_cast<int *>(w + pl.off_cnt);
        kp.lmap = reinterpret_cast<unsigned char *>(w + pl.off_map);
        kp.qwork = w + pl.off_log;
        kp.lcap = pl.lcap;
        const void *fns[3] = {pl.k->fn, pl.k->fn2, pl.k->fn3};
        const long long grids[3] = {pl.grid, pl.grid2, pl.grid3};
        const int tpbs[3] = {pl.tpb, pl.tpb2, pl.tpb3};
        const size_t smems[3] = {pl.smem, pl.smem2, pl.smem3};
        for (int i = 0; i < 3; ++i) {
            if (!fns[i])
                return -10;
            if (grids[i] > 0x7fffffffLL)
                return -4;
        }
        for (int i = 0; i < 3; ++i) {
            if (smems[i] > 48 * 1024) {
                cudaError_t err =
                    cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smems[i]);
                if (err != cudaSuccess)
                    return cuda_fail(err, "cudaFuncSetAttribute");
            }
            cudaError_t err = cudaLaunchKernel(fns[i], dim3((unsigned)grids[i]), dim3(tpbs[i]), args, smems[i], st);
            if (err != cudaSuccess)
                return cuda_fail(err, "cudaLaunchKernel");
        }
        return 0;
    }
    if (pl.smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(pl.k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (err != cudaSuccess)
            return cuda_fail(err, "cudaFuncSetAttribute");
    }
    if (pl.grid > 0x7fffffffLL)
        return -4;
    cudaError_t err = cudaLaunchKernel(pl.k->fn, dim3((unsigned)pl.grid), dim3(pl.tpb), args, pl.smem, st);
    return err == cudaSuccess ? 0 : cuda_fail(err, "cudaLaunchKernel");
}

bool misaligned(const void *ptr, size_t a) { return ptr && (reinterpret_cast<uintptr_t>(ptr) % a) != 0; }

}  // namespace
}  // namespace bstq

using namespace bstq;

extern "C" size_t bstq_work_size_ex(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                                    const bstq_params *p)
{
    if (check_args(dtype, jobz, n, batch, p) != 0)
        return 0;
    Plan pl;
    if (make_plan(dtype, jobz, n, batch, p, pl) != 0)
        return 0;
    return pl.work_bytes;
}

extern "C" size_t bstq_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch)
{
    return bstq_work_size_ex(dtype, jobz, n, batch, nullptr);
}

extern "C" int bstq_solve_ex(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, void *d,
                             const void *e, void *Q, void *work, void *stream, const bstq_params *p)
{
    int rc = check_args(dtype, jobz, n, batch, p);
    if (rc)
        return rc;
    if (batch == 0)
        return 0;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    if (!d || misaligned(d, elem))
        return -5;
    if ((n > 1 && !e) || misaligned(e, elem))
        return -6;
    if (jobz == BSTQ_JOBZ_V && (!Q || misaligned(Q, elem)))
        return -7;
    if (!work || misaligned(work, 16))
        return -8;
    Plan pl;
    rc = make_plan(dtype, jobz, n, batch, p, pl);
    if (rc)
        return rc;
    return launch(pl, n, batch, dtype, d, e, Q, work, reinterpret_cast<cudaStream_t>(stream), p);
}

extern "C" int bstq_solve(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, void *d, const void *e,
                          void *Q, void *work, void *stream)
{
    return bstq_solve_ex(dtype, jobz, n, batch, d, e, Q, work, stream, nullptr);
}

// Device workspace layout of bstq_solve_host: d | e | Q | work, each 256-byte
// aligned.
extern "C" size_t bstq_host_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                                      const bstq_params *p)
{
    if (check_args(dtype, jobz, n, batch, p) != 0)
        return 0;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    size_t w = bstq_work_size_ex(dtype, jobz, n, batch, p);
    if (w == 0)
        return 0;
    size_t total = align256(elem * n * batch) + align256(elem * (n > 1 ? n - 1 : 1) * batch) +
                   (jobz == BSTQ_JOBZ_V ? align256(elem * n * n * batch) : 0) + w;
    return total;
}

extern "C" int bstq_solve_host(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, void *h_d,
                               const void *h_e, void *h_Q, int32_t *h_info, void *dev, void *stream,
                               const bstq_params *p)
{
    int rc = check_args(dtype, jobz, n, batch, p);
    if (rc)
        return rc == -10 ? -11 : rc;
    if (batch == 0)
        return 0;
    if (!h_d)
        return -5;
    if (n > 1 && !h_e)
        return -6;
    if (jobz == BSTQ_JOBZ_V && !h_Q)
        return -7;
    if (!h_info)
        return -8;
    if (!dev || misaligned(dev, 256))
        return -9;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    char *base = reinterpret_cast<char *>(dev);
    const size_t bd = elem * n * batch, be = elem * (n > 1 ? n - 1 : 0) * batch;
    const size_t bq = jobz == BSTQ_JOBZ_V ? elem * n * n * batch : 0;
    char *dd = base;
    char *de = dd + align256(bd);
    char *dq = de + align256(be > 0 ? be : elem * batch);
    char *dw = dq + (bq ? align256(bq) : 0);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if ((err = cudaMemcpyAsync(dd, h_d, bd, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync d");
    if (be && (err = cudaMemcpyAsync(de, h_e, be, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync e");
    if (bq && p && p->back_transform &&
        (err = cudaMemcpyAsync(dq, h_Q, bq, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync Q (basis)");
    rc = bstq_solve_ex(dtype, jobz, n, batch, dd, de, bq ? dq : nullptr, dw, stream, p);
    if (rc)
        return rc == -10 ? -11 : (rc < 0 ? -9 : rc);
    if ((err = cudaMemcpyAsync(h_d, dd, bd, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync lambda");
    if (bq && (err = cudaMemcpyAsync(h_Q, dq, bq, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync Q");
    if ((err = cudaMemcpyAsync(h_info, dw, 4 * size_t(batch), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(err, "cudaMemcpyAsync info");
    return 0;
}

// ---------------------------------------------------------------------------
// Fused small-n syev.  Workspace: info[batch] | Q scratch of the solve |
// off-diagonal scratch batch x (n-1) | the reduction's scratch (grid x tpb x
// 2 n^2: the copy of A and the reduction's Q), each 256-byte aligned.
// ---------------------------------------------------------------------------
namespace bstq {
namespace {

struct SyevPlan {
    Plan pl;
    size_t off_q = 0, off_e = 0, off_s = 0, total = 0;
};

int make_syev_plan(int dtype, int jobz, int n, long long batch, const bstq_params *p, SyevPlan &sp)
{
    if (n > kSyevMaxN)
        return -3;
    if (p && (p->back_transform || p->qstore || (p->kernel && p->kernel != BSTQ_KERNEL_DYNAMIC)))
        return -10;  // the fused kernel is one form; these do not apply
    int rc = make_plan(dtype, jobz, n, batch, p, sp.pl, FAMILY_SYEV);
    if (rc)
        return rc;
    const size_t elem = dtype ? 8 : 4;
    sp.off_q = align256(size_t(batch) * 4);
    sp.off_e = sp.off_q + align256(sp.pl.qwork_bytes);
    sp.off_s = sp.off_e + align256(elem * size_t(n > 1 ? n - 1 : 1) * size_t(batch));
    sp.total = sp.off_s + align256(elem * 2 * size_t(n) * n * size_t(sp.pl.tpb) * size_t(sp.pl.grid));
    return 0;
}

}  // namespace
}  // namespace bstq

extern "C" size_t bstq_syev_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch,
                                      const bstq_params *p)
{
    if (check_args(dtype, jobz, n, batch, p) != 0)
        return 0;
    SyevPlan sp;
    if (make_syev_plan(dtype, jobz, n, batch, p, sp) != 0)
        return 0;
    return sp.total > 256 ? sp.total : 256;
}

extern "C" int bstq_syev(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, const void *A, void *W,
                         void *V, void *work, void *stream, const bstq_params *p)
{
    int rc = check_args(dtype, jobz, n, batch, p);
    if (rc)
        return rc;
    if (n > kSyevMaxN)
        return -3;
    if (batch == 0)
        return 0;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    if (!A || misaligned(A, elem))
        return -5;
    if (!W || misaligned(W, elem))
        return -6;
    if (jobz == BSTQ_JOBZ_V && (!V || misaligned(V, elem)))
        return -7;
    if (!work || misaligned(work, 256))
        return -8;
    SyevPlan sp;
    rc = make_syev_plan(dtype, jobz, n, batch, p, sp);
    if (rc)
        return rc;
    const Plan &pl = sp.pl;
    char *w = reinterpret_cast<char *>(work);
    KParams kp{};
    kp.d = W;
    kp.e = w + sp.off_e;
    kp.Q = jobz == BSTQ_JOBZ_V ? V : nullptr;
    kp.info = reinterpret_cast<int *>(w);
    kp.qwork = pl.qwork_bytes ? w + sp.off_q : nullptr;
    kp.batch = batch;
    kp.n = n;
    kp.budget = ((p && p->max_sweeps_per_n) ? p->max_sweeps_per_n : 30) * n;
    kp.sort = (p && p->no_sort) ? 0 : 1;
    kp.ppb = pl.ppb;
    kp.back = 0;  // the kernel sets it for its solve
    kp.scheme = (p && p->update_scheme) ? 1 : 0;
    kp.A = A;
    kp.sscr = w + sp.off_s;
    if (pl.smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(pl.k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (err != cudaSuccess)
            return cuda_fail(err, "cudaFuncSetAttribute");
    }
    void *args[] = {&kp};
    if (pl.grid > 0x7fffffffLL)
        return -4;
    cudaError_t err = cudaLaunchKernel(pl.k->fn, dim3((unsigned)pl.grid), dim3(pl.tpb), args, pl.smem,
                                       reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? 0 : cuda_fail(err, "cudaLaunchKernel");
}

// ---------------------------------------------------------------------------
// stedc leaf solve.  Workspace: leaf diagonals of the full leaves | of the
// tail leaves | leaf off-diagonals (full | tail) | the full leaves' solve
// workspace | the tail leaves' solve workspace, each 256-byte aligned.
// ---------------------------------------------------------------------------
namespace bstq {
namespace {

struct LeafPlan {
    int L = 0, nfull = 0, t = 0;
    size_t off_dtail = 0, off_efull = 0, off_etail = 0, off_wfull = 0, off_wtail = 0, total = 0;
};

int make_leaf_plan(int dtype, int jobz, int n, int leaf, long long batch, const bstq_params *p, LeafPlan &lp)
{
    if (n < 1 || leaf < 1 || leaf > BSTQ_MAX_N)
        return -3;
    if (batch < 0 || (batch > 0 && (long long)n > (0x7fffffffffffffffLL / 8) / batch))
        return -4;
    if (p && p->back_transform)
        return -10;  // leaves start from the identity
    lp.L = leaf < n ? leaf : n;
    lp.nfull = n / lp.L;
    lp.t = n % lp.L;
    return 0;
}

// Workspace offsets (needs the current device: the solves' plans do).
int size_leaf_plan(int dtype, int jobz, long long batch, const bstq_params *p, LeafPlan &lp)
{
    const size_t elem = dtype ? 8 : 4;
    const size_t bf = size_t(batch) * size_t(lp.nfull), bt = lp.t ? size_t(batch) : 0;
    size_t wfull = 0, wtail = 0;
    if (bf) {
        int rc = check_args(dtype, jobz, lp.L, (long long)bf, p);
        if (rc)
            return rc;
        wfull = bstq_work_size_ex((bstq_dtype)dtype, (bstq_jobz)jobz, lp.L, (int64_t)bf, p);
        if (!wfull)
            return -10;
    }
    if (bt) {
        int rc = check_args(dtype, jobz, lp.t, (long long)bt, p);
        if (rc)
            return rc;
        wtail = bstq_work_size_ex((bstq_dtype)dtype, (bstq_jobz)jobz, lp.t, (int64_t)bt, p);
        if (!wtail)
            return -10;
    }
    lp.off_dtail = align256(elem * bf * lp.L);
    lp.off_efull = lp.off_dtail + align256(elem * bt * lp.t);
    lp.off_etail = lp.off_efull + align256(elem * bf * (lp.L - 1));
    lp.off_wfull = lp.off_etail + align256(elem * bt * (lp.t > 1 ? lp.t - 1 : 0));
    lp.off_wtail = lp.off_wfull + align256(wfull);
    lp.total = lp.off_wtail + align256(wtail);
    return 0;
}

}  // namespace
}  // namespace bstq

extern "C" size_t bstq_stedc_leaves_work_size(bstq_dtype dtype, bstq_jobz jobz, int n, int leaf, int64_t batch,
                                              const bstq_params *p)
{
    if (dtype != BSTQ_F32 && dtype != BSTQ_F64)
        return 0;
    if (jobz != BSTQ_JOBZ_N && jobz != BSTQ_JOBZ_V)
        return 0;
    LeafPlan lp;
    if (make_leaf_plan(dtype, jobz, n, leaf, batch, p, lp) != 0 || size_leaf_plan(dtype, jobz, batch, p, lp) != 0)
        return 0;
    return lp.total > 256 ? lp.total : 256;
}

extern "C" int bstq_stedc_leaves(bstq_dtype dtype, bstq_jobz jobz, int n, int leaf, int64_t batch, void *d,
                                 const void *e, void *Q, int32_t *info, void *work, void *stream,
                                 const bstq_params *p)
{
    if (dtype != BSTQ_F32 && dtype != BSTQ_F64)
        return -1;
    if (jobz != BSTQ_JOBZ_N && jobz != BSTQ_JOBZ_V)
        return -2;
    LeafPlan lp;
    int rc = make_leaf_plan(dtype, jobz, n, leaf, batch, p, lp);
    if (rc)
        return rc;
    if (batch == 0)
        return 0;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    if (!d || misaligned(d, elem))
        return -5;
    if ((n > 1 && !e) || misaligned(e, elem))
        return -6;
    if (jobz == BSTQ_JOBZ_V && (!Q || misaligned(Q, elem)))
        return -7;
    if (!info || misaligned(info, 4) || !work || misaligned(work, 256))
        return -8;
    DevInfo di;
    if (!dev_info(di))
        return BSTQ_ERR_NODEVICE;
    rc = size_leaf_plan(dtype, jobz, batch, p, lp);
    if (rc)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char *w = reinterpret_cast<char *>(work);
    char *dfull = w, *dtail = w + lp.off_dtail, *efull = w + lp.off_efull, *etail = w + lp.off_etail;
    char *wfull = w + lp.off_wfull, *wtail = w + lp.off_wtail;
    const int f64 = dtype == BSTQ_F64;
    cudaError_t err = launch_leaf_tear(f64, batch, n, lp.L, d, e, dfull, efull, dtail, etail, di.sms, st);
    if (err != cudaSuccess)
        return cuda_fail(err, "leaf tear");
    const long long bf = (long long)batch * lp.nfull;
    if (bf) {
        rc = bstq_solve_ex(dtype, jobz, lp.L, bf, dfull, lp.L > 1 ? efull : nullptr, Q, wfull, stream, p);
        if (rc)
            return rc < 0 ? -10 : rc;
    }
    if (lp.t) {
        char *qt = Q ? reinterpret_cast<char *>(Q) + elem * size_t(bf) * lp.L * lp.L : nullptr;
        rc = bstq_solve_ex(dtype, jobz, lp.t, batch, dtail, lp.t > 1 ? etail : nullptr,
                           jobz == BSTQ_JOBZ_V ? qt : nullptr, wtail, stream, p);
        if (rc)
            return rc < 0 ? -10 : rc;
    }
    err = launch_leaf_gather(f64, batch, n, lp.L, d, dfull, dtail, reinterpret_cast<const int *>(wfull),
                             reinterpret_cast<const int *>(wtail), info, di.sms, st);
    return err == cudaSuccess ? 0 : cuda_fail(err, "leaf gather");
}

extern "C" int bstq_describe(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, const bstq_params *p,
                             char *buf, size_t len)
{
    int rc = check_args(dtype, jobz, n, batch, p);
    if (rc)
        return rc;
    Plan pl;
    rc = make_plan(dtype, jobz, n, batch, p, pl);
    if (rc)
        return rc;
    if (buf && len) {
        cudaFuncAttributes fa;
        int regs = 0;
        if (cudaFuncGetAttributes(&fa, pl.k->fn) == cudaSuccess)
            regs = fa.numRegs;
        else
            cudaGetLastError();
        int w = snprintf(buf, len, "%s<%s,%d,%s,%s,%s> tpb=%d grid=%lld smem=%zu regs=%d work=%zu",
                         pl.k->family == FAMILY_DYNAMIC ? "dyn" : "lane", dtype ? "f64" : "f32", pl.k->nm,
                         jobz ? "V" : "N", jobz ? qs_name(pl.k->qs) : "none",
                         pl.k->sched == SCHED_FLAT ? "flat" : "nested", pl.tpb, pl.grid, pl.smem, regs,
                         pl.work_bytes);
        if (pl.k->qs == QS_LOG && w > 0 && (size_t)w < len) {
            // the record-and-apply path's other two launches
            int regs2 = 0;
            if (cudaFuncGetAttributes(&fa, pl.k->fn2) == cudaSuccess)
                regs2 = fa.numRegs;
            else
                cudaGetLastError();
            snprintf(buf + w, len - w, " apply: tpb=%d grid=%lld smem=%zu regs=%d; finish: tpb=%d grid=%lld",
                     pl.tpb2, pl.grid2, pl.smem2, regs2, pl.tpb3, pl.grid3);
        }
    }
    return 0;
}

extern "C" const char *bstq_status_string(int code)
{
    switch (code) {
    case 0: return "success";
    case BSTQ_ERR_CUDA: return "CUDA launch or copy failed";
    case BSTQ_ERR_NODEVICE: return "no usable CUDA device is current";
    case -1: return "invalid dtype";
    case -2: return "invalid jobz";
    case -3: return "n outside [1, 128]";
    case -4: return "invalid batch (bstq_solve_noalloc: more problems than its fixed scratch array holds)";
    case -5: return "d is NULL or misaligned";
    case -6: return "e is NULL or misaligned";
    case -7: return "Q is NULL or misaligned";
    case -8: return "work is NULL, misaligned or info buffer missing";
    case -9: return "invalid device workspace";
    case -10: return "invalid or unsupported parameters";
    case -11: return "invalid or unsupported parameters";
    default: return "unknown status";
    }
}

extern "C" const char *bstq_version(void) { return "bstq 0.1.0 sm_103a"; }

extern "C" const char *bstq_last_error(void) { return g_last_error; }

extern "C" size_t bstq_diag_work_size(int op, bstq_dtype dtype, int64_t count)
{
    if ((dtype != BSTQ_F32 && dtype != BSTQ_F64) || count < 0 || diag_check_op(op, dtype == BSTQ_F64) != 0)
        return 0;
    return diag_work_bytes(op, dtype == BSTQ_F64, count);
}

extern "C" int bstq_diag(int op, bstq_dtype dtype, int64_t count, int arg, const void *in, void *out, void *work,
                         void *stream)
{
    if (dtype != BSTQ_F32 && dtype != BSTQ_F64)
        return -2;
    const int f64 = dtype == BSTQ_F64;
    if (diag_check_op(op, f64) != 0)
        return -1;
    if (count < 0 || count > (1LL << 36))
        return -3;
    if (op == BSTQ_DIAG_FASTQ && (arg < 0 || arg > 1000000))
        return -4;
    if (count == 0)
        return 0;
    const size_t elem = f64 ? 8 : 4;
    if (misaligned(in, elem) || !in)
        return -5;
    if (misaligned(out, elem) || !out)
        return -6;
    if (diag_uses_work(op) && (!work || misaligned(work, 16)))
        return -7;
    DevInfo di;
    if (!dev_info(di))
        return BSTQ_ERR_NODEVICE;
    const cudaError_t err = launch_diag(op, f64, count, arg, in, out, work, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? 0 : cuda_fail(err, "diagnostic launch");
}

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot allocate device memory at the moment they solve: code
// running inside a captured CUDA graph or a custom allocator's hook, plugins
// that are handed fixed buffers by a host framework, or real-time loops that
// must never call cudaMalloc.  bstq_solve needs a `work` buffer whose size
// depends on the launch; this variant instead keeps the eigenvector scratch
// of the global-memory Q kernel in a fixed array that lives in the library's
// own device image.  The array is reserved on every GPU that loads this
// library and stays reserved until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol's name only stands for the array; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
int noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return bstq::cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return BSTQ_ERR_NODEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess)
            return bstq::cuda_fail(err, "cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return 0;
}

}  // namespace

extern "C" int bstq_solve_noalloc(bstq_dtype dtype, bstq_jobz jobz, int n, int64_t batch, void *d,
                                  const void *e, void *Q, int32_t *info, void *stream,
                                  const bstq_params *p)
{
    int rc = check_args(dtype, jobz, n, batch, p);
    if (rc)
        return rc;
    if (jobz != BSTQ_JOBZ_V)
        return -2;
    if (batch == 0)
        return 0;
    const size_t elem = dtype == BSTQ_F64 ? 8 : 4;
    if (!d || misaligned(d, elem))
        return -5;
    if ((n > 1 && !e) || misaligned(e, elem))
        return -6;
    if (!Q || misaligned(Q, elem))
        return -7;
    if (!info || misaligned(info, 4))
        return -8;
    bstq_params q = p ? *p : bstq_params{};
    q.qstore = BSTQ_QSTORE_GLOBAL;
    Plan pl;
    rc = make_plan(dtype, jobz, n, batch, &q, pl);
    if (rc == -10 && q.kernel == 0) {
        // the static family keeps small Q in registers and has no scratch
        // variant there; the dynamic family covers every n
        q.kernel = BSTQ_KERNEL_DYNAMIC;
        rc = make_plan(dtype, jobz, n, batch, &q, pl);
    }
    if (rc)
        return rc;
    if (pl.k->qs != QS_GLOBAL)
        return -10;
    if (pl.qwork_bytes > kNoAllocScratchBytes)
        return -4;  // more problems than the fixed scratch holds
    void *scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc)
        return rc;
    KParams kp{};
    kp.d = d;
    kp.e = e;
    kp.Q = Q;
    kp.info = info;
    kp.qwork = scratch;
    kp.batch = batch;
    kp.n = n;
    kp.budget = (q.max_sweeps_per_n ? q.max_sweeps_per_n : 30) * n;
    kp.sort = q.no_sort ? 0 : 1;
    kp.ppb = pl.ppb;
    kp.back = q.back_transform ? 1 : 0;
    kp.scheme = q.update_scheme ? 1 : 0;
    if (pl.smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(pl.k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (err != cudaSuccess)
            return cuda_fail(err, "cudaFuncSetAttribute");
    }
    void *args[] = {&kp};
    cudaError_t err = cudaLaunchKernel(pl.k->fn, dim3((unsigned)pl.grid), dim3(pl.tpb), args, pl.smem,
                                       reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? 0 : cuda_fail(err, "cudaLaunchKernel");
}
