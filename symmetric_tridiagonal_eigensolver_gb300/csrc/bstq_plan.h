// Block size of the lane-per-problem kernels (one problem per thread), as a
// plain host function so it can be checked without a GPU.
//   batch  problems in the call;
//   sms    streaming multiprocessors of the device;
//   cap    the most threads one block of this kernel may hold (its registers,
//          shared memory and launch limit), a multiple of 32;
//   f64    the kernel computes in double.
// One wave of one block per SM when the whole batch fits: ceil(batch / sms)
// threads rounded up to 32, so the problems spread evenly over all SMs.
// Beyond one wave, double kernels (bound by the FP64 pipe, where an even
// load per SM pays) take the fewest waves of one block per SM with the
// problems spread evenly over them; float kernels (bound by their
// dependency chains) take 128-thread blocks, several per SM.
#pragma once

#include <stddef.h>

namespace bstq {

// ---------------------------------------------------------------------------
// Record-and-apply path (bstq_rlog.cuh): log pages, rows per apply warp and
// the workspace layout, as plain host functions so they can be checked
// without a GPU.
// ---------------------------------------------------------------------------
constexpr int kRlogPage = 256;  // log entries per page; a pass never crosses one

// Rows of Q one warp of the apply holds at once: two rows per lane for
// 32 < n_pad <= 64, one otherwise.
constexpr int rlog_rows(int nm) { return (nm > 32 && nm <= 64) ? 64 : 32; }

struct RlogLayout {
    long long lcap;          // log entries per problem (whole pages)
    size_t off_cnt;          // int[batch]: log length or state code per problem
    size_t off_map;          // unsigned char[batch][2 n]: the column maps
    size_t off_log;          // float2[batch][lcap]: the logs
    size_t total;            // bytes of work (info[batch] at offset 0)
    long long apply_warps;   // warps of the apply launch: problems x row chunks
};

inline size_t rlog_align256(size_t x) { return (x + 255) & ~size_t(255); }

// log_entries <= 0: the default 1.5 n^2 + 8 n entries (an N(0,1) solve
// writes about n^2 entries of rotations and headers, plus page ends and
// padding); any length is rounded up to whole pages.
inline RlogLayout rlog_layout(long long batch, int n, int nm, long long log_entries)
{
    RlogLayout r;
    const long long want = log_entries > 0 ? log_entries : 3LL * n * n / 2 + 8LL * n;
    r.lcap = (want + kRlogPage - 1) / kRlogPage * kRlogPage;
    r.off_cnt = rlog_align256(size_t(batch) * 4);
    r.off_map = r.off_cnt + rlog_align256(size_t(batch) * 4);
    r.off_log = r.off_map + rlog_align256(size_t(batch) * 2 * size_t(n));
    r.total = r.off_log + size_t(batch) * size_t(r.lcap) * 8;
    if (r.total < 256)
        r.total = 256;
    const int rows = rlog_rows(nm);
    r.apply_warps = batch * ((n + rows - 1) / rows);
    return r;
}

inline int choose_block_size(long long batch, int sms, int cap, bool f64)
{
    if (batch <= (long long)sms * cap || f64) {
        const long long per_wave = (long long)sms * cap;
        const long long waves = batch > 0 ? (batch + per_wave - 1) / per_wave : 1;
        const long long want = (batch + sms * waves - 1) / (sms * waves);
        long long tpb = (want + 31) / 32 * 32;
        if (tpb < 32)
            tpb = 32;
        if (tpb > cap)
            tpb = cap;
        return (int)tpb;
    }
    return cap < 128 ? cap : 128;
}

}  // namespace bstq
