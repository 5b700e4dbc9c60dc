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

namespace bstq {

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
