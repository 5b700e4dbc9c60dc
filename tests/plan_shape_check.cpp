// Host-only check of the launch plan's block size (csrc/bstq_plan.h):
// reads lines "batch sms cap f64" on stdin and prints the block size and
// grid the plan gives for each.  Built and run by tests/test_plan_shape.py.
#include <cstdio>

#include "bstq_plan.h"

int main()
{
    long long batch;
    int sms, cap, f64;
    while (std::scanf("%lld %d %d %d", &batch, &sms, &cap, &f64) == 4) {
        const int tpb = bstq::choose_block_size(batch, sms, cap, f64 != 0);
        const long long grid = batch > 0 ? (batch + tpb - 1) / tpb : 0;
        std::printf("%d %lld\n", tpb, grid);
    }
    return 0;
}
