// Host-only check of the record-and-apply workspace layout
// (csrc/bstq_plan.h): reads lines "batch n nm log_entries" on stdin and
// prints the log length, the offsets, the total bytes and the apply warps.
// Built and run by tests/test_plan_shape.py.
#include <cstdio>

#include "bstq_plan.h"

int main()
{
    long long batch, log_entries;
    int n, nm;
    while (std::scanf("%lld %d %d %lld", &batch, &n, &nm, &log_entries) == 4) {
        const bstq::RlogLayout r = bstq::rlog_layout(batch, n, nm, log_entries);
        std::printf("%lld %zu %zu %zu %zu %lld\n", r.lcap, r.off_cnt, r.off_map, r.off_log, r.total, r.apply_warps);
    }
    return 0;
}
