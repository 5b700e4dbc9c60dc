// Table of compiled kernel variants, filled by the instantiation units that
// gen_instances.py writes (one lister function per unit).
#pragma once

#include "bstq_registry_list.inc"

namespace bstq {

struct KernelEntry {
    int dtype;   // 0 f32, 1 f64
    int jobz;    // 0 N, 1 V
    int nm;      // compile-time maximum n
    int qs;      // Q storage (QS_*; 0 for jobz N)
    int sched;   // SCHED_FLAT / SCHED_NESTED
    const void *fn;
    int family;  // FAMILY_STATIC (bstq_lane.cuh) / FAMILY_DYNAMIC (bstq_dyn.cuh) /
                 // FAMILY_SYEV (bstq_syev.cuh, fused dense solve)
    const void *fn2 = nullptr;  // record-and-apply: the apply kernel
    const void *fn3 = nullptr;  // record-and-apply: the finishing kernel
};

enum { FAMILY_STATIC = 1, FAMILY_DYNAMIC = 2, FAMILY_SYEV = 3 };

#define BSTQ_DECLARE_UNIT(name) const KernelEntry *entries_##name(int *count);
BSTQ_FOR_EACH_UNIT(BSTQ_DECLARE_UNIT)
#undef BSTQ_DECLARE_UNIT

}  // namespace bstq
