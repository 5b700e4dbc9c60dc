// Launchers of the leaf tear and gather kernels (bstq_leaves.cu), used by
// the stedc leaf-solve entry point.  Pointers of unused groups (no full
// leaves, or no tail leaf) are never dereferenced.
#pragma once

#include <cuda_runtime.h>

namespace bstq {

// d, e -> leaf diagonals and off-diagonals: full leaves at dfull/efull
// ((b * nfull + k) * L, (b * nfull + k) * (L - 1)), the tail leaf at
// dtail/etail (b * t, b * (t - 1)); nfull = n / L, t = n % L.
cudaError_t launch_leaf_tear(int f64, long long batch, int n, int L, const void *d, const void *e, void *dfull,
                             void *efull, void *dtail, void *etail, int sms, cudaStream_t st);

// leaf eigenvalues -> d (each leaf's rows), leaf status -> info[b * leaves + k]
cudaError_t launch_leaf_gather(int f64, long long batch, int n, int L, void *d, const void *dfull,
                               const void *dtail, const int *info_full, const int *info_tail, int *info, int sms,
                               cudaStream_t st);

}  // namespace bstq
