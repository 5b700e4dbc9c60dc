// Launcher of the diagnostic kernels (bstq_diag.cu), used by bstq_diag in
// the C ABI.  Each runs one building block of the solve on a table of
// inputs; the operations and record layouts are those of include/bstq.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace bstq {

// 0 when op exists for the dtype, -1 otherwise.
int diag_check_op(int op, int f64);
// whether op needs the work buffer, and its size in bytes
bool diag_uses_work(int op);
size_t diag_work_bytes(int op, int f64, long long count);
cudaError_t launch_diag(int op, int f64, long long count, int arg, const void *in, void *out, void *work,
                        cudaStream_t st);

}  // namespace bstq
