// Launcher of the shifting reduction (dt_reduce_shift.cu): AllReduce and
// ReduceScatter over rank buffers that lie at different offsets past a
// 16-byte boundary.  Every input address must be a whole number of elements;
// the outputs of a job must share their offset.  Not part of the C ABI.
#pragma once

#include "dt_internal.h"

namespace dt {

cudaError_t launch_reduce_shift(const ReduceParams &p, int dtype, int op, int jobs, int device,
                                cudaStream_t s);

}  // namespace dt
