// Host side of the kernel timeline (builds made with DT_TIMELINE=1): the
// buffer the kernels append to, and the function of each instrumented
// translation unit that points its kernels at it.  The device side is
// dt_timeline.cuh.  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "dt.h"

namespace dt {

#ifdef DT_TIMELINE

struct TimelineSink {
    dt_timeline_record *rec;
    unsigned long long *count;
    unsigned long long cap;
};

void bind_timeline_reduce(const void *sink);
void bind_timeline_reduce_shift(const void *sink);
void bind_timeline_copy(const void *sink);
void bind_timeline_bucket(const void *sink);
void bind_timeline_barrier(const void *sink);
cudaError_t launch_timeline_mark(uint32_t tag, cudaStream_t s);

#endif

}  // namespace dt
