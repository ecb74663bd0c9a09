// Per-block timeline of the kernels (builds made with DT_TIMELINE=1; see
// dt_timeline_start in dt.h).  Every instrumented kernel notes %globaltimer
// at its start (DT_TL_BEGIN), after its wait on the previous kernel
// (DT_TL_WAITED) and at its end, where one thread of the block appends a
// record.  In other builds the macros expand to nothing.
#pragma once

#include <cstdint>

#include "dt.h"
#include "dt_device.cuh"
#include "dt_timeline.h"

namespace dt {

#ifdef DT_TIMELINE

// One copy per translation unit (internal linkage); that unit's
// bind_timeline_* function points it at the buffer.
static __device__ TimelineSink g_timeline;

__device__ __forceinline__ void timeline_record(uint32_t kind, uint64_t t0, uint64_t t1)
{
    const TimelineSink s = g_timeline;
    if (!s.rec) return;
    const uint64_t t2 = global_ns();
    const unsigned long long k = atomicAdd(s.count, 1ull);
    if (k >= s.cap) return;
    uint64_t grid;
    uint32_t sm;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(grid));
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    dt_timeline_record r;
    r.grid = grid;
    r.kind = kind;
    r.block = blockIdx.x + gridDim.x * blockIdx.y;
    r.sm = sm;
    r.pad = 0;
    r.t_start = t0;
    r.t_waited = t1;
    r.t_end = t2;
    s.rec[k] = r;
}

#define DT_TL_BEGIN() const uint64_t dt_tl_t0 = ::dt::global_ns()
#define DT_TL_WAITED() const uint64_t dt_tl_t1 = ::dt::global_ns()
// every thread of the block calls it: the block's last thread is done
#define DT_TL_END_BLOCK(kind)                                                     \
    do {                                                                          \
        __syncthreads();                                                          \
        if (threadIdx.x == 0) ::dt::timeline_record((kind), dt_tl_t0, dt_tl_t1); \
    } while (0)
// one thread (the block's only working one) calls it
#define DT_TL_END_THREAD(kind) ::dt::timeline_record((kind), dt_tl_t0, dt_tl_t1)
#define DT_TL_BINDER(name)                                                        \
    void name(const void *sink)                                                   \
    {                                                                             \
        cudaMemcpyToSymbol(g_timeline, sink, sizeof(TimelineSink));               \
    }

#else

#define DT_TL_BEGIN()
#define DT_TL_WAITED()
#define DT_TL_END_BLOCK(kind)
#define DT_TL_END_THREAD(kind)
#define DT_TL_BINDER(name)

#endif

}  // namespace dt
