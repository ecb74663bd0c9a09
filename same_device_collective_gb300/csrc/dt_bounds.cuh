// Bounds-checked builds (DT_BOUNDS=1 when building): every global load and
// store of the data kernels is checked against the extent of the buffer it
// belongs to, as the host computed it from the call's arguments (not from
// the kernel's own index arithmetic).  An access outside records
// DT_ERR_INVALID in the group's error word once -- rank = the kernel
// (kBounds*), peer = the buffer index, gen = the low 31 bits of the byte
// offset from the buffer's start -- and is skipped; nothing traps.  In other
// builds DT_IN_BOUNDS(...) is `true` and its arguments are not compiled.
#pragma once

#include <cstdint>

#include "dt_device.cuh"
#include "dt_internal.h"

namespace dt {

enum BoundsKernel : int {
    kBoundsReduce = DT_BOUNDS_REDUCE,
    kBoundsReduceShift = DT_BOUNDS_REDUCE_SHIFT,
    kBoundsCopyBulk = DT_BOUNDS_COPY_BULK,
    kBoundsCopyVec = DT_BOUNDS_COPY_VEC,
    kBoundsCopyEdge = DT_BOUNDS_COPY_EDGE,
    kBoundsCopyShift = DT_BOUNDS_COPY_SHIFT,
    kBoundsCopy2d = DT_BOUNDS_COPY_2D,
    kBoundsBucket = DT_BOUNDS_BUCKET,
};

#ifdef DT_BOUNDS

// [a, a + n) lies inside [lo, hi)
__device__ __forceinline__ bool span_in(const void *a, uint64_t n, uint64_t lo, uint64_t hi)
{
    const uint64_t x = reinterpret_cast<uint64_t>(a);
    return x >= lo && x + n <= hi;
}

// an aligned 16-byte vector read that holds at least one byte of [lo, hi)
// and no byte outside the 16-byte blocks that [lo, hi) touches
__device__ __forceinline__ bool vector_touches(const void *a, uint64_t lo, uint64_t hi)
{
    const uint64_t x = reinterpret_cast<uint64_t>(a);
    return x + 16 > lo && x < hi && x >= (lo & ~15ull) && x + 16 <= ((hi + 15) & ~15ull);
}

static __device__ __noinline__ void bounds_fail(const ErrorSink &s, int kernel, int buffer, const void *a,
                                                uint64_t lo)
{
    if (s.err == nullptr) return;   // dt_bucket_allreduce_static: no error word; the access is still skipped
    record_error(s, DT_ERR_INVALID, kernel, buffer,
                 (int)((reinterpret_cast<uint64_t>(a) - lo) & 0x7FFFFFFFull));
}

#define DT_IN_BOUNDS(ok, sink, kernel, buffer, addr, lo) \
    ((ok) ? true : (::dt::bounds_fail((sink), (kernel), (buffer), (addr), (lo)), false))

// Element i of job j's reduction (reduce_elem's operands): every input's
// element in_off + i and every output's element i lie in their buffers.
template <int ES>
__device__ bool reduce_elem_in_bounds(const ReduceParams &p, int kernel, int64_t in_off, int64_t i,
                                      void *const *dst, int ndst, int job)
{
    bool ok = true;
    for (int r = 0; r < p.P; ++r) {
        const unsigned char *a = static_cast<const unsigned char *>(p.in[r]) + (in_off + i) * ES;
        ok = ok && DT_IN_BOUNDS(span_in(a, ES, p.in_lo[r], p.in_hi[r]), p.sink, kernel, r, a, p.in_lo[r]);
    }
    for (int k = 0; k < ndst; ++k) {
        const int q = job * p.out_per_job + k;
        const unsigned char *a = static_cast<const unsigned char *>(dst[k]) + i * ES;
        ok = ok && DT_IN_BOUNDS(span_in(a, ES, p.out_lo[q], p.out_hi[q]), p.sink, kernel, DT_MAX_RANKS + q,
                                a, p.out_lo[q]);
    }
    return ok;
}

#define DT_REDUCE_ELEM_OK(ES, p, kernel, in_off, i, dst, ndst, job) \
    ::dt::reduce_elem_in_bounds<ES>((p), (kernel), (in_off), (i), (dst), (ndst), (job))

#else

#define DT_IN_BOUNDS(ok, sink, kernel, buffer, addr, lo) true
#define DT_REDUCE_ELEM_OK(ES, p, kernel, in_off, i, dst, ndst, job) true

#endif

}  // namespace dt
