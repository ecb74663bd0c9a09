// Byte-shifted 16-byte vectors for buffers that do not start on a 16-byte
// boundary, shared by the shifting copy and the shifting reduction.
//
// Sixteen bytes that start `sh` bytes into an aligned vector end in the next
// one.  A warp reads such a run as aligned vectors: lane L loads vector c,
// receives vector c + 1 from lane L + 1 (__shfl_down_sync) and funnel-shifts
// the pair by sh bytes.
#pragma once

#include <cstdint>

namespace dt {

// bytes [sh, sh + 16) of the 32-byte little-endian sequence a, b (sh < 16)
__device__ __forceinline__ uint4 shift_pair(const uint4 &a, const uint4 &b, uint32_t sh)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t bits = (sh & 3) * 8;
    uint32_t o[4];
    switch (sh >> 2) {
#define DT_SHIFT_CASE(q)                                                                  \
    case q:                                                                               \
        o[0] = __funnelshift_r(w[q + 0], w[q + 1], bits);                                 \
        o[1] = __funnelshift_r(w[q + 1], w[q + 2], bits);                                 \
        o[2] = __funnelshift_r(w[q + 2], w[q + 3], bits);                                 \
        o[3] = __funnelshift_r(w[q + 3], w[q + 4], bits);                                 \
        break;
        DT_SHIFT_CASE(0)
        DT_SHIFT_CASE(1)
        DT_SHIFT_CASE(2)
        DT_SHIFT_CASE(3)
#undef DT_SHIFT_CASE
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// v of lane L + 1 (lane 31 gets its own v back)
__device__ __forceinline__ uint4 shfl_down_uint4(const uint4 &v)
{
    return make_uint4(__shfl_down_sync(0xFFFFFFFFu, v.x, 1), __shfl_down_sync(0xFFFFFFFFu, v.y, 1),
                      __shfl_down_sync(0xFFFFFFFFu, v.z, 1), __shfl_down_sync(0xFFFFFFFFu, v.w, 1));
}

}  // namespace dt
