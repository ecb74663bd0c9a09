// Element arithmetic of the reducing collectives, shared by the AllReduce /
// ReduceScatter kernel and the fused bucket kernel.
//
// Ranks are combined in ascending order, rank 0 first: the same-device
// AllReduce of the DTorch collective-communication page (§2.3) starts from
// rank 0's tensor and adds ranks 1..P-1 onto it in turn.  fp32 and bf16
// accumulate in fp32 (bf16 widens exactly), with one round-to-nearest-even
// narrowing at the store; AVG divides the fp32 sum by P (the hyper-parallel
// page divides each reduced gradient by the replicate world size); int32
// sums wrap.  MAX / MIN select an input element: a NaN wins, equal values
// keep the lower rank's element.  SUM_STEPWISE is the page's literal `+=` in
// the element type: bf16 rounds after every rank.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "dt.h"

namespace dt {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x -> low half, .y -> high half
    uint32_t w;
    memcpy(&w, &h, sizeof w);
    return w;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    uint16_t b;
    memcpy(&b, &h, sizeof b);
    return b;
}

__device__ __forceinline__ float avg_of(float sum, int P, float scale, int pow2)
{
    // For P = 2^k, sum * 2^-k and sum / P are the same real number and round
    // identically; other P take the IEEE division.
    return pow2 ? __fmul_rn(sum, scale) : __fdiv_rn(sum, (float)P);
}

template <int OP>
__device__ __forceinline__ bool take_f(float x, float best)
{
    return (x != x) || (OP == DT_MAX ? x > best : x < best);
}

// MAX / MIN on two packed bf16 elements: per 16-bit half, x replaces the
// running choice where x is a NaN or compares strictly above (MAX) / below
// (MIN) it.  The bf16x2 comparisons give an all-ones half where they hold;
// ordered comparisons are false against a NaN and between equal values (+0
// and -0 included), so ties keep the lower rank's element and a NaN, once
// chosen, gives way only to a later NaN.  The halves move as raw bits, so the
// chosen element (NaN payload included) is stored unchanged: the same choice
// as take_f on the widened values, since bf16 -> fp32 is exact.
template <int OP>
__device__ __forceinline__ uint32_t select_bf16x2(uint32_t x, uint32_t best)
{
    uint32_t beats, nan;
    if constexpr (OP == DT_MAX)
        asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(beats) : "r"(x), "r"(best));
    else
        asm("set.lt.u32.bf16x2 %0, %1, %2;" : "=r"(beats) : "r"(x), "r"(best));
    asm("set.nan.u32.bf16x2 %0, %1, %1;" : "=r"(nan) : "r"(x));
    const uint32_t m = beats | nan;
    return (x & m) | (best & ~m);
}

// fp32 -> bf16 (round to nearest even) -> fp32: where a stepwise sum lands.
__device__ __forceinline__ float round_bf16(float f)
{
    return __uint_as_float((uint32_t)f32_to_bf16(f) << 16);
}

template <int OP>
__device__ __forceinline__ int32_t pick_i(int32_t acc, int32_t x)
{
    if (OP == DT_SUM || OP == DT_SUM_STEPWISE) return (int32_t)((uint32_t)acc + (uint32_t)x);
    if (OP == DT_MAX) return x > acc ? x : acc;
    return x < acc ? x : acc;
}

// Reduce one 16-byte vector position across the first P of PMAX rank vectors.
template <int DT, int OP, int PMAX>
__device__ __forceinline__ uint4 reduce_vec16(const uint4 (&x)[PMAX], int P, float scale, int pow2)
{
    uint32_t w[PMAX][4];
#pragma unroll
    for (int r = 0; r < PMAX; ++r) {
        w[r][0] = x[r].x; w[r][1] = x[r].y; w[r][2] = x[r].z; w[r][3] = x[r].w;
    }
    uint32_t o[4];
    if constexpr (DT == DT_I32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            int32_t acc = (int32_t)w[0][k];
#pragma unroll
            for (int r = 1; r < PMAX; ++r)
                if (r < P) acc = pick_i<OP>(acc, (int32_t)w[r][k]);
            o[k] = (uint32_t)acc;
        }
    } else if constexpr (DT == DT_F32 && (OP == DT_MAX || OP == DT_MIN) && PMAX == 16) {
        // More than 8 ranks: ranks 0..7 and 8..P-1 are scanned as two
        // independent chains, then the upper chain's choice replaces the lower
        // one's by the same rule.  Splitting the scan cannot change the
        // choice: either way it is the last NaN if there is one, else the
        // first element equal to the extreme value.
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float lo = __uint_as_float(w[0][k]);
#pragma unroll
            for (int r = 1; r < 8; ++r) {
                if (r < P) {
                    const float x = __uint_as_float(w[r][k]);
                    lo = take_f<OP>(x, lo) ? x : lo;
                }
            }
            if (P > 8) {
                float hi = __uint_as_float(w[8][k]);
#pragma unroll
                for (int r = 9; r < 16; ++r) {
                    if (r < P) {
                        const float x = __uint_as_float(w[r][k]);
                        hi = take_f<OP>(x, hi) ? x : hi;
                    }
                }
                lo = take_f<OP>(hi, lo) ? hi : lo;
            }
            o[k] = __float_as_uint(lo);
        }
    } else if constexpr (DT == DT_F32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float acc = __uint_as_float(w[0][k]);
#pragma unroll
            for (int r = 1; r < PMAX; ++r) {
                if (r < P) {
                    float x1 = __uint_as_float(w[r][k]);
                    if constexpr (OP == DT_SUM || OP == DT_AVG || OP == DT_SUM_STEPWISE)
                        acc = __fadd_rn(acc, x1);
                    else acc = take_f<OP>(x1, acc) ? x1 : acc;
                }
            }
            if constexpr (OP == DT_AVG) acc = avg_of(acc, P, scale, pow2);
            o[k] = __float_as_uint(acc);
        }
    } else {  // bf16: two elements per 32-bit word, low half first
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (OP == DT_SUM || OP == DT_AVG || OP == DT_SUM_STEPWISE) {
                float lo = bf16_lo(w[0][k]), hi = bf16_hi(w[0][k]);
#pragma unroll
                for (int r = 1; r < PMAX; ++r) {
                    if (r < P) {
                        lo = __fadd_rn(lo, bf16_lo(w[r][k]));
                        hi = __fadd_rn(hi, bf16_hi(w[r][k]));
                        if constexpr (OP == DT_SUM_STEPWISE) {
                            lo = round_bf16(lo);
                            hi = round_bf16(hi);
                        }
                    }
                }
                if constexpr (OP == DT_AVG) {
                    lo = avg_of(lo, P, scale, pow2);
                    hi = avg_of(hi, P, scale, pow2);
                }
                o[k] = pack_bf16x2(lo, hi);
            } else {
                // both elements of the word at once, without widening
                uint32_t best = w[0][k];
#pragma unroll
                for (int r = 1; r < PMAX; ++r)
                    if (r < P) best = select_bf16x2<OP>(w[r][k], best);
                o[k] = best;
            }
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Element-wise form: reduce element in_off + i of each rank buffer base[r]
// and store it as element i of dst[k], k < ndst.  Used for ragged tails and
// unaligned buffers, and (with i < 0) for the elements just before buffers
// that the vector kernel was handed from their first 16-byte boundary on.
template <int DT, int OP>
__device__ __forceinline__ void reduce_elem(const void *const *base, int64_t in_off, int64_t i,
                                            int P, void *const *dst, int ndst, float scale,
                                            int pow2)
{
    const int64_t j = in_off + i;
    if constexpr (DT == DT_I32) {
        int32_t acc = static_cast<const int32_t *>(base[0])[j];
        for (int r = 1; r < P; ++r) acc = pick_i<OP>(acc, static_cast<const int32_t *>(base[r])[j]);
        for (int k = 0; k < ndst; ++k) static_cast<int32_t *>(dst[k])[i] = acc;
    } else if constexpr (DT == DT_F32) {
        float acc = static_cast<const float *>(base[0])[j];
        for (int r = 1; r < P; ++r) {
            const float x = static_cast<const float *>(base[r])[j];
            if constexpr (OP == DT_SUM || OP == DT_AVG || OP == DT_SUM_STEPWISE) acc = __fadd_rn(acc, x);
            else acc = take_f<OP>(x, acc) ? x : acc;
        }
        if constexpr (OP == DT_AVG) acc = avg_of(acc, P, scale, pow2);
        for (int k = 0; k < ndst; ++k) static_cast<float *>(dst[k])[i] = acc;
    } else {
        float acc = bf16_to_f32(static_cast<const uint16_t *>(base[0])[j]);
        for (int r = 1; r < P; ++r) {
            const float x = bf16_to_f32(static_cast<const uint16_t *>(base[r])[j]);
            if constexpr (OP == DT_SUM || OP == DT_AVG) acc = __fadd_rn(acc, x);
            else if constexpr (OP == DT_SUM_STEPWISE) acc = round_bf16(__fadd_rn(acc, x));
            else acc = take_f<OP>(x, acc) ? x : acc;
        }
        uint16_t b;
        if constexpr (OP == DT_SUM || OP == DT_AVG || OP == DT_SUM_STEPWISE) {
            if constexpr (OP == DT_AVG) acc = avg_of(acc, P, scale, pow2);
            b = f32_to_bf16(acc);
        } else {
            b = (uint16_t)(__float_as_uint(acc) >> 16);   // the chosen element's bits
        }
        for (int k = 0; k < ndst; ++k) static_cast<uint16_t *>(dst[k])[i] = b;
    }
}

}  // namespace dt
