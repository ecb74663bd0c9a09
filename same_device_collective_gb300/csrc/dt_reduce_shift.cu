// Reduction (AllReduce, ReduceScatter) for rank buffers at different
// offsets past a 16-byte boundary.
//
// The vector kernel (dt_reduce.cu) needs every buffer of a job at one offset.
// When the inputs lie at different offsets -- views into larger tensors, each
// rank's at its own element -- this kernel keeps the 16-byte path: the job's
// outputs decide the chunk grid (their elements before the first 16-byte
// boundary and after the last whole vector go element by element), and each
// rank's input for a chunk is read as aligned 16-byte vectors and
// funnel-shifted into place (dt_shift.cuh).  Each warp covers 31 chunks per
// step: its 32 lanes load 32 consecutive aligned vectors per rank, and lanes
// 0..30 combine their own vector with the next lane's.  The arithmetic is
// the vector kernel's (reduce_vec16: ascending ranks, fp32 accumulation, one
// rounding at the store), so results are identical.
#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_math.cuh"
#include "dt_reduce_shift.h"
#include "dt_shift.cuh"
#include "dt_timeline.cuh"
#include "dt_bounds.cuh"

namespace dt {
namespace {

template <int DT, int OP, int PMAX>
__global__ void __launch_bounds__(kThreads)
reduce_shift_kernel(const __grid_constant__ ReduceParams p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;   // elements per 16-byte vector
    constexpr int ES = 16 / EPV;
    constexpr int kChunksPerWarp = 31;
    const int P = p.P;
    const int j = blockIdx.y;
    void *const *dst = p.out + j * p.out_per_job;
    const int ndst = p.out_per_job;
    // the outputs' elements before their first 16-byte boundary
    uint64_t dh = ((16 - (reinterpret_cast<uintptr_t>(dst[0]) & 15)) & 15) / ES;
    if (dh > p.n) dh = p.n;
    const uint64_t nch = (p.n - dh) / EPV;
    const int64_t in_elem_off = (int64_t)j * (int64_t)p.job_stride;
    const uint64_t out_byte = dh * ES;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t warps = (uint64_t)gridDim.x * (kThreads / 32);
    for (uint64_t base = ((uint64_t)blockIdx.x * (kThreads / 32) + warp) * kChunksPerWarp; base < nch;
         base += warps * kChunksPerWarp) {
        const uint64_t c = base + lane;           // lanes 0..30: chunk c; lane 31 only loads
        uint4 x[PMAX];
#pragma unroll
        for (int r = 0; r < PMAX; ++r) {
            x[r] = make_uint4(0, 0, 0, 0);
            if (r < P) {
                const unsigned char *ip =
                    static_cast<const unsigned char *>(p.in[r]) + (in_elem_off + (int64_t)dh) * ES;
                const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(ip) & 15);
                // vector c holds bytes of chunk c (c < nch) and, when sh > 0,
                // of chunk c - 1 (c <= nch)
                const uint4 *a = reinterpret_cast<const uint4 *>(ip - sh) + c;
                if ((c < nch || (sh && c == nch)) &&
                    DT_IN_BOUNDS(vector_touches(a, p.in_lo[r], p.in_hi[r]), p.sink, kBoundsReduceShift, r, a,
                                 p.in_lo[r]))
                    x[r] = __ldcs(a);
            }
        }
#pragma unroll
        for (int r = 0; r < PMAX; ++r) {
            if (r < P) {   // P is the same for every lane: the shuffle is warp-uniform
                const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(
                    static_cast<const unsigned char *>(p.in[r]) + (in_elem_off + (int64_t)dh) * ES) & 15);
                const uint4 nx = shfl_down_uint4(x[r]);   // every lane sends before any overwrites
                if (sh) x[r] = shift_pair(x[r], nx, sh);
            }
        }
        if (lane < kChunksPerWarp && c < nch) {
            const uint4 y = reduce_vec16<DT, OP, PMAX>(x, P, p.avg_scale, p.avg_pow2);
            for (int k = 0; k < ndst; ++k) {
                uint4 *a = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(dst[k]) + out_byte) + c;
                const int q = j * p.out_per_job + k;   // for the bounds checks
                (void)q;
                if (DT_IN_BOUNDS(span_in(a, 16, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsReduceShift,
                                 DT_MAX_RANKS + q, a, p.out_lo[q]))
                    __stcg(a, y);
            }
        }
    }

    // the elements before the outputs' boundary and after the last whole chunk
    if (blockIdx.x == 0) {
        for (uint64_t i = threadIdx.x; i < dh; i += kThreads)
            if (DT_REDUCE_ELEM_OK(ES, p, kBoundsReduceShift, in_elem_off, (int64_t)i, dst, ndst, j))
                reduce_elem<DT, OP>(p.in, in_elem_off, (int64_t)i, P, dst, ndst, p.avg_scale, p.avg_pow2);
        for (uint64_t i = dh + nch * EPV + threadIdx.x; i < p.n; i += kThreads)
            if (DT_REDUCE_ELEM_OK(ES, p, kBoundsReduceShift, in_elem_off, (int64_t)i, dst, ndst, j))
                reduce_elem<DT, OP>(p.in, in_elem_off, (int64_t)i, P, dst, ndst, p.avg_scale, p.avg_pow2);
    }
    DT_TL_END_BLOCK(DT_TL_REDUCE_SHIFT);
}

using ShiftFn = void (*)(ReduceParams);

template <int DT, int OP>
ShiftFn pick_p(int P)
{
    if (P <= 2) return reduce_shift_kernel<DT, OP, 2>;
    if (P <= 4) return reduce_shift_kernel<DT, OP, 4>;
    if (P <= 8) return reduce_shift_kernel<DT, OP, 8>;
    return reduce_shift_kernel<DT, OP, 16>;
}

template <int DT>
ShiftFn pick_op(int op, int P)
{
    switch (op) {
    case DT_SUM: return pick_p<DT, DT_SUM>(P);
    case DT_MAX: return pick_p<DT, DT_MAX>(P);
    case DT_MIN: return pick_p<DT, DT_MIN>(P);
    case DT_AVG:
        if constexpr (DT != DT_I32) return pick_p<DT, DT_AVG>(P);
        return nullptr;
    case DT_SUM_STEPWISE:
        if constexpr (DT == DT_BF16) return pick_p<DT, DT_SUM_STEPWISE>(P);
        return pick_p<DT, DT_SUM>(P);   // fp32 / int32: identical results
    default: return nullptr;
    }
}

}  // namespace

DT_TL_BINDER(bind_timeline_reduce_shift)

cudaError_t launch_reduce_shift(const ReduceParams &p, int dtype, int op, int jobs, int device,
                                cudaStream_t s)
{
    ShiftFn fn = nullptr;
    if (dtype == DT_F32) fn = pick_op<DT_F32>(op, p.P);
    else if (dtype == DT_BF16) fn = pick_op<DT_BF16>(op, p.P);
    else if (dtype == DT_I32) fn = pick_op<DT_I32>(op, p.P);
    if (!fn) return cudaErrorInvalidValue;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;
    const uint64_t epv = dtype == DT_BF16 ? 8 : 4;
    const uint64_t per_block = (uint64_t)(kThreads / 32) * 31;   // chunks a block takes per step
    uint64_t want = (p.n / epv + per_block - 1) / per_block;
    if (want < 1) want = 1;
    // up to eight blocks per resident slot, as the vector kernel
    uint64_t cap = (uint64_t)8 * resident / jobs;
    if (cap < 1) cap = 1;
    const unsigned gx = (unsigned)(want < cap ? want : cap);
    return launch_kernel(fn, dim3(gx, (unsigned)jobs), dim3(kThreads), 0, s, false, p);
}

}  // namespace dt
