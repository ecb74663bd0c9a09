// One-pass reduction kernel for AllReduce and ReduceScatter among P ranks on
// one GPU.
//
// The same-device AllReduce of the DTorch collective-communication page
// (§2.3) publishes every rank's tensor and lets rank 0 add ranks 1..P-1 onto
// its own, one add kernel per rank, before handing the result back.  Here a
// single launch reads all P rank buffers straight from HBM: each thread loads
// its 16-byte vector from every rank before combining them (P x U loads in
// flight per thread), reduces in registers in ascending rank order, and
// stores the result to every destination.  HBM traffic is the algorithmic
// minimum: P reads and (number of outputs) writes per vector position.
// Inputs are read once, so their loads carry the evict-first (streaming) cache
// policy; results use the normal policy because the usual next consumer (the
// AllGather after a ReduceScatter) reads them straight back.
//
// Grid: blockIdx.y is the job (1 for AllReduce, P for ReduceScatter), and
// blockIdx.x strides over the job's vectors; the launcher sizes the grid to
// the work, up to eight times the blocks the SMs hold at once.
#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_math.cuh"
#include "dt_timeline.cuh"
#include "dt_bounds.cuh"

namespace dt {
namespace {

// Vector positions per thread per iteration (U), measured on GB300: a
// ReduceScatter keeps 8 loads of 16 bytes in flight per thread (U = 8 / P,
// 16 loads at P > 8), which its step needs; an AllReduce does best with one
// position per thread at every size (a P=2 fp32 AllReduce of 4 MiB per rank
// 3.8 -> 2.55 us in a CUDA graph, 16 MiB per rank +11%, P=4 256 MiB +3%),
// because its P output stores per position already keep the thread busy.
template <int PMAX>
struct Unroll {
    static constexpr int kScatter = PMAX >= 8 ? 1 : 8 / PMAX;
};

template <int DT, int OP, int PMAX, int U>
__global__ void __launch_bounds__(kThreads)
reduce_vec_kernel(const __grid_constant__ ReduceParams p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;   // elements per 16-byte vector
    const int P = p.P;
    const int j = blockIdx.y;
    const uint64_t nvec = p.n / EPV;
    const uint64_t in_off = (uint64_t)j * (p.job_stride / EPV);
    const uint64_t step = (uint64_t)gridDim.x * kThreads * U;
    void *const *dst = p.out + j * p.out_per_job;
    const int ndst = p.out_per_job;

    for (uint64_t base = (uint64_t)blockIdx.x * kThreads * U + threadIdx.x; base < nvec;
         base += step) {
        uint4 x[U][PMAX];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = base + (uint64_t)u * kThreads;
            if (v < nvec) {
#pragma unroll
                for (int r = 0; r < PMAX; ++r) {
                    if (r < P) {
                        const uint4 *a = static_cast<const uint4 *>(p.in[r]) + in_off + v;
                        if (DT_IN_BOUNDS(span_in(a, 16, p.in_lo[r], p.in_hi[r]), p.sink, kBoundsReduce, r, a,
                                         p.in_lo[r]))
                            x[u][r] = __ldcs(a);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = base + (uint64_t)u * kThreads;
            if (v < nvec) {
                const uint4 y = reduce_vec16<DT, OP, PMAX>(x[u], P, p.avg_scale, p.avg_pow2);
                for (int k = 0; k < ndst; ++k) {
                    uint4 *a = static_cast<uint4 *>(dst[k]) + v;
                    const int q = j * p.out_per_job + k;   // for the bounds checks
                    (void)q;
                    if (DT_IN_BOUNDS(span_in(a, 16, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsReduce,
                                     DT_MAX_RANKS + q, a, p.out_lo[q]))
                        __stcg(a, y);
                }
            }
        }
    }

    // ragged tail: the last n % EPV elements of the job, element by element,
    // and the head elements before the job's first vector
    if (blockIdx.x == 0) {
        const int64_t in_elem_off = (int64_t)j * (int64_t)p.job_stride;
        for (uint64_t i = nvec * EPV + threadIdx.x; i < p.n; i += kThreads)
            if (DT_REDUCE_ELEM_OK(16 / EPV, p, kBoundsReduce, in_elem_off, (int64_t)i, dst, ndst, j))
                reduce_elem<DT, OP>(p.in, in_elem_off, (int64_t)i, P, dst, ndst, p.avg_scale, p.avg_pow2);
        const int64_t hi = (int64_t)threadIdx.x - (int64_t)p.head;
        if (threadIdx.x < p.head &&
            DT_REDUCE_ELEM_OK(16 / EPV, p, kBoundsReduce, in_elem_off, hi, dst, ndst, j))
            reduce_elem<DT, OP>(p.in, in_elem_off, hi, P, dst, ndst, p.avg_scale, p.avg_pow2);
    }
    DT_TL_END_BLOCK(DT_TL_REDUCE);
}

// Any alignment: element by element, same arithmetic.
template <int DT, int OP>
__global__ void __launch_bounds__(kThreads)
reduce_scalar_kernel(const __grid_constant__ ReduceParams p)
{
    pdl_begin();
    const int j = blockIdx.y;
    const int64_t in_elem_off = (int64_t)j * (int64_t)p.job_stride;
    void *const *dst = p.out + j * p.out_per_job;
    for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < p.n;
         i += (uint64_t)gridDim.x * kThreads)
        if (DT_REDUCE_ELEM_OK(DT == DT_BF16 ? 2 : 4, p, kBoundsReduce, in_elem_off, (int64_t)i, dst,
                              p.out_per_job, j))
            reduce_elem<DT, OP>(p.in, in_elem_off, (int64_t)i, p.P, dst, p.out_per_job, p.avg_scale,
                                p.avg_pow2);
}

using ReduceFn = void (*)(ReduceParams);

struct KernelInfo {
    ReduceFn fn = nullptr;
    int per_vec_iter = 1;   // vectors (or elements) per thread per iteration
};

template <int DT, int OP, int PMAX>
KernelInfo pick_unroll(bool scatter)
{
    constexpr int U = Unroll<PMAX>::kScatter;
    if (scatter && U > 1) return KernelInfo{reduce_vec_kernel<DT, OP, PMAX, U>, U};
    return KernelInfo{reduce_vec_kernel<DT, OP, PMAX, 1>, 1};
}

template <int DT, int OP>
KernelInfo pick_vec(int P, bool scatter)
{
    if (P <= 2) return pick_unroll<DT, OP, 2>(scatter);
    if (P <= 4) return pick_unroll<DT, OP, 4>(scatter);
    if (P <= 8) return pick_unroll<DT, OP, 8>(scatter);
    return pick_unroll<DT, OP, 16>(scatter);
}

template <int DT>
KernelInfo pick_op(int op, int P, bool vec, bool scatter)
{
    KernelInfo k;
    switch (op) {
    case DT_SUM: k = vec ? pick_vec<DT, DT_SUM>(P, scatter) : KernelInfo{reduce_scalar_kernel<DT, DT_SUM>, 1}; break;
    case DT_MAX: k = vec ? pick_vec<DT, DT_MAX>(P, scatter) : KernelInfo{reduce_scalar_kernel<DT, DT_MAX>, 1}; break;
    case DT_MIN: k = vec ? pick_vec<DT, DT_MIN>(P, scatter) : KernelInfo{reduce_scalar_kernel<DT, DT_MIN>, 1}; break;
    case DT_AVG:
        if constexpr (DT != DT_I32)
            k = vec ? pick_vec<DT, DT_AVG>(P, scatter) : KernelInfo{reduce_scalar_kernel<DT, DT_AVG>, 1};
        break;
    case DT_SUM_STEPWISE:   // only bf16 rounds between adds; the launcher maps the rest to SUM
        if constexpr (DT == DT_BF16)
            k = vec ? pick_vec<DT, DT_SUM_STEPWISE>(P, scatter)
                    : KernelInfo{reduce_scalar_kernel<DT, DT_SUM_STEPWISE>, 1};
        break;
    default: break;
    }
    return k;
}

}  // namespace

DT_TL_BINDER(bind_timeline_reduce)

constexpr int kGridPerResident = 8;

cudaError_t launch_reduce(const ReduceParams &p, int dtype, int op, int jobs, bool vec,
                          int device, cudaStream_t s)
{
    KernelInfo k;
    if (op == DT_SUM_STEPWISE && dtype != DT_BF16) op = DT_SUM;   // identical results
    const bool scatter = jobs > 1;
    if (dtype == DT_F32) k = pick_op<DT_F32>(op, p.P, vec, scatter);
    else if (dtype == DT_BF16) k = pick_op<DT_BF16>(op, p.P, vec, scatter);
    else if (dtype == DT_I32) k = pick_op<DT_I32>(op, p.P, vec, scatter);
    if (!k.fn) return cudaErrorInvalidValue;

    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(k.fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;

    const int epv = vec ? (dtype == DT_BF16 ? 8 : 4) : 1;
    const uint64_t units = p.n / epv;
    const uint64_t per_block = (uint64_t)kThreads * k.per_vec_iter;
    uint64_t want = (units + per_block - 1) / per_block;
    if (want < 1) want = 1;
    // Eight blocks per resident slot: the grid-stride work of a large call is
    // then handed out block by block as SMs free up, so SMs that stream slower
    // take fewer blocks and no SM's share stretches the tail (measured on the
    // RS+AG step: 104.0 us at one block per slot, 100.7 us at eight; a P=8
    // 64 MiB AllReduce 6.33 -> 6.76 TB/s).
    uint64_t cap = (uint64_t)kGridPerResident * resident / jobs;
    if (cap < 1) cap = 1;
    const unsigned gx = (unsigned)(want < cap ? want : cap);

    return launch_kernel(k.fn, dim3(gx, (unsigned)jobs), dim3(kThreads), 0, s, false, p);
}

}  // namespace dt
