// Fused gradient-bucket all-reduce kernel: one launch per bucket.
//
// The hyper-parallel pipelining page ("异步融合 AllReduce 流水线优化",
// AllReduceParamGroup) all-reduces one fused gradient buffer per parameter
// group and then divides each gradient view by the replicate world size; DDP
// (PyTorch communication page §六.5) gathers gradients into 25 MB buckets so
// that one bandwidth-bound call replaces many latency-bound ones.  Here the
// bucket is never flattened into a copy: the host hands the kernel a table of
// the bucket's tensors (their place in the bucket's flattened element space)
// and the P rank pointers of each, and every block reduces an equal,
// contiguous slice of that space in place in every rank's gradient, reading
// each element once per rank and writing it once per rank.  Equal slices keep
// the blocks balanced however uneven the tensor sizes are.
#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_math.cuh"

namespace dt {
namespace {

template <int PMAX>
struct BucketUnroll {   // 8 loads of 16 bytes in flight per thread (16 at P > 8)
    static constexpr int U = PMAX >= 8 ? 1 : 8 / PMAX;
};

template <int DT, int OP, int PMAX>
__global__ void __launch_bounds__(kThreads)
bucket_kernel(const __grid_constant__ BucketParams p)
{
    constexpr int U = BucketUnroll<PMAX>::U;
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;   // elements per 16-byte vector
    __shared__ void *sp[DT_MAX_RANKS];
    const int P = p.P;
    // Let the next kernel begin launching, then fetch this block's first
    // tensor entry and that tensor's P rank pointers before waiting for the
    // previous kernel: the plan table is staged by a host copy that precedes
    // the call's first kernel in stream order, and no kernel writes it.  The
    // gradients themselves are touched only after griddepcontrol.wait.  This
    // takes two dependent table reads off the start of every bucket.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t lo = (uint64_t)blockIdx.x * p.per_block;
    if (lo >= p.total) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const uint64_t hi = lo + p.per_block < p.total ? lo + p.per_block : p.total;
    uint32_t t = p.block_start[blockIdx.x];   // its first <= lo < hi
    BucketTensor bt = p.tensors[t];
    if (threadIdx.x < P) sp[threadIdx.x] = p.ptrs[(uint64_t)(bt.slot & 0x7FFFFFFFu) * P + threadIdx.x];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    for (;;) {
        const uint64_t s = (lo > bt.first ? lo : bt.first) - bt.first;   // local range [s, e)
        uint64_t e = hi - bt.first;
        if (e > bt.count) e = bt.count;
        if (s < e) {   // else only padding of this tensor lies in the slice
            uint64_t scalar_from = s;
            if (bt.slot >> 31) {
                const uint64_t vs = s / EPV, ve = e / EPV;   // s is a multiple of EPV
                for (uint64_t base = vs + threadIdx.x; base < ve; base += (uint64_t)kThreads * U) {
                    uint4 x[U][PMAX];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const uint64_t v = base + (uint64_t)u * kThreads;
                        if (v < ve) {
#pragma unroll
                            for (int r = 0; r < PMAX; ++r)
                                if (r < P) x[u][r] = __ldcs(static_cast<const uint4 *>(sp[r]) + v);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const uint64_t v = base + (uint64_t)u * kThreads;
                        if (v < ve) {
                            const uint4 y = reduce_vec16<DT, OP, PMAX>(x[u], P, p.avg_scale, p.avg_pow2);
#pragma unroll
                            for (int r = 0; r < PMAX; ++r)
                                if (r < P) __stcs(static_cast<uint4 *>(sp[r]) + v, y);
                        }
                    }
                }
                scalar_from = ve * EPV;   // ragged end of the tensor, if it is in this slice
            }
            for (uint64_t i = scalar_from + threadIdx.x; i < e; i += kThreads)
                reduce_elem<DT, OP>(sp, 0, i, P, sp, P, p.avg_scale, p.avg_pow2);
        }
        if (++t >= p.ntensors) break;
        bt = p.tensors[t];
        if (bt.first >= hi) break;
        __syncthreads();   // every thread is done with the previous tensor's pointers
        if (threadIdx.x < P) sp[threadIdx.x] = p.ptrs[(uint64_t)(bt.slot & 0x7FFFFFFFu) * P + threadIdx.x];
        __syncthreads();
    }
}

using BucketFn = void (*)(BucketParams);

template <int DT, int OP>
BucketFn pick(int P)
{
    if (P <= 2) return bucket_kernel<DT, OP, 2>;
    if (P <= 4) return bucket_kernel<DT, OP, 4>;
    if (P <= 8) return bucket_kernel<DT, OP, 8>;
    return bucket_kernel<DT, OP, 16>;
}

BucketFn pick_fn(int dtype, int op, int P)
{
    if (op != DT_AVG && op != DT_SUM) return nullptr;
    if (dtype == DT_BF16) return op == DT_AVG ? pick<DT_BF16, DT_AVG>(P) : pick<DT_BF16, DT_SUM>(P);
    if (dtype == DT_F32) return op == DT_AVG ? pick<DT_F32, DT_AVG>(P) : pick<DT_F32, DT_SUM>(P);
    return nullptr;
}

}  // namespace

uint64_t bucket_padded(uint64_t count, int dtype)
{
    const uint64_t epv = dtype == DT_BF16 ? 8 : 4;
    return (count + epv - 1) / epv * epv;
}

cudaError_t bucket_grid(int dtype, int op, int P, uint64_t total, int device, uint32_t *blocks,
                        uint64_t *per_block)
{
    BucketFn fn = pick_fn(dtype, op, P);
    if (!fn) return cudaErrorInvalidValue;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;
    const uint64_t epv = dtype == DT_BF16 ? 8 : 4;
    // at least one full pass of the block's threads per slice
    const uint64_t min_slice = (uint64_t)kThreads * epv;
    uint64_t g = (total + min_slice - 1) / min_slice;
    // Up to sixteen slices per resident block: blocks that finish early take
    // the next slices, so SMs that stream slower do not stretch the bucket's
    // tail.  For 25 MiB buckets the minimum slice binds first, so every block
    // makes exactly one pass; that measured best (200 gradients of 8 ranks:
    // 440 us per call at one slice per resident block, 406 at four, 410 at
    // eight, whose last pass is mostly idle, 391 at one pass per block).  The
    // cap keeps the per-bucket start table bounded.
    constexpr uint64_t kSlicesPerResident = 16;
    if (g > (uint64_t)resident * kSlicesPerResident) g = (uint64_t)resident * kSlicesPerResident;
    if (g < 1) g = 1;
    uint64_t per = (total + g - 1) / g;
    per = (per + epv - 1) / epv * epv;
    if (per == 0) per = epv;
    *per_block = per;
    *blocks = (uint32_t)((total + per - 1) / per);
    if (*blocks == 0) *blocks = 1;
    return cudaSuccess;
}

cudaError_t launch_bucket(const BucketParams &p, int dtype, int op, int device, cudaStream_t s)
{
    BucketFn fn = pick_fn(dtype, op, p.P);
    if (!fn) return cudaErrorInvalidValue;
    if (p.total == 0 || p.ntensors == 0) return cudaSuccess;
    (void)device;
    const unsigned gx = (unsigned)((p.total + p.per_block - 1) / p.per_block);
    return launch_kernel(fn, dim3(gx), dim3(kThreads), 0, s, false, p);
}

}  // namespace dt
