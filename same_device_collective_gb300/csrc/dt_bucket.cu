// Fused gradient-bucket all-reduce kernel: one launch per bucket.
//
// The hyper-parallel pipelining page ("异步融合 AllReduce 流水线优化",
// AllReduceParamGroup) all-reduces one fused gradient buffer per parameter
// group and then divides each gradient view by the replicate world size; DDP
// (PyTorch communication page §六.5) gathers gradients into 25 MB buckets so
// that one bandwidth-bound call replaces many latency-bound ones.  Here the
// bucket is never flattened: the host hands the kernel a chunk table (tensor
// slot, element range) and a table of the P rank pointers of every tensor, and
// each block reduces its chunks in place in every rank's gradient, reading
// each element once per rank and writing it once per rank.
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
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;
    __shared__ void *sp[DT_MAX_RANKS];
    const int P = p.P;
    pdl_begin();

    for (uint32_t c = blockIdx.x; c < p.nchunks; c += gridDim.x) {
        const BucketChunk ch = p.chunks[c];
        const uint32_t slot = ch.slot & 0x7FFFFFFFu;
        __syncthreads();   // the previous chunk is done with sp
        if (threadIdx.x < P) sp[threadIdx.x] = p.ptrs[(uint64_t)slot * P + threadIdx.x];
        __syncthreads();

        if (ch.slot >> 31) {
            const uint64_t nvec = ch.nelem / EPV;
            const uint64_t v0 = ch.begin / EPV;   // chunk starts are multiples of EPV
            const uint4 *in[PMAX];
#pragma unroll
            for (int r = 0; r < PMAX; ++r)
                in[r] = r < P ? static_cast<const uint4 *>(sp[r]) + v0 : nullptr;
            for (uint64_t base = threadIdx.x; base < nvec; base += (uint64_t)kThreads * U) {
                uint4 x[U][PMAX];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = base + (uint64_t)u * kThreads;
                    if (v < nvec) {
#pragma unroll
                        for (int r = 0; r < PMAX; ++r)
                            if (r < P) x[u][r] = __ldcs(in[r] + v);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = base + (uint64_t)u * kThreads;
                    if (v < nvec) {
                        const uint4 y = reduce_vec16<DT, OP, PMAX>(x[u], P, p.avg_scale, p.avg_pow2);
#pragma unroll
                        for (int r = 0; r < PMAX; ++r)
                            if (r < P) __stcs(static_cast<uint4 *>(sp[r]) + v0 + v, y);
                    }
                }
            }
            for (uint64_t i = nvec * EPV + threadIdx.x; i < ch.nelem; i += kThreads)
                reduce_elem<DT, OP>(sp, 0, ch.begin + i, P, sp, P, p.avg_scale, p.avg_pow2);
        } else {
            for (uint64_t i = threadIdx.x; i < ch.nelem; i += kThreads)
                reduce_elem<DT, OP>(sp, 0, ch.begin + i, P, sp, P, p.avg_scale, p.avg_pow2);
        }
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

}  // namespace

cudaError_t launch_bucket(const BucketParams &p, int dtype, int op, int device, cudaStream_t s)
{
    BucketFn fn = nullptr;
    if (dtype == DT_BF16) fn = op == DT_AVG ? pick<DT_BF16, DT_AVG>(p.P) : pick<DT_BF16, DT_SUM>(p.P);
    else if (dtype == DT_F32) fn = op == DT_AVG ? pick<DT_F32, DT_AVG>(p.P) : pick<DT_F32, DT_SUM>(p.P);
    if (!fn || (op != DT_AVG && op != DT_SUM)) return cudaErrorInvalidValue;
    if (p.nchunks == 0) return cudaSuccess;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;
    const unsigned gx = p.nchunks < (uint32_t)resident ? p.nchunks : (unsigned)resident;
    return launch_kernel(fn, dim3(gx), dim3(kThreads), 0, s, false, p);
}

}  // namespace dt
