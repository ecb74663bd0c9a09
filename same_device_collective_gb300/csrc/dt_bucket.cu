// Fused gradient-bucket all-reduce kernel: one launch per bucket.
//
// The hyper-parallel pipelining page ("异步融合 AllReduce 流水线优化",
// AllReduceParamGroup) all-reduces one fused gradient buffer per parameter
// group and then divides each gradient view by the replicate world size; DDP
// (PyTorch communication page §六.5) gathers gradients into 25 MB buckets so
// that one bandwidth-bound call replaces many latency-bound ones.  Here the
// bucket is never flattened into a copy: the host hands the kernel a table of
// the bucket's tensors and the P rank pointers of each, and every block
// reduces one slice of one tensor in place in every rank's gradient, reading
// each element once per rank and writing it once per rank.  The slices have
// one length for the whole bucket (a tensor's last one is shorter), which
// keeps the blocks balanced however uneven the tensor sizes are.
#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_math.cuh"
#include "dt_timeline.cuh"
#include "dt_bounds.cuh"

namespace dt {
namespace {

template <int PMAX>
struct BucketUnroll {   // 8 loads of 16 bytes in flight per thread (16 at P > 8)
    static constexpr int U = PMAX >= 8 ? 1 : 8 / PMAX;
};

// Threads per bucket block.  Blocks make one pass over their slice, so the
// block size sets the slice and with it how long the last blocks of a bucket
// run alone at its end.  On the 200-gradient, 8-rank workload, with slices cut
// at tensor ends: 256 threads 363.0 us per call, 192 363.1, 128 364.2, 64
// 390-408, and two passes of 128 threads 372.7.  (While slices could cross
// into a second tensor, 128 threads had been best: 380 against 384 at 256.)
constexpr int kBucketThreads = 256;

// The signal-window barrier between this bucket and the next, run by the
// grid's extra last block (the page's notify / wait with a generation; the
// stand-alone form is barrier_kernel, one warp per rank).  The data blocks
// count themselves out in the group's finished-block counter as they end;
// this block, dispatched after all of them, waits for the previous kernel,
// then until the count is complete, resets it for the next bucket kernel, and
// then acts for all P ranks at once: thread cell (r, q) adds 1 to row r of
// peer q's window (rank r's notify, AtomicAdd) and then waits until row q of
// rank r's window reaches rank r's generation (Ge).  The next kernel stores
// nothing before this grid has completed, so it sees every gradient this
// bucket wrote, as it would after a barrier kernel -- whose own
// launch-to-completion hop is what this saves at every bucket boundary.
// Every wait is bounded: one that runs out records DT_ERR_TIMEOUT and ends
// the block.
__device__ void bucket_barrier_block(const BucketParams &p)
{
    __shared__ int ok;
    const int P = p.P;
    int32_t *rank_gen = p.win + P * P;
    uint32_t *done = reinterpret_cast<uint32_t *>(rank_gen + P);
    // The previous kernel may still be running (this grid was launched while
    // it drained): it may be a bucket kernel whose own blocks are still
    // counting themselves out and whose barrier block has yet to update the
    // window.  Touch neither before it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        ok = 1;
        const uint32_t others = gridDim.x - 1;
        const uint64_t t0 = global_ns();
        const uint64_t max_polls = p.sink.timeout_ns / 64 + 4096;
        for (uint64_t it = 0;; ++it) {
            uint32_t v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(done) : "memory");
            if (v >= others) break;
            if (it >= max_polls || global_ns() - t0 > p.sink.timeout_ns) {
                record_error(p.sink, DT_ERR_TIMEOUT, -1, -1, 0);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        if (ok) asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(done), "r"(0u) : "memory");
    }
    __syncthreads();
    if (!ok) return;
    for (int c = threadIdx.x; c < P * P; c += blockDim.x) {
        const int r = c / P, q = c - r * P;
        if (r != q) asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(&p.win[q * P + r]), "r"(1) : "memory");
    }
    for (int c = threadIdx.x; c < P * P; c += blockDim.x) {
        const int r = c / P, s = c - r * P;
        if (r == s) continue;
        const int32_t g = rank_gen[r] + 1;
        const int32_t *cell = &p.win[r * P + s];
        const uint64_t t0 = global_ns();
        const uint64_t max_polls = p.sink.timeout_ns / 64 + 4096;
        for (uint64_t it = 0;; ++it) {
            int32_t v;
            asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cell) : "memory");
            if ((int32_t)(v - g) >= 0) break;             // Ge, safe across wrap-around
            if (it >= max_polls || global_ns() - t0 > p.sink.timeout_ns) {
                record_error(p.sink, DT_ERR_TIMEOUT, r, s, g);
                break;
            }
            if (it >= 64) __nanosleep(128);
        }
    }
    __syncthreads();   // every rank has read its generation and passed its wait
    if (threadIdx.x < P) rank_gen[threadIdx.x] += 1;
}

// A data block of a bucket followed by a barrier counts itself out.  The
// barrier block only needs to know that every data block has finished its
// work: the next kernel waits for this whole grid before it reads anything.
__device__ __forceinline__ void count_out(const BucketParams &p)
{
    if (!p.win) return;
    __syncthreads();
    if (threadIdx.x == 0)
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;"
                     ::"l"(p.win + p.P * p.P + p.P), "r"(1u) : "memory");
}

template <int DT, int OP, int PMAX>
__global__ void __launch_bounds__(kBucketThreads)
bucket_kernel(const __grid_constant__ BucketParams p)
{
    constexpr int U = BucketUnroll<PMAX>::U;
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;   // elements per 16-byte vector
    __shared__ void *sp[DT_MAX_RANKS];
    const int P = p.P;
    // Fetch this block's tensor entry and that tensor's P rank pointers before
    // waiting for the previous kernel: the plan table is staged by a host copy
    // that precedes the call's first kernel in stream order, and no kernel
    // writes it.  This takes two dependent table reads off the start of every
    // bucket.  A block works on one tensor: blocks whose slice crossed into a
    // second tensor took it after the first, ran 2.7x as long as the others
    // and were the last to end in nearly every bucket.
    //
    // Every bucket kernel of a call after the first also loads its block's
    // first pass of gradients before the wait, so the blocks that become
    // resident while the previous bucket drains (up to one per free slot)
    // have their data in flight when it completes; nothing is stored before
    // the wait, and so before the barrier between the buckets.  Those loads
    // read this bucket's tensors, which no kernel of the call writes before
    // this one; the call's first kernel lets the next launch begin only after
    // its own wait, so no early load can overtake the work queued before the
    // call.  The other kernels let the next one launch at once.
    DT_TL_BEGIN();
    if (p.early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.win && blockIdx.x == gridDim.x - 1) {
        bucket_barrier_block(p);
        DT_TL_WAITED();
        DT_TL_END_BLOCK(DT_TL_BUCKET_BARRIER);
        return;
    }
    const uint32_t t = p.block_start[blockIdx.x];
    const BucketTensor bt = p.tensors[t];
    const uint64_t lo = (uint64_t)(blockIdx.x - bt.block0) * p.per_block;   // within the tensor
    const uint64_t hi = lo + p.per_block < bt.count ? lo + p.per_block : bt.count;
    if (threadIdx.x < P) sp[threadIdx.x] = p.ptrs[(uint64_t)(bt.slot & 0x7FFFFFFFu) * P + threadIdx.x];

    uint4 x[U][PMAX];
    // U vectors from every rank at vector positions base, base + kBucketThreads, ... below ve
    auto load_vectors = [&](uint64_t base, uint64_t ve) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = base + (uint64_t)u * kBucketThreads;
            if (v < ve) {
#pragma unroll
                for (int r = 0; r < PMAX; ++r) {
                    if (r < P) {
                        const uint4 *a = static_cast<const uint4 *>(sp[r]) + v;
                        if (DT_IN_BOUNDS(span_in(a, 16, reinterpret_cast<uint64_t>(sp[r]),
                                                 reinterpret_cast<uint64_t>(sp[r]) + bt.count * (16 / EPV)),
                                         p.sink, kBoundsBucket, (int)t, a, reinterpret_cast<uint64_t>(sp[r])))
                            x[u][r] = __ldcs(a);
                    }
                }
            }
        }
    };
    // the slice's whole vectors (all ranks 16-byte aligned), then its other elements
    const bool aligned = bt.slot >> 31;
    const uint64_t vs = lo / EPV, ve = aligned ? hi / EPV : vs;   // lo is a multiple of EPV
    bool loaded = false;   // x holds the first pass
    if (p.early) {
        __syncthreads();   // sp
        if (vs + threadIdx.x < ve) {
            load_vectors(vs + threadIdx.x, ve);
            loaded = true;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    DT_TL_WAITED();

    for (uint64_t base = vs + threadIdx.x; base < ve; base += (uint64_t)kBucketThreads * U) {
        if (loaded)
            loaded = false;   // loaded before the wait
        else
            load_vectors(base, ve);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = base + (uint64_t)u * kBucketThreads;
            if (v < ve) {
                const uint4 y = reduce_vec16<DT, OP, PMAX>(x[u], P, p.avg_scale, p.avg_pow2);
#pragma unroll
                for (int r = 0; r < PMAX; ++r) {
                    if (r < P) {
                        uint4 *a = static_cast<uint4 *>(sp[r]) + v;
                        if (DT_IN_BOUNDS(span_in(a, 16, reinterpret_cast<uint64_t>(sp[r]),
                                                 reinterpret_cast<uint64_t>(sp[r]) + bt.count * (16 / EPV)),
                                         p.sink, kBoundsBucket, (int)t, a, reinterpret_cast<uint64_t>(sp[r])))
                            __stcs(a, y);
                    }
                }
            }
        }
    }
    // the ragged end of the tensor, if it is in this slice, or the whole slice
    // of a tensor whose ranks are not all 16-byte aligned
    for (uint64_t i = ve * EPV + threadIdx.x; i < hi; i += kBucketThreads)
        if (DT_IN_BOUNDS(i < bt.count, p.sink, kBoundsBucket, (int)t, (const void *)(uintptr_t)i, 0))
            reduce_elem<DT, OP>(sp, 0, (int64_t)i, P, sp, P, p.avg_scale, p.avg_pow2);
    count_out(p);
    DT_TL_END_BLOCK(DT_TL_BUCKET);
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

DT_TL_BINDER(bind_timeline_bucket)

uint64_t bucket_padded(uint64_t count, int dtype)
{
    const uint64_t epv = dtype == DT_BF16 ? 8 : 4;
    return (count + epv - 1) / epv * epv;
}

uint64_t bucket_tensor_blocks(uint64_t count, int dtype, uint64_t per_block)
{
    return (bucket_padded(count, dtype) + per_block - 1) / per_block;
}

cudaError_t bucket_grid(int dtype, int op, int P, uint64_t total, int device, uint32_t *blocks,
                        uint64_t *per_block)
{
    BucketFn fn = pick_fn(dtype, op, P);
    if (!fn) return cudaErrorInvalidValue;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kBucketThreads, device, &resident);
    if (e != cudaSuccess) return e;
    const uint64_t epv = dtype == DT_BF16 ? 8 : 4;
    // at least one full pass of the block's threads per slice
    const uint64_t min_slice = (uint64_t)kBucketThreads * epv;
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

cudaError_t launch_bucket(const BucketParams &p, int dtype, int op, int device, cudaStream_t s,
                          bool *launched)
{
    if (launched) *launched = false;
    BucketFn fn = pick_fn(dtype, op, p.P);
    if (!fn) return cudaErrorInvalidValue;
    if (p.blocks == 0 || p.ntensors == 0) return cudaSuccess;
    (void)device;
    // data blocks, plus the barrier block when a barrier follows the bucket
    const unsigned gx = p.blocks + (p.win ? 1u : 0u);
    const cudaError_t e = launch_kernel(fn, dim3(gx), dim3(kBucketThreads), 0, s, false, p);
    if (launched) *launched = e == cudaSuccess;
    return e;
}

}  // namespace dt
