// Signal-window barrier among the P ranks of a group, and the ordering test
// kernel built on it.
//
// The PyPTO page "Barrier：仅信号（Signals Only）" builds an N-rank barrier from
// two primitives: notify adds 1 (AtomicAdd) to a cell of a peer's signal
// window, wait blocks until a cell of one's own window reaches a threshold
// (Ge).  Rank r notifies every peer q != r at row r of q's window and then
// waits on every row s != r of its own window; a rank never notifies itself,
// so its own row stays 0.  Because the counters only grow, every reuse of the
// window raises the threshold: the g-th barrier waits for g.
//
// Here the window is int32 win[P][P] in HBM (win[q][r] is row r of rank q's
// window).  In the stand-alone barrier each rank is one warp of a single
// block (warps of one block are always resident together, so the ranks can
// wait on each other without a cooperative launch); in the ordering test
// each rank is a block of a cooperative launch.  Lane q of rank r's warp
// notifies peer q with a release reduction and then polls row q of rank r's
// window with acquire loads.  The generation is kept per rank on the device
// (rank_gen), so a captured and replayed launch still raises the threshold
// each time.  Every poll loop ends after the group's time limit (or an
// iteration bound); a rank that gives up records DT_ERR_TIMEOUT once in the
// error word and its host-mapped mirror and returns, so the GPU is never held.
#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_timeline.cuh"

namespace dt {
namespace {

// The notify (AtomicAdd) and the poll (Ge).  kOrder makes them a release add
// and an acquire load at GPU scope, which order data written before the
// barrier in the same kernel against reads after it.  The stand-alone barrier
// kernel has no such data: the kernels before it finished and flushed before
// it started (griddepcontrol.wait), and the kernels after it start only once
// it has finished, so it only counts arrivals, with relaxed GPU-scope atomics
// and strong loads that read L2 (11% less latency per barrier than the ordered
// forms at P=16).
template <bool kOrder>
__device__ __forceinline__ void notify_add(int32_t *cell)
{
    if (kOrder) asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(cell), "r"(1) : "memory");
    else asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(cell), "r"(1) : "memory");
}

template <bool kOrder>
__device__ __forceinline__ int32_t load_poll(const int32_t *cell)
{
    int32_t v;
    if (kOrder) asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cell) : "memory");
    else asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cell) : "memory");
    return v;
}

// Run by the 32 lanes of one warp for rank r; true when every wait ended in
// time.  kFence orders writes made earlier in the same kernel (by any thread
// of the block, after a __syncthreads) before the notifies, and the peers'
// writes before the block's later reads; the stand-alone barrier kernel has
// no such writes (everything before it finished in stream order) and skips it.
template <bool kFence>
__device__ bool rank_barrier(const BarrierParams &p, int r)
{
    const int lane = threadIdx.x & 31;
    const int P = p.P;
    const int32_t g = p.rank_gen[r] + 1;
    const bool peer = lane < P && lane != r;

    if (kFence) __threadfence();         // this rank's earlier writes before its notifies
    if (peer) notify_add<kFence>(&p.win[lane * P + r]);

    bool ok = true;
    if (peer) {
        const int32_t want = g + p.extra;
        const uint64_t t0 = global_ns();
        const uint64_t max_polls = p.sink.timeout_ns / 256 + 4096;
        uint32_t sleep_ns = 0;
        for (uint64_t it = 0;; ++it) {
            const int32_t v = load_poll<kFence>(&p.win[r * P + lane]);
            if ((int32_t)(v - want) >= 0) break;          // Ge, safe across wrap-around
            if (it >= max_polls || global_ns() - t0 > p.sink.timeout_ns) { ok = false; break; }
            if (it >= 64) {
                sleep_ns = sleep_ns ? (sleep_ns < 256 ? sleep_ns * 2 : 256) : 32;
                __nanosleep(sleep_ns);
            }
        }
    }
    if (kFence) __threadfence();         // peers' writes before this rank's later reads
    const unsigned bad = __ballot_sync(0xFFFFFFFFu, !ok);
    if (lane == 0) {
        if (bad) record_error(p.sink, DT_ERR_TIMEOUT, r, __ffs(bad) - 1, g);
        p.rank_gen[r] = g;
    }
    __syncwarp();
    return bad == 0;
}

// One block of 32 * P threads: warp r is rank r.
__global__ void __launch_bounds__(32 * DT_MAX_RANKS) barrier_kernel(const __grid_constant__ BarrierParams p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    rank_barrier<false>(p, threadIdx.x >> 5);
    DT_TL_END_BLOCK(DT_TL_BARRIER);
}

__device__ void copy_bytes(unsigned char *dst, const unsigned char *src, uint64_t n)
{
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | n) & 15) == 0;
    if (vec) {
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (uint64_t i = threadIdx.x; i < n / 16; i += blockDim.x) d[i] = s[i];
    } else {
        for (uint64_t i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
    }
}

// The barrier page's ordering example: stage, barrier, read the next rank.
__global__ void __launch_bounds__(kThreads) ring_kernel(const __grid_constant__ RingParams p)
{
    __shared__ int ok;
    const int r = blockIdx.x;
    pdl_begin();
    copy_bytes(p.stage[r], p.in[r], p.bytes);
    __syncthreads();
    if (threadIdx.x < 32) {
        const bool passed = rank_barrier<true>(p.bar, r);
        if (threadIdx.x == 0) ok = passed;
    }
    __syncthreads();
    if (ok) copy_bytes(p.out[r], p.stage[(r + 1) % p.bar.P], p.bytes);
}

#ifdef DT_TIMELINE
// dt_timeline_mark: one thread records a mark carrying the caller's tag
__global__ void mark_kernel(uint32_t tag)
{
    const uint64_t t = global_ns();
    const TimelineSink s = g_timeline;
    if (!s.rec) return;
    const unsigned long long k = atomicAdd(s.count, 1ull);
    if (k >= s.cap) return;
    uint64_t grid;
    uint32_t sm;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(grid));
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    dt_timeline_record r;
    r.grid = grid;
    r.kind = DT_TL_MARK;
    r.block = tag;
    r.sm = sm;
    r.pad = 0;
    r.t_start = r.t_waited = r.t_end = t;
    s.rec[k] = r;
}
#endif

}  // namespace

DT_TL_BINDER(bind_timeline_barrier)

#ifdef DT_TIMELINE
cudaError_t launch_timeline_mark(uint32_t tag, cudaStream_t s)
{
    return launch_kernel(mark_kernel, dim3(1), dim3(1), 0, s, false, tag);
}
#endif

cudaError_t launch_barrier(const BarrierParams &p, cudaStream_t s)
{
    return launch_kernel(barrier_kernel, dim3(1), dim3(32 * p.P), 0, s, false, p);
}

cudaError_t launch_ring(const RingParams &p, cudaStream_t s)
{
    return launch_kernel(ring_kernel, dim3(p.bar.P), dim3(kThreads), 0, s, true, p);
}

}  // namespace dt
