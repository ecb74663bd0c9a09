// Host side of the same-device collective library: the group object,
// argument validation, launch planning and the C ABI entry points.
//
// DTorch's same-device backend ("集合通信组件" §2.3, §3.4) moves every
// collective through a TensorStore: each rank thread publishes its tensor
// under a key (SrcSet, which records a CUDA event), consumers wait on that
// event (DestGet), and two host barriers (Reset) close every operation.  A
// group-wide call here plays all of those roles at once: the P rank pointers
// the caller passes are the store's slots, they travel to the device as the
// kernel's parameter block (or, for buckets, as a table staged in HBM), and
// ordering is the order of the caller's stream.
#include <cxxabi.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <new>
#include <string>
#include <thread>
#include <tuple>
#include <unordered_map>
#include <utility>
#include <vector>

#include "dt_group.h"
#include "dt_reduce_shift.h"
#include "dt_timeline.h"

// Built with -DDT_NVTX (DT_NVTX=1 when building), every public entry point
// opens an NVTX range named after itself for profiler timelines.
#ifdef DT_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace
#define DT_TRACE() NvtxRange dt_nvtx_range_(__func__)
#else
#define DT_TRACE() ((void)0)
#endif

namespace dt {

static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool pdl_enabled()
{
    static const bool on = [] {
        const char *env = std::getenv("DT_PDL");
        return !(env && env[0] == '0');
    }();
    return on;
}

bool log_enabled()
{
    static const bool on = [] {
        const char *env = std::getenv("DT_LOG");
        return env && env[0] && env[0] != '0';
    }();
    return on;
}

bool debug_enabled()
{
    static const bool on = [] {
        const char *env = std::getenv("DT_DEBUG");
        return env && env[0] && env[0] != '0';
    }();
    return on;
}

cudaError_t debug_sync(cudaStream_t s, cudaError_t launched)
{
    if (launched != cudaSuccess) return launched;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return e;
    if (cap != cudaStreamCaptureStatusNone) return cudaSuccess;   // nothing runs while capturing
    return cudaStreamSynchronize(s);
}

void log_launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool cooperative,
                cudaError_t result)
{
    const char *mangled = nullptr;
    std::string name = "?";
    if (cudaFuncGetName(&mangled, fn) == cudaSuccess && mangled) {
        int status = 0;
        char *d = abi::__cxa_demangle(mangled, nullptr, nullptr, &status);
        name = (status == 0 && d) ? d : mangled;
        std::free(d);
    }
    std::fprintf(stderr,
                 "dt: launch %s grid=(%u,%u,%u) block=(%u,%u,%u) smem=%zu stream=%p pdl=%d "
                 "cooperative=%d -> %s\n",
                 name.c_str(), grid.x, grid.y, grid.z, block.x, block.y, block.z, smem,
                 static_cast<void *>(s), pdl_enabled() ? 1 : 0, cooperative ? 1 : 0,
                 cudaGetErrorName(result));
}

int sm_count(int device)
{
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(device);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
        n = 1;
    cache[device] = n;
    return n;
}

uint64_t l2_bytes(int device)
{
    static std::mutex mu;
    static std::unordered_map<int, uint64_t> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(device);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, device) != cudaSuccess || n < 0) n = 0;
    cache[device] = (uint64_t)n;
    return (uint64_t)n;
}

cudaError_t resident_blocks(const void *fn, int threads, int device, int *out, size_t dyn_smem)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int, size_t>, int> cache;
    const auto key = std::make_tuple(fn, device, threads, dyn_smem);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) { *out = it->second; return cudaSuccess; }
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, dyn_smem);
    if (e != cudaSuccess) return e;
    const int n = sm_count(device) * (per_sm > 0 ? per_sm : 1);
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    *out = n;
    return cudaSuccess;
}

}  // namespace dt

namespace {

using dt::DevError;

size_t elem_bytes(int dtype) { return dtype == DT_BF16 ? 2 : 4; }
bool valid_dtype(int dtype) { return dtype == DT_F32 || dtype == DT_BF16 || dtype == DT_I32; }
bool valid_op(int op) { return op >= DT_SUM && op <= DT_SUM_STEPWISE; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Switch to the group's device for the duration of a call.
struct DeviceScope {
    int prev = -1;
    bool ok = true;
    explicit DeviceScope(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceScope()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
    int rank;
    int kind;           // 0 input, 1 output
};

bool overlaps(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

// Status of a call that finds an error recorded by the device.
dt_status take_device_error(dt_group *g)
{
    if (g->poisoned) return DT_ERR_POISONED;
    const int code = static_cast<volatile DevError *>(g->h_err)->code;
    if (code != 0) {
        g->poisoned = true;
        g->poison_code = static_cast<dt_status>(code);
        return static_cast<dt_status>(code);
    }
    return DT_OK;
}

dt_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return DT_OK;
    if (e == cudaErrorMemoryAllocation) return DT_ERR_OOM;
    return DT_ERR_CUDA;
}

dt_status check_rank(dt_group *g, int rank)
{
    (void)g;
    return rank == DT_ALL_RANKS ? DT_OK : DT_ERR_INVALID;   // rank-local calls go elsewhere
}

bool is_pow2(int P) { return P > 0 && (P & (P - 1)) == 0; }

void set_avg(int P, float *scale, int32_t *pow2)
{
    *pow2 = is_pow2(P);
    *scale = *pow2 ? 1.0f / (float)P : 0.0f;   // exact for powers of two
}

dt::BarrierParams barrier_params(dt_group *g, int extra, uint64_t timeout_ns)
{
    dt::BarrierParams b;
    b.win = g->d_win;
    b.rank_gen = g->d_win + (size_t)g->P * g->P;
    b.sink = dt::ErrorSink{g->d_err, g->h_err_dev, timeout_ns};
    b.P = g->P;
    b.extra = extra;
    return b;
}

uint64_t timeout_ns(const dt_group *g) { return (uint64_t)g->timeout_ms * 1000000ull; }

dt::ErrorSink error_sink(dt_group *g) { return dt::ErrorSink{g->d_err, g->h_err_dev, timeout_ns(g)}; }

dt_status issue_barrier(dt_group *g, cudaStream_t s)
{
    const dt::BarrierParams b = barrier_params(g, 0, timeout_ns(g));
    cudaError_t e = dt::launch_barrier(b, s);
    if (e != cudaSuccess) return cuda_status(e);
    g->barriers_issued++;
    return DT_OK;
}

void release_plan_slot(dt_group::PlanSlot &sl)
{
    if (sl.h) cudaFreeHost(sl.h);
    if (sl.d) cudaFree(sl.d);
    sl.h = nullptr;
    sl.d = nullptr;
    sl.bytes = 0;
}

void destroy_all(dt_group *g)
{
    for (dt_group::PlanSlot &sl : g->plans) {
        release_plan_slot(sl);
        if (sl.done) cudaEventDestroy(sl.done);
    }
    for (dt_work *w : g->work_all) {
        if (w->end) cudaEventDestroy(w->end);
        delete w;
    }
    if (g->scope_start) cudaEventDestroy(g->scope_start);
    if (g->comm) cudaStreamDestroy(g->comm);
    for (int r = 0; r < DT_MAX_RANKS; ++r)
        if (g->rv_ready[r]) cudaEventDestroy(g->rv_ready[r]);
    for (int k = 0; k < 2; ++k)
        if (g->rv_done[k]) cudaEventDestroy(g->rv_done[k]);
    if (g->d_win) cudaFree(g->d_win);
    if (g->d_err) cudaFree(g->d_err);
    if (g->h_err) cudaFreeHost(g->h_err);
    delete g;
}

cudaError_t grow_plan_slot(dt_group::PlanSlot &sl, size_t bytes)
{
    if (bytes <= sl.bytes) return cudaSuccess;
    size_t cap = sl.bytes ? sl.bytes : ((size_t)1 << 20);
    while (cap < bytes) cap *= 2;
    release_plan_slot(sl);
    cudaError_t e = cudaHostAlloc(&sl.h, cap, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaMalloc(&sl.d, cap);
    if (e != cudaSuccess) { release_plan_slot(sl); return e; }
    sl.bytes = cap;
    return cudaSuccess;
}

// A new, empty plan slot (its buffers grow on first use).
cudaError_t add_plan_slot(dt_group *g)
{
    g->plans.emplace_back();
    return cudaEventCreateWithFlags(&g->plans.back().done, cudaEventDisableTiming);
}

// Greedy bucket plan shared by dt_bucket_plan and dt_bucket_allreduce.
size_t plan_buckets(const size_t *counts, size_t T, size_t es, size_t cap, size_t *bucket_of)
{
    size_t b = 0, filled = 0;
    for (size_t t = 0; t < T; ++t) {
        const size_t bytes = counts[t] * es;
        if (filled > 0 && filled + bytes > cap) { ++b; filled = 0; }
        bucket_of[t] = b;
        filled += bytes;
    }
    return T ? b + 1 : 0;
}

enum CallKind {
    CK_ALLREDUCE = 1, CK_REDUCE_SCATTER, CK_ALL_GATHER, CK_ALL_TO_ALL, CK_BARRIER,
    CK_REPLICATE_TO_SHARD, CK_ALL_GATHER_INTO_VEC, CK_ALL_TO_ALL_2D
};

bool same_call(const dt_group::RankCall &a, const dt_group::RankCall &b)
{
    // every rank of a round must make the same call; an uneven AllGather's
    // row counts are each rank's own
    const bool own_rows = a.kind == CK_ALL_GATHER || a.kind == CK_ALL_GATHER_INTO_VEC;
    const bool own_op = a.kind == CK_REPLICATE_TO_SHARD;   // op holds the rank's shard index
    return a.kind == b.kind && a.dtype == b.dtype && (own_op || a.op == b.op) &&
           a.flags == b.flags && a.dim2 == b.dim2 && a.row_bytes == b.row_bytes &&
           (own_rows || a.count == b.count);
}

// The last rank of a round launches the group-wide call on its own stream,
// after that stream has waited for every other rank's inputs (their ready
// events: the DestGet / StreamWaitEvent step of the TensorStore protocol).
// Ranks that passed the launching stream itself need no wait, either way.
dt_status launch_round(dt_group *g, int last)
{
    const int P = g->P;
    const dt_group::RankCall &c0 = g->rv_call[0];
    for (int r = 1; r < P; ++r)
        if (!same_call(g->rv_call[r], c0)) return DT_ERR_INVALID;
    cudaStream_t s = g->rv_call[last].stream;
    for (int r = 0; r < P; ++r)
        if (r != last && g->rv_call[r].stream != s &&
            cudaStreamWaitEvent(s, g->rv_ready[r], 0) != cudaSuccess)
            return DT_ERR_CUDA;
    const void *ins[DT_MAX_RANKS];
    void *outs[DT_MAX_RANKS];
    size_t rows[DT_MAX_RANKS];
    for (int r = 0; r < P; ++r) {
        ins[r] = g->rv_call[r].in;
        outs[r] = g->rv_call[r].out;
        rows[r] = g->rv_call[r].count;
    }
    switch (c0.kind) {
    case CK_ALLREDUCE:
        return dt_allreduce(g, DT_ALL_RANKS, ins, outs, c0.count, c0.dtype, c0.op, c0.flags, s);
    case CK_REDUCE_SCATTER:
        return dt_reduce_scatter(g, DT_ALL_RANKS, ins, outs, c0.count, c0.dtype, c0.op, s);
    case CK_ALL_GATHER:
        return dt_all_gather(g, DT_ALL_RANKS, ins, outs, rows, 0, c0.row_bytes, c0.flags, s);
    case CK_ALL_TO_ALL:
        return dt_all_to_all(g, DT_ALL_RANKS, ins, outs, c0.count, s);
    case CK_BARRIER:
        return dt_barrier(g, DT_ALL_RANKS, s);
    case CK_REPLICATE_TO_SHARD: {
        int shard[DT_MAX_RANKS];
        for (int r = 0; r < P; ++r) shard[r] = g->rv_call[r].op;
        return dt_replicate_to_shard(g, DT_ALL_RANKS, ins, outs, shard, c0.count, c0.row_bytes, s);
    }
    case CK_ALL_GATHER_INTO_VEC: {
        void *vec[DT_MAX_RANKS * DT_MAX_RANKS];
        for (int q = 0; q < P; ++q)
            for (int r = 0; r < P; ++r) vec[q * P + r] = g->rv_call[q].outv[r];
        return dt_all_gather_into_vec(g, DT_ALL_RANKS, ins, vec, rows, 0, c0.row_bytes, s);
    }
    case CK_ALL_TO_ALL_2D:
        return dt_all_to_all_2d(g, DT_ALL_RANKS, ins, outs, c0.count, c0.row_bytes,
                                (size_t)c0.dtype, c0.op, c0.dim2, s);
    }
    return DT_ERR_INVALID;
}

void poison(dt_group *g, dt_status code)
{
    std::lock_guard<std::mutex> lock(g->mu);
    if (!g->poisoned) {
        g->poisoned = true;
        g->poison_code = code;
    }
}

// One rank's part of a rank-local call.  The rank records a ready event on its
// stream (SrcSet), then meets the other ranks.  All but the last wait, at most
// the group's time limit, for the round to complete and then make their
// stream wait on the round's done event; the last launches for everyone.  A
// wait that runs out abandons the round: every rank of it returns
// DT_ERR_TIMEOUT and the group is poisoned until dt_group_reset.
constexpr std::chrono::microseconds kRendezvousSpin(200);

dt_status rank_local(dt_group *g, int rank, const dt_group::RankCall &call)
{
    if (rank < 0 || rank >= g->P) return DT_ERR_INVALID;
    {
        std::lock_guard<std::mutex> lock(g->mu);
        dt_status st = take_device_error(g);
        if (st != DT_OK) return st;
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    if (cudaEventRecord(g->rv_ready[rank], call.stream) != cudaSuccess) return DT_ERR_CUDA;

    std::unique_lock<std::mutex> lk(g->rv_mu);
    if (g->rv_aborted) return DT_ERR_POISONED;
    if (g->rv_present[rank]) return DT_ERR_INVALID;   // this rank is already in the round
    g->rv_call[rank] = call;
    g->rv_present[rank] = true;
    const uint64_t my_round = g->rv_round;
    const int slot = (int)(my_round & 1);

    if (++g->rv_arrived < g->P) {
        const auto start = std::chrono::steady_clock::now();
        const auto deadline = start + std::chrono::milliseconds(g->timeout_ms);
        // The other ranks' calls usually arrive within microseconds; a sleep
        // on the condition variable would add a futex wake-up per rank per
        // call, more than the launch itself.  So spin first, without the lock
        // and yielding the core, for up to kRendezvousSpin; then sleep.
        const uint64_t epoch = g->rv_epoch.load(std::memory_order_relaxed);
        lk.unlock();
        const auto spin_end = start + kRendezvousSpin;
        for (unsigned it = 1; g->rv_epoch.load(std::memory_order_acquire) == epoch; ++it) {
            if ((it & 15) == 0) {
                if (std::chrono::steady_clock::now() >= spin_end) break;
                std::this_thread::yield();
            }
        }
        lk.lock();
        g->rv_cv.wait_until(lk, deadline, [&] { return g->rv_round != my_round || g->rv_aborted; });
        if (g->rv_round != my_round) {
            dt_status st = g->rv_status[slot];
            cudaEvent_t done = g->rv_done[slot];
            const bool same_stream = g->rv_launch[slot] == call.stream;
            lk.unlock();
            if (st == DT_OK && !same_stream && cudaStreamWaitEvent(call.stream, done, 0) != cudaSuccess)
                st = DT_ERR_CUDA;
            return st;
        }
        g->rv_aborted = true;
        g->rv_epoch.fetch_add(1, std::memory_order_release);
        g->rv_present[rank] = false;
        --g->rv_arrived;
        lk.unlock();
        g->rv_cv.notify_all();
        poison(g, DT_ERR_TIMEOUT);
        return DT_ERR_TIMEOUT;
    }

    dt_status st = launch_round(g, rank);
    if (st == DT_OK && cudaEventRecord(g->rv_done[slot], call.stream) != cudaSuccess) st = DT_ERR_CUDA;
    g->rv_status[slot] = st;
    g->rv_launch[slot] = call.stream;
    for (int r = 0; r < DT_MAX_RANKS; ++r) g->rv_present[r] = false;
    g->rv_arrived = 0;
    ++g->rv_round;
    g->rv_epoch.fetch_add(1, std::memory_order_release);
    lk.unlock();
    g->rv_cv.notify_all();
    return st;
}

dt_group::RankCall make_call(int kind, const void *const *in, void *const *out, size_t count,
                             size_t row_bytes, int dtype, int op, unsigned flags, void *stream)
{
    dt_group::RankCall c;
    c.kind = kind;
    c.in = in ? in[0] : nullptr;
    c.out = out ? out[0] : nullptr;
    c.outv = out;
    c.dim2 = 0;
    c.count = count;
    c.row_bytes = row_bytes;
    c.dtype = dtype;
    c.op = op;
    c.flags = flags;
    c.stream = static_cast<cudaStream_t>(stream);
    return c;
}

}  // namespace

extern "C" {

const char *dt_status_string(dt_status st)
{
    switch (st) {
    case DT_OK: return "ok";
    case DT_ERR_INVALID: return "invalid argument";
    case DT_ERR_UNSUPPORTED: return "unsupported";
    case DT_ERR_CUDA: return "CUDA error";
    case DT_ERR_TIMEOUT: return "device wait timed out";
    case DT_ERR_OOM: return "out of memory";
    case DT_ERR_POISONED: return "group poisoned by an earlier device error; reset it";
    case DT_ERR_TOO_LARGE: return "request exceeds the fixed scratch of the allocation-free entry point";
    case DT_NOT_READY: return "work not finished yet";
    }
    return "unknown status";
}

uint64_t dt_launch_count(void) { return dt::g_launches.load(std::memory_order_relaxed); }

dt_status dt_group_create(int world_size, int cuda_device, dt_group_t *out)
{
    DT_TRACE();
    if (!out) return DT_ERR_INVALID;
    *out = nullptr;
    if (world_size < 1 || world_size > DT_MAX_RANKS || cuda_device < 0) return DT_ERR_INVALID;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return DT_ERR_CUDA;
    if (cuda_device >= ndev) return DT_ERR_INVALID;
    DeviceScope scope(cuda_device);
    if (!scope.ok) return DT_ERR_CUDA;

    dt_group *g = new (std::nothrow) dt_group;
    if (!g) return DT_ERR_OOM;
    g->P = world_size;
    g->device = cuda_device;
    if (const char *env = std::getenv("DT_TIMEOUT_MS")) {
        const long v = std::strtol(env, nullptr, 10);
        if (v >= 1 && v <= 3600000) g->timeout_ms = (uint32_t)v;
    }
    const size_t win_bytes = dt::win_words(world_size) * sizeof(int32_t);
    cudaError_t e = cudaMalloc(&g->d_win, win_bytes);
    if (e == cudaSuccess) e = cudaMemset(g->d_win, 0, win_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&g->d_err, sizeof(DevError));
    if (e == cudaSuccess) e = cudaMemset(g->d_err, 0, sizeof(DevError));
    if (e == cudaSuccess) e = cudaHostAlloc(&g->h_err, sizeof(DevError), cudaHostAllocMapped);
    if (e == cudaSuccess) {
        memset(g->h_err, 0, sizeof(DevError));
        e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&g->h_err_dev), g->h_err, 0);
    }
    for (int k = 0; k < dt_group::kPlanSlots && e == cudaSuccess; ++k) {
        e = add_plan_slot(g);
        if (e == cudaSuccess) e = grow_plan_slot(g->plans.back(), (size_t)1 << 20);
    }
    for (int r = 0; r < world_size && e == cudaSuccess; ++r)
        e = cudaEventCreateWithFlags(&g->rv_ready[r], cudaEventDisableTiming);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k)
        e = cudaEventCreateWithFlags(&g->rv_done[k], cudaEventDisableTiming);
    // the async scopes' stream runs at the device's highest priority, so its
    // blocks take SMs ahead of queued compute blocks as they free up
    int prio_least = 0, prio_greatest = 0;
    if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&g->comm, cudaStreamNonBlocking, prio_greatest);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->scope_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        destroy_all(g);
        return cuda_status(e);
    }
    *out = g;
    return DT_OK;
}

dt_status dt_group_destroy(dt_group_t g)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    DeviceScope scope(g->device);
    for (dt_group::PlanSlot &sl : g->plans)
        if (sl.used) cudaEventSynchronize(sl.done);
    cudaDeviceSynchronize();
    destroy_all(g);
    return DT_OK;
}

dt_status dt_group_reset(dt_group_t g, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t win_bytes = dt::win_words(g->P) * sizeof(int32_t);
    cudaError_t e = cudaMemsetAsync(g->d_win, 0, win_bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(g->d_err, 0, sizeof(DevError), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    memset(g->h_err, 0, sizeof(DevError));
    g->poisoned = false;
    g->poison_code = DT_OK;
    g->barriers_issued = 0;
    {
        std::lock_guard<std::mutex> rv(g->rv_mu);
        for (int r = 0; r < DT_MAX_RANKS; ++r) g->rv_present[r] = false;
        g->rv_arrived = 0;
        g->rv_aborted = false;
        ++g->rv_round;
        g->rv_epoch.fetch_add(1, std::memory_order_release);
    }
    g->rv_cv.notify_all();
    return DT_OK;
}

dt_status dt_group_check(dt_group_t g)
{
    if (!g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    const dt_status st = take_device_error(g);
    return g->poisoned ? g->poison_code : st;
}

dt_status dt_group_error_detail(dt_group_t g, int *rank, int *peer, int *generation)
{
    if (!g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    volatile DevError *h = g->h_err;
    if (rank) *rank = h->rank;
    if (peer) *peer = h->peer;
    if (generation) *generation = h->gen;
    return static_cast<dt_status>(h->code);
}

int dt_group_size(dt_group_t g) { return g ? g->P : 0; }

int64_t dt_group_generation(dt_group_t g) { return g ? g->barriers_issued : -1; }

dt_status dt_group_set_timeout_ms(dt_group_t g, uint32_t timeout_ms)
{
    if (!g || timeout_ms < 1) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    g->timeout_ms = timeout_ms;
    return DT_OK;
}

dt_status dt_bucket_plan(const size_t *counts, size_t n_tensors, size_t elem_bytes_,
                         size_t cap_bytes, size_t *bucket_of, size_t *n_buckets)
{
    if (!n_buckets || (n_tensors && (!counts || !bucket_of)) || elem_bytes_ == 0 || cap_bytes == 0)
        return DT_ERR_INVALID;
    for (size_t t = 0; t < n_tensors; ++t)
        if (counts[t] > SIZE_MAX / elem_bytes_) return DT_ERR_INVALID;
    *n_buckets = plan_buckets(counts, n_tensors, elem_bytes_, cap_bytes, bucket_of);
    return DT_OK;
}

dt_status dt_allreduce(dt_group_t g, int rank, const void *const *in, void *const *out,
                       size_t count, int dtype, int op, unsigned flags, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out) return DT_ERR_INVALID;
        return rank_local(g, rank, make_call(CK_ALLREDUCE, in, out, count, 0, dtype, op, flags, stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if ((st = check_rank(g, rank)) != DT_OK) return st;
    if (!in || !out || !valid_dtype(dtype) || !valid_op(op) || (flags & ~DT_SHARED_OUTPUT))
        return DT_ERR_INVALID;
    if (dtype == DT_I32 && op == DT_AVG) return DT_ERR_UNSUPPORTED;
    if (count > SIZE_MAX / 16) return DT_ERR_INVALID;
    const int P = g->P;
    const bool shared = flags & DT_SHARED_OUTPUT;
    const size_t bytes = count * elem_bytes(dtype);
    for (int r = 0; r < P; ++r)
        if (!in[r] || !out[r]) return DT_ERR_INVALID;
    if (shared)
        for (int r = 1; r < P; ++r)
            if (out[r] != out[0]) return DT_ERR_INVALID;
    if (count == 0) return DT_OK;

    // Outputs may alias only their own rank's input exactly (in place), never
    // another buffer; a shared output aliases nothing.
    const int nout = shared ? 1 : P;
    for (int q = 0; q < nout; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + bytes, q, 1};
        for (int r = 0; r < P; ++r) {
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + bytes, r, 0};
            if (overlaps(o, i) && (shared || r != q || in[r] != out[q])) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < nout; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + bytes, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }

    dt::ReduceParams p;
    memset(&p, 0, sizeof p);
    // The vector kernel runs when every buffer lies the same whole number of
    // elements past a 16-byte boundary (aligned buffers, or views that share
    // an offset): it gets the buffers from that boundary on, and reduces the
    // head elements before it on the element path.
    const size_t es = elem_bytes(dtype);
    const uintptr_t mis = (uintptr_t)in[0] & 15;
    const size_t head = ((16 - mis) & 15) / es;
    bool vec = mis % es == 0 && head < count;
    for (int r = 0; r < P; ++r) vec = vec && ((uintptr_t)in[r] & 15) == mis;
    for (int q = 0; q < nout; ++q) vec = vec && ((uintptr_t)out[q] & 15) == mis;
    const size_t skip = vec ? head * es : 0;
    for (int r = 0; r < P; ++r) p.in[r] = static_cast<const unsigned char *>(in[r]) + skip;
    for (int q = 0; q < nout; ++q) p.out[q] = static_cast<unsigned char *>(out[q]) + skip;
    p.head = vec ? (uint32_t)head : 0;
    p.n = count - p.head;
    p.job_stride = 0;
    dt::set_reduce_bounds(p, in, bytes, out, bytes, P, nout, error_sink(g));
    p.P = P;
    p.out_per_job = nout;
    set_avg(P, &p.avg_scale, &p.avg_pow2);

    // Other element-aligned layouts whose outputs share an offset: the
    // shifting kernel reads the inputs as aligned vectors and shifts them.
    bool shift = !vec;
    for (int r = 0; r < P && shift; ++r) shift = ((uintptr_t)in[r] % es) == 0;
    for (int q = 0; q < nout && shift; ++q)
        shift = ((uintptr_t)out[q] & 15) == ((uintptr_t)out[0] & 15) && ((uintptr_t)out[q] % es) == 0;

    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    if (shift)
        return cuda_status(dt::launch_reduce_shift(p, dtype, op, 1, g->device,
                                                   static_cast<cudaStream_t>(stream)));
    return cuda_status(dt::launch_reduce(p, dtype, op, 1, vec, g->device,
                                         static_cast<cudaStream_t>(stream)));
}

dt_status dt_reduce_scatter(dt_group_t g, int rank, const void *const *in, void *const *out,
                            size_t recv_count, int dtype, int op, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out) return DT_ERR_INVALID;
        return rank_local(g, rank, make_call(CK_REDUCE_SCATTER, in, out, recv_count, 0, dtype, op, 0,
                                             stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if ((st = check_rank(g, rank)) != DT_OK) return st;
    if (!in || !out || !valid_dtype(dtype) || !valid_op(op)) return DT_ERR_INVALID;
    if (dtype == DT_I32 && op == DT_AVG) return DT_ERR_UNSUPPORTED;
    const int P = g->P;
    if (recv_count > SIZE_MAX / 16 / (size_t)P) return DT_ERR_INVALID;
    for (int r = 0; r < P; ++r)
        if (!in[r] || !out[r]) return DT_ERR_INVALID;
    if (recv_count == 0) return DT_OK;
    const size_t es = elem_bytes(dtype);
    const size_t in_bytes = recv_count * P * es, out_bytes = recv_count * es;
    for (int q = 0; q < P; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + out_bytes, q, 1};
        for (int r = 0; r < P; ++r) {
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + in_bytes, r, 0};
            if (overlaps(o, i)) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < P; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + out_bytes, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }

    dt::ReduceParams p;
    memset(&p, 0, sizeof p);
    // Job (shard) j reads every input at element j * recv_count and writes
    // out[j].  The vector kernel runs when shards are whole 16-byte vectors
    // and every input and output lies the same whole number of elements past
    // a 16-byte boundary: it gets the buffers from that boundary on, and
    // reduces each shard's head elements before it on the element path.
    const uintptr_t mis = (uintptr_t)in[0] & 15;
    const size_t head = ((16 - mis) & 15) / es;
    bool vec = (recv_count * es) % 16 == 0 && mis % es == 0 && head < recv_count;
    for (int r = 0; r < P; ++r)
        vec = vec && ((uintptr_t)in[r] & 15) == mis && ((uintptr_t)out[r] & 15) == mis;
    const size_t skip = vec ? head * es : 0;
    for (int r = 0; r < P; ++r) {
        p.in[r] = static_cast<const unsigned char *>(in[r]) + skip;
        p.out[r] = static_cast<unsigned char *>(out[r]) + skip;
    }
    p.head = vec ? (uint32_t)head : 0;
    p.n = recv_count - p.head;
    p.job_stride = recv_count;
    dt::set_reduce_bounds(p, in, in_bytes, out, out_bytes, P, P, error_sink(g));
    p.P = P;
    p.out_per_job = 1;
    set_avg(P, &p.avg_scale, &p.avg_pow2);

    bool shift = !vec;
    for (int r = 0; r < P && shift; ++r)
        shift = ((uintptr_t)in[r] % es) == 0 && ((uintptr_t)out[r] % es) == 0;

    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    if (shift)
        return cuda_status(dt::launch_reduce_shift(p, dtype, op, P, g->device,
                                                   static_cast<cudaStream_t>(stream)));
    return cuda_status(dt::launch_reduce(p, dtype, op, P, vec, g->device,
                                         static_cast<cudaStream_t>(stream)));
}

dt_status dt_all_gather(dt_group_t g, int rank, const void *const *in, void *const *out,
                        const size_t *rows, size_t rows_equal, size_t row_bytes, unsigned flags,
                        void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        // a rank passes its own shard: rows must be NULL, rows_equal its row count
        if (!in || !out || rows) return DT_ERR_INVALID;
        return rank_local(g, rank, make_call(CK_ALL_GATHER, in, out, rows_equal, row_bytes, 0, 0,
                                             flags, stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if ((st = check_rank(g, rank)) != DT_OK) return st;
    if (!in || !out || (flags & ~DT_SHARED_OUTPUT)) return DT_ERR_INVALID;
    const int P = g->P;
    const bool shared = flags & DT_SHARED_OUTPUT;
    size_t nrows[DT_MAX_RANKS], off[DT_MAX_RANKS], total = 0;
    for (int r = 0; r < P; ++r) {
        nrows[r] = rows ? rows[r] : rows_equal;
        if (row_bytes && nrows[r] > SIZE_MAX / 4 / row_bytes) return DT_ERR_INVALID;
        off[r] = total;
        total += nrows[r];
        if (total > SIZE_MAX / 4 / (row_bytes ? row_bytes : 1)) return DT_ERR_INVALID;
    }
    for (int r = 0; r < P; ++r)
        if (!out[r] || (nrows[r] && !in[r])) return DT_ERR_INVALID;
    if (shared)
        for (int r = 1; r < P; ++r)
            if (out[r] != out[0]) return DT_ERR_INVALID;
    const size_t out_bytes = total * row_bytes;
    if (out_bytes == 0) return DT_OK;
    const int nout = shared ? 1 : P;
    for (int q = 0; q < nout; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + out_bytes, q, 1};
        for (int r = 0; r < P; ++r) {
            if (!nrows[r]) continue;
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + nrows[r] * row_bytes, r, 0};
            if (overlaps(o, i)) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < nout; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + out_bytes, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }

    dt::CopySeg segs[DT_MAX_RANKS] = {};
    bool vec = true;
    for (int r = 0; r < P; ++r) {
        segs[r].src = static_cast<const unsigned char *>(in[r]);
        segs[r].bytes = nrows[r] * row_bytes;
        segs[r].dst_off = off[r] * row_bytes;
        segs[r].tile_begin = 0;
        segs[r].dst_first = 0;
        segs[r].dst_count = (int16_t)nout;
        dt::set_src_bounds(segs[r], in[r], segs[r].bytes);
        if (segs[r].bytes)
            vec = vec && aligned16(in[r]) && segs[r].bytes % 16 == 0 && segs[r].dst_off % 16 == 0;
    }
    void *outs[DT_MAX_RANKS] = {};
    uint64_t ob[DT_MAX_RANKS] = {};
    for (int q = 0; q < nout; ++q) {
        outs[q] = out[q];
        ob[q] = out_bytes;
        vec = vec && aligned16(out[q]);
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(dt::launch_copy(segs, P, outs, ob, nout, vec, error_sink(g), g->device,
                                       static_cast<cudaStream_t>(stream)));
}

dt_status dt_all_to_all(dt_group_t g, int rank, const void *const *in, void *const *out,
                        size_t chunk_bytes, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out) return DT_ERR_INVALID;
        return rank_local(g, rank, make_call(CK_ALL_TO_ALL, in, out, chunk_bytes, 0, 0, 0, 0, stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if ((st = check_rank(g, rank)) != DT_OK) return st;
    if (!in || !out) return DT_ERR_INVALID;
    const int P = g->P;
    if (chunk_bytes > SIZE_MAX / 4 / (size_t)P) return DT_ERR_INVALID;
    for (int r = 0; r < P; ++r)
        if (!in[r] || !out[r]) return DT_ERR_INVALID;
    if (chunk_bytes == 0) return DT_OK;
    const size_t bytes = chunk_bytes * P;
    for (int q = 0; q < P; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + bytes, q, 1};
        for (int r = 0; r < P; ++r) {
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + bytes, r, 0};
            if (overlaps(o, i)) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < P; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + bytes, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }

    // segment (i, j): chunk j of rank i -> rank j at offset i * chunk_bytes;
    // ordered by source rank so that each block streams one input in order
    std::vector<dt::CopySeg> segs((size_t)P * P);
    bool vec = chunk_bytes % 16 == 0;
    for (int i = 0; i < P; ++i) {
        vec = vec && aligned16(in[i]) && aligned16(out[i]);
        for (int j = 0; j < P; ++j) {
            dt::CopySeg &sg = segs[(size_t)i * P + j];
            sg.src = static_cast<const unsigned char *>(in[i]) + (size_t)j * chunk_bytes;
            sg.bytes = chunk_bytes;
            sg.dst_off = (size_t)i * chunk_bytes;
            sg.tile_begin = 0;
            sg.dst_first = (int16_t)j;
            sg.dst_count = 1;
            dt::set_src_bounds(sg, in[i], bytes);
        }
    }
    void *outs[DT_MAX_RANKS] = {};
    uint64_t ob[DT_MAX_RANKS] = {};
    for (int q = 0; q < P; ++q) {
        outs[q] = out[q];
        ob[q] = bytes;
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(dt::launch_copy(segs.data(), P * P, outs, ob, P, vec, error_sink(g), g->device,
                                       static_cast<cudaStream_t>(stream)));
}

dt_status dt_bucket_allreduce(dt_group_t g, void *const *grads, const size_t *counts,
                              size_t n_tensors, int dtype, int op, size_t bucket_cap_bytes,
                              void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (dtype != DT_BF16 && dtype != DT_F32) return valid_dtype(dtype) ? DT_ERR_UNSUPPORTED : DT_ERR_INVALID;
    if (op != DT_SUM && op != DT_AVG) return valid_op(op) ? DT_ERR_UNSUPPORTED : DT_ERR_INVALID;
    if (n_tensors && (!grads || !counts)) return DT_ERR_INVALID;
    if (n_tensors > (1u << 30)) return DT_ERR_INVALID;
    const int P = g->P;
    const size_t es = elem_bytes(dtype);
    const size_t cap = bucket_cap_bytes ? bucket_cap_bytes : DT_DEFAULT_BUCKET_CAP_BYTES;

    // the call's arguments, as the key of a cached plan
    std::vector<uint64_t> key;
    key.reserve(4 + n_tensors * (P + 1));
    key.push_back((uint64_t)dtype);
    key.push_back((uint64_t)op);
    key.push_back((uint64_t)cap);
    key.push_back((uint64_t)n_tensors);
    for (size_t t = 0; t < n_tensors; ++t) key.push_back((uint64_t)counts[t]);
    for (size_t i = 0; i < n_tensors * P; ++i) key.push_back((uint64_t)(uintptr_t)grads[i]);

    int k = -1;
    for (size_t j = 0; j < g->plans.size(); ++j)
        if (g->plans[j].used && g->plans[j].key == key) k = (int)j;

    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) return DT_ERR_CUDA;
    const bool capturing = capture != cudaStreamCaptureStatusNone;

    if (k < 0 && capturing) {
        // building a plan may allocate, which a capture forbids: the call must
        // follow an eager call with the same arguments
        return DT_ERR_UNSUPPORTED;
    }
    if (k < 0) {
        // validate and find overlapping gradient buffers (sorted sweep)
        std::vector<Range> ranges;
        ranges.reserve(n_tensors * P);
        for (size_t t = 0; t < n_tensors; ++t) {
            if (counts[t] > SIZE_MAX / 16) return DT_ERR_INVALID;
            if (counts[t] == 0) continue;
            for (int p = 0; p < P; ++p) {
                const void *ptr = grads[t * P + p];
                if (!ptr) return DT_ERR_INVALID;
                ranges.push_back({(uintptr_t)ptr, (uintptr_t)ptr + counts[t] * es, p, 1});
            }
        }
        if (ranges.empty()) return DT_OK;
        std::sort(ranges.begin(), ranges.end(), [](const Range &a, const Range &b) { return a.lo < b.lo; });
        for (size_t i = 1; i < ranges.size(); ++i)
            if (ranges[i].lo < ranges[i - 1].hi) return DT_ERR_INVALID;

        std::vector<size_t> bucket_of(n_tensors);
        const size_t nb = plan_buckets(counts, n_tensors, es, cap, bucket_of.data());

        // per bucket: its tensors [tb, te), padded size, grid and slice length
        std::vector<dt_group::PlanLaunch> bl(nb);
        size_t n_starts = 0;
        for (size_t b = 0, t = 0; b < nb; ++b) {
            dt_group::PlanLaunch &L = bl[b];
            L.tb = t;
            L.total = 0;
            while (t < n_tensors && bucket_of[t] == b) L.total += dt::bucket_padded(counts[t++], dtype);
            L.te = t;
            L.blocks = 0;
            L.per_block = 1;
            if (L.total) {
                e = dt::bucket_grid(dtype, op, P, L.total, g->device, &L.blocks, &L.per_block);
                if (e != cudaSuccess) return cuda_status(e);
                // one block per slice of a tensor: the grid's slice length, cut at tensor ends
                uint64_t nblk = 0;
                for (size_t u = L.tb; u < L.te; ++u) nblk += dt::bucket_tensor_blocks(counts[u], dtype, L.per_block);
                if (nblk > UINT32_MAX / 2) return DT_ERR_INVALID;
                L.blocks = (uint32_t)nblk;
            }
            L.start_off = n_starts;
            n_starts += L.blocks;
        }

        // plan layout: [T * P pointers][T tensor entries][block starts]
        const size_t ptr_bytes = n_tensors * P * sizeof(void *);
        const size_t tab_bytes = n_tensors * sizeof(dt::BucketTensor);
        const size_t plan_bytes = ptr_bytes + tab_bytes + n_starts * sizeof(uint32_t);
        // the next unpinned slot, round robin; a new one when all are pinned
        const int nslots = (int)g->plans.size();
        for (int i = 0; i < nslots && k < 0; ++i) {
            const int j = (g->next_plan + i) % nslots;
            if (!g->plans[j].pinned) k = j;
        }
        if (k < 0) {
            e = add_plan_slot(g);
            if (e != cudaSuccess) return cuda_status(e);
            k = (int)g->plans.size() - 1;
        }
        g->next_plan = (k + 1) % (int)g->plans.size();
        dt_group::PlanSlot &sl = g->plans[k];
        if (sl.used) e = cudaEventSynchronize(sl.done);
        sl.key.clear();   // the slot no longer holds a valid plan
        if (e == cudaSuccess) e = grow_plan_slot(sl, plan_bytes);
        if (e != cudaSuccess) return cuda_status(e);

        unsigned char *h = static_cast<unsigned char *>(sl.h);
        memcpy(h, grads, ptr_bytes);
        dt::BucketTensor *tab = reinterpret_cast<dt::BucketTensor *>(h + ptr_bytes);
        uint32_t *starts = reinterpret_cast<uint32_t *>(h + ptr_bytes + tab_bytes);
        for (const dt_group::PlanLaunch &L : bl) {
            uint64_t first = 0;
            uint32_t block = 0;   // the bucket's blocks, tensor by tensor
            for (size_t t = L.tb; t < L.te; ++t) {
                bool al = true;
                for (int p = 0; p < P; ++p) al = al && aligned16(grads[t * P + p]);
                tab[t].first = first;
                tab[t].count = counts[t];
                tab[t].slot = (uint32_t)t | (al ? 0x80000000u : 0u);
                tab[t].block0 = block;
                first += dt::bucket_padded(counts[t], dtype);
                const uint64_t nb_t = L.total ? dt::bucket_tensor_blocks(counts[t], dtype, L.per_block) : 0;
                for (uint64_t j = 0; j < nb_t; ++j) starts[L.start_off + block++] = (uint32_t)(t - L.tb);
            }
        }
        e = cudaMemcpyAsync(sl.d, h, plan_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_status(e);
        if (dt::log_enabled()) {
            std::string blocks;
            for (const dt_group::PlanLaunch &L : bl) blocks += (blocks.empty() ? "" : ",") + std::to_string(L.blocks);
            std::fprintf(stderr, "dt: bucket plan in slot %d: %zu tensors x %d ranks, %zu buckets, blocks [%s]\n",
                         k, n_tensors, P, bl.size(), blocks.c_str());
        }
        sl.key = std::move(key);
        sl.launches = std::move(bl);
        sl.ptr_bytes = ptr_bytes;
        sl.tab_bytes = tab_bytes;
    } else if (dt::log_enabled()) {
        std::fprintf(stderr, "dt: bucket plan in slot %d reused%s\n", k,
                     capturing ? " under stream capture (slot pinned)" : "");
    }

    dt_group::PlanSlot &sl = g->plans[k];
    if (capturing) sl.pinned = true;   // a graph now holds this plan's address
    const unsigned char *d = static_cast<const unsigned char *>(sl.d);
    const size_t ptr_bytes = sl.ptr_bytes, tab_bytes = sl.tab_bytes;
    const std::vector<dt_group::PlanLaunch> &bl = sl.launches;
    dt::BucketParams bp;
    memset(&bp, 0, sizeof bp);
    bp.ptrs = reinterpret_cast<void *const *>(d);
    bp.P = P;
    set_avg(P, &bp.avg_scale, &bp.avg_pow2);
    bp.sink = error_sink(g);
    // The barrier between buckets b and b + 1 runs in an extra last block of
    // bucket b's kernel (the buckets' data decides nothing about it, so an
    // empty bucket still gets its barrier from a kernel of its own).
    bool kernel_before = false;   // a bucket kernel of this call is already queued
    for (size_t b = 0; b < bl.size(); ++b) {
        const dt_group::PlanLaunch &L = bl[b];
        bp.tensors = reinterpret_cast<const dt::BucketTensor *>(d + ptr_bytes) + L.tb;
        bp.block_start = reinterpret_cast<const uint32_t *>(d + ptr_bytes + tab_bytes) + L.start_off;
        bp.ntensors = (uint32_t)(L.te - L.tb);
        bp.total = L.total;
        bp.per_block = L.per_block;
        bp.blocks = L.blocks;
        const bool barrier_after = b + 1 < bl.size();
        bp.win = barrier_after ? g->d_win : nullptr;
        bp.early = kernel_before ? 1u : 0u;
        bool launched = false;
        e = dt::launch_bucket(bp, dtype, op, g->device, s, &launched);
        if (e != cudaSuccess) break;
        kernel_before = kernel_before || launched;
        if (barrier_after) {
            if (launched) {
                g->barriers_issued++;
            } else {
                st = issue_barrier(g, s);
                if (st != DT_OK) return st;
            }
        }
    }
    cudaError_t e2 = capturing ? cudaSuccess : cudaEventRecord(sl.done, s);
    sl.used = true;
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(e2);
}

dt_status dt_replicate_to_shard(dt_group_t g, int rank, const void *const *in, void *const *out,
                                const int *shard_idx, size_t rows, size_t row_bytes, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out) return DT_ERR_INVALID;
        const int own = shard_idx ? shard_idx[0] : rank;
        return rank_local(g, rank, make_call(CK_REPLICATE_TO_SHARD, in, out, rows, row_bytes, 0, own,
                                             0, stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (!in || !out) return DT_ERR_INVALID;
    const int P = g->P;
    if (rows % (size_t)P || (row_bytes && rows > SIZE_MAX / 4 / row_bytes)) return DT_ERR_INVALID;
    const size_t block = rows / P * row_bytes, whole = rows * row_bytes;
    int sidx[DT_MAX_RANKS];
    for (int r = 0; r < P; ++r) {
        sidx[r] = shard_idx ? shard_idx[r] : r;
        if (sidx[r] < 0 || sidx[r] >= P) return DT_ERR_INVALID;
        if (block && (!in[r] || !out[r])) return DT_ERR_INVALID;
    }
    if (block == 0) return DT_OK;
    for (int q = 0; q < P; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + block, q, 1};
        for (int r = 0; r < P; ++r) {
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + whole, r, 0};
            if (overlaps(o, i)) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < P; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + block, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }
    dt::CopySeg segs[DT_MAX_RANKS] = {};
    void *outs[DT_MAX_RANKS] = {};
    uint64_t ob[DT_MAX_RANKS] = {};
    bool vec = block % 16 == 0;
    for (int r = 0; r < P; ++r) {
        segs[r].src = static_cast<const unsigned char *>(in[r]) + (size_t)sidx[r] * block;
        segs[r].bytes = block;
        segs[r].dst_off = 0;
        segs[r].tile_begin = 0;
        segs[r].dst_first = (int16_t)r;
        segs[r].dst_count = 1;
        dt::set_src_bounds(segs[r], in[r], whole);
        outs[r] = out[r];
        ob[r] = block;
        vec = vec && aligned16(in[r]) && aligned16(out[r]);
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(dt::launch_copy(segs, P, outs, ob, P, vec, error_sink(g), g->device,
                                       static_cast<cudaStream_t>(stream)));
}

dt_status dt_all_gather_into_vec(dt_group_t g, int rank, const void *const *in, void *const *out,
                                 const size_t *rows, size_t rows_equal, size_t row_bytes,
                                 void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out || rows) return DT_ERR_INVALID;
        return rank_local(g, rank, make_call(CK_ALL_GATHER_INTO_VEC, in, out, rows_equal, row_bytes, 0,
                                             0, 0, stream));
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (!in || !out) return DT_ERR_INVALID;
    const int P = g->P;
    size_t nb[DT_MAX_RANKS];
    for (int r = 0; r < P; ++r) {
        const size_t n = rows ? rows[r] : rows_equal;
        if (row_bytes && n > SIZE_MAX / 4 / row_bytes) return DT_ERR_INVALID;
        nb[r] = n * row_bytes;
        if (nb[r] && !in[r]) return DT_ERR_INVALID;
        for (int q = 0; q < P; ++q)
            if (nb[r] && !out[q * P + r]) return DT_ERR_INVALID;
    }
    // no destination may overlap a source or another destination
    std::vector<Range> ranges;
    for (int r = 0; r < P; ++r) {
        if (!nb[r]) continue;
        ranges.push_back({(uintptr_t)in[r], (uintptr_t)in[r] + nb[r], r, 0});
        for (int q = 0; q < P; ++q)
            ranges.push_back({(uintptr_t)out[q * P + r], (uintptr_t)out[q * P + r] + nb[r], q, 1});
    }
    if (ranges.empty()) return DT_OK;
    // sweep in start order: an output may not start before the end of any
    // earlier range, an input not before the end of any earlier output
    // (inputs may overlap each other: they are only read)
    std::sort(ranges.begin(), ranges.end(), [](const Range &a, const Range &b) { return a.lo < b.lo; });
    uintptr_t end_any = 0, end_out = 0;
    for (const Range &r : ranges) {
        if (r.kind == 1 ? r.lo < end_any : r.lo < end_out) return DT_ERR_INVALID;
        end_any = std::max(end_any, r.hi);
        if (r.kind == 1) end_out = std::max(end_out, r.hi);
    }

    // segment r: rank r's shard to out[q * P + r] for every q; the table is
    // stored by source (outs[r * P + q]) so a segment's destinations are adjacent
    dt::CopySeg segs[DT_MAX_RANKS] = {};
    std::vector<void *> outs((size_t)P * P);
    std::vector<uint64_t> ob((size_t)P * P);
    bool vec = true;
    for (int r = 0; r < P; ++r) {
        segs[r].src = static_cast<const unsigned char *>(in[r]);
        segs[r].bytes = nb[r];
        segs[r].dst_off = 0;
        segs[r].tile_begin = 0;
        segs[r].dst_first = (int16_t)(r * P);
        segs[r].dst_count = (int16_t)P;
        dt::set_src_bounds(segs[r], in[r], nb[r]);
        if (nb[r]) vec = vec && aligned16(in[r]) && nb[r] % 16 == 0;
        for (int q = 0; q < P; ++q) {
            outs[(size_t)r * P + q] = out[q * P + r];
            ob[(size_t)r * P + q] = nb[r];
            if (nb[r]) vec = vec && aligned16(out[q * P + r]);
        }
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(dt::launch_copy(segs, P, outs.data(), ob.data(), P * P, vec, error_sink(g),
                                       g->device, static_cast<cudaStream_t>(stream)));
}

dt_status dt_all_to_all_2d(dt_group_t g, int rank, const void *const *in, void *const *out,
                           size_t R, size_t C, size_t elem_bytes, int src_dim, int dest_dim,
                           void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS) {
        if (!in || !out) return DT_ERR_INVALID;
        dt_group::RankCall c = make_call(CK_ALL_TO_ALL_2D, in, out, R, C, (int)elem_bytes, src_dim, 0,
                                         stream);
        c.dim2 = dest_dim;
        return rank_local(g, rank, c);
    }
    if ((src_dim != 0 && src_dim != 1) || (dest_dim != 0 && dest_dim != 1) || elem_bytes == 0 ||
        elem_bytes > 16)
        return DT_ERR_INVALID;
    if (src_dim == 0 && dest_dim == 0) {
        if (R % (size_t)g->P) return DT_ERR_INVALID;
        return dt_all_to_all(g, DT_ALL_RANKS, in, out, R / g->P * C * elem_bytes, stream);
    }
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (!in || !out) return DT_ERR_INVALID;
    const int P = g->P;
    if ((dest_dim == 0 && R % (size_t)P) || (dest_dim == 1 && C % (size_t)P)) return DT_ERR_INVALID;
    if (C && R > SIZE_MAX / 4 / C / elem_bytes) return DT_ERR_INVALID;
    const size_t es = elem_bytes, bytes = R * C * es;
    for (int r = 0; r < P; ++r)
        if (bytes && (!in[r] || !out[r])) return DT_ERR_INVALID;
    if (bytes == 0) return DT_OK;
    for (int q = 0; q < P; ++q) {
        const Range o{(uintptr_t)out[q], (uintptr_t)out[q] + bytes, q, 1};
        for (int r = 0; r < P; ++r) {
            const Range i{(uintptr_t)in[r], (uintptr_t)in[r] + bytes, r, 0};
            if (overlaps(o, i)) return DT_ERR_INVALID;
        }
        for (int k = q + 1; k < P; ++k) {
            const Range o2{(uintptr_t)out[k], (uintptr_t)out[k] + bytes, k, 1};
            if (overlaps(o, o2)) return DT_ERR_INVALID;
        }
    }
    // the part of rank i bound for rank j: h x w elements (h = R/P or R,
    // w = C or C/P) at (j h, 0) or (0, j w) of X_i; it lands at row i h
    // (src_dim 0, output width w) or column i w (src_dim 1, output width P w)
    const size_t h = dest_dim == 0 ? R / P : R, w = dest_dim == 1 ? C / P : C;
    const size_t out_w = src_dim == 1 ? (size_t)P * w : w;
    std::vector<dt::Copy2dSeg> segs((size_t)P * P);
    bool vec = (w * es) % 16 == 0 && (C * es) % 16 == 0 && (out_w * es) % 16 == 0;
    for (int i = 0; i < P; ++i) {
        vec = vec && aligned16(in[i]) && aligned16(out[i]);
        for (int j = 0; j < P; ++j) {
            dt::Copy2dSeg &sg = segs[(size_t)i * P + j];
            memset(&sg, 0, sizeof sg);
            const size_t src_off = dest_dim == 0 ? (size_t)j * h * C : (size_t)j * w;
            sg.src = static_cast<const unsigned char *>(in[i]) + src_off * es;
            sg.src_pitch = C * es;
            sg.dst = j;
            sg.dst_off = (src_dim == 0 ? (size_t)i * h * out_w : (size_t)i * w) * es;
            sg.dst_pitch = out_w * es;
            sg.rows = h;
            sg.row_bytes = w * es;
            dt::set_src_bounds(sg, in[i], bytes);
        }
    }
    void *outs[DT_MAX_RANKS] = {};
    uint64_t ob[DT_MAX_RANKS] = {};
    for (int q = 0; q < P; ++q) {
        outs[q] = out[q];
        ob[q] = bytes;
    }
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(dt::launch_copy2d(segs.data(), P * P, outs, ob, vec, error_sink(g), g->device,
                                         static_cast<cudaStream_t>(stream)));
}

dt_status dt_barrier(dt_group_t g, int rank, void *stream)
{
    DT_TRACE();
    if (!g) return DT_ERR_INVALID;
    if (rank != DT_ALL_RANKS)
        return rank_local(g, rank, make_call(CK_BARRIER, nullptr, nullptr, 0, 0, 0, 0, 0, stream));
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if ((st = check_rank(g, rank)) != DT_OK) return st;
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return issue_barrier(g, static_cast<cudaStream_t>(stream));
}

dt_status dt_async_begin(dt_group_t g, void *stream, void **comm_stream)
{
    DT_TRACE();
    if (!g || !comm_stream) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (g->scope_open) return DT_ERR_INVALID;
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    // syncStream: the communication stream waits for the caller's stream
    cudaError_t e = cudaEventRecord(g->scope_start, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamWaitEvent(g->comm, g->scope_start, 0);
    if (e != cudaSuccess) return cuda_status(e);
    g->scope_open = true;
    *comm_stream = g->comm;
    return DT_OK;
}

dt_status dt_async_end(dt_group_t g, dt_work_t *work)
{
    DT_TRACE();
    if (!g || !work) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    if (!g->scope_open) return DT_ERR_INVALID;
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    dt_work *w = nullptr;
    if (!g->work_free.empty()) {
        w = g->work_free.back();
        g->work_free.pop_back();
    } else {
        w = new (std::nothrow) dt_work;
        if (!w) return DT_ERR_OOM;
        w->g = g;
        cudaError_t e = cudaEventCreateWithFlags(&w->end, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            delete w;
            return cuda_status(e);
        }
        g->work_all.push_back(w);
    }
    cudaError_t e = cudaEventRecord(w->end, g->comm);
    g->scope_open = false;
    if (e != cudaSuccess) {
        g->work_free.push_back(w);
        return cuda_status(e);
    }
    *work = w;
    return DT_OK;
}

dt_status dt_work_wait(dt_work_t w, void *stream)
{
    DT_TRACE();
    if (!w || !w->g) return DT_ERR_INVALID;
    DeviceScope scope(w->g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    return cuda_status(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), w->end, 0));
}

dt_status dt_work_query(dt_work_t w)
{
    if (!w || !w->g) return DT_ERR_INVALID;
    DeviceScope scope(w->g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    const cudaError_t e = cudaEventQuery(w->end);
    if (e == cudaSuccess) return DT_OK;
    if (e == cudaErrorNotReady) {
        (void)cudaGetLastError();   // a not-ready query is not an error
        return DT_NOT_READY;
    }
    return DT_ERR_CUDA;
}

dt_status dt_work_free(dt_work_t w)
{
    if (!w || !w->g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(w->g->mu);
    w->g->work_free.push_back(w);
    return DT_OK;
}

dt_status dt_debug_read_window(dt_group_t g, int32_t *host_out, void *stream)
{
    if (!g || !host_out) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, g->d_win, (size_t)g->P * g->P * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

dt_status dt_debug_ring_after_barrier(dt_group_t g, const void *const *in, void *const *stage,
                                      void *const *out, size_t bytes, void *stream)
{
    if (!g) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    if (!in || !stage || !out) return DT_ERR_INVALID;
    const int P = g->P;
    dt::RingParams rp;
    memset(&rp, 0, sizeof rp);
    for (int r = 0; r < P; ++r) {
        if (bytes && (!in[r] || !stage[r] || !out[r])) return DT_ERR_INVALID;
        rp.in[r] = static_cast<const unsigned char *>(in[r]);
        rp.stage[r] = static_cast<unsigned char *>(stage[r]);
        rp.out[r] = static_cast<unsigned char *>(out[r]);
    }
    rp.bytes = bytes;
    rp.bar = barrier_params(g, 0, timeout_ns(g));
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    cudaError_t e = dt::launch_ring(rp, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    g->barriers_issued++;
    return DT_OK;
}

dt_status dt_debug_barrier_expect(dt_group_t g, int extra, uint32_t timeout_ms, void *stream)
{
    if (!g || extra < 1 || timeout_ms < 1 || timeout_ms > 10000) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g->mu);
    dt_status st = take_device_error(g);
    if (st != DT_OK) return st;
    DeviceScope scope(g->device);
    if (!scope.ok) return DT_ERR_CUDA;
    const dt::BarrierParams b = barrier_params(g, extra, (uint64_t)timeout_ms * 1000000ull);
    cudaError_t e = dt::launch_barrier(b, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    g->barriers_issued++;
    return DT_OK;
}

// ---- tracing (DT_TIMELINE=1 builds) ------------------------------------------

#ifdef DT_TIMELINE
namespace {
std::mutex g_tl_mu;
dt_timeline_record *g_tl_rec = nullptr;
unsigned long long *g_tl_count = nullptr;
size_t g_tl_cap = 0;
int g_tl_device = -1;
}  // namespace
#endif

dt_status dt_timeline_start(size_t max_records)
{
#ifdef DT_TIMELINE
    if (max_records == 0 || max_records > ((size_t)1 << 28)) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_tl_mu);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return DT_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DT_ERR_CUDA;
    if (g_tl_rec) cudaFree(g_tl_rec);
    if (g_tl_count) cudaFree(g_tl_count);
    g_tl_rec = nullptr;
    g_tl_count = nullptr;
    cudaError_t e = cudaMalloc(&g_tl_rec, max_records * sizeof(dt_timeline_record));
    if (e == cudaSuccess) e = cudaMalloc(&g_tl_count, sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(g_tl_count, 0, sizeof(unsigned long long));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? DT_ERR_OOM : DT_ERR_CUDA;
    g_tl_cap = max_records;
    g_tl_device = device;
    const dt::TimelineSink sink{g_tl_rec, g_tl_count, (unsigned long long)max_records};
    dt::bind_timeline_reduce(&sink);
    dt::bind_timeline_reduce_shift(&sink);
    dt::bind_timeline_copy(&sink);
    dt::bind_timeline_bucket(&sink);
    dt::bind_timeline_barrier(&sink);
    return cudaDeviceSynchronize() == cudaSuccess ? DT_OK : DT_ERR_CUDA;
#else
    (void)max_records;
    return DT_ERR_UNSUPPORTED;
#endif
}

uint32_t dt_build_flags(void)
{
    uint32_t f = 0;
#ifdef DT_NVTX
    f |= DT_BUILD_NVTX;
#endif
#ifdef DT_TIMELINE
    f |= DT_BUILD_TIMELINE;
#endif
#ifdef DT_BOUNDS
    f |= DT_BUILD_BOUNDS;
#endif
    return f;
}

dt_status dt_timeline_mark(void *stream, uint32_t tag)
{
#ifdef DT_TIMELINE
    return cuda_status(dt::launch_timeline_mark(tag, static_cast<cudaStream_t>(stream)));
#else
    (void)stream;
    (void)tag;
    return DT_ERR_UNSUPPORTED;
#endif
}

dt_status dt_timeline_read(dt_timeline_record *out, size_t max_records, size_t *n_records)
{
#ifdef DT_TIMELINE
    if (!n_records || (max_records && !out)) return DT_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_tl_mu);
    if (!g_tl_rec) return DT_ERR_INVALID;
    DeviceScope scope(g_tl_device);
    if (!scope.ok || cudaDeviceSynchronize() != cudaSuccess) return DT_ERR_CUDA;
    unsigned long long n = 0;
    if (cudaMemcpy(&n, g_tl_count, sizeof n, cudaMemcpyDeviceToHost) != cudaSuccess) return DT_ERR_CUDA;
    *n_records = (size_t)n;
    size_t k = n < g_tl_cap ? (size_t)n : g_tl_cap;
    if (k > max_records) k = max_records;
    if (k && cudaMemcpy(out, g_tl_rec, k * sizeof(dt_timeline_record), cudaMemcpyDeviceToHost) !=
                 cudaSuccess)
        return DT_ERR_CUDA;
    return DT_OK;
#else
    (void)out;
    (void)max_records;
    (void)n_records;
    return DT_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
