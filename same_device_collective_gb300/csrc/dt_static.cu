// Allocation-free variant of the fused bucket all-reduce.
//
// Some callers cannot let a library call cudaMalloc: applications that own
// all device memory through their own pool (a library's cudaMalloc bypasses
// their accounting and can fail once the pool has taken the device), and code
// on a latency-critical path that must not stall the other streams
// (cudaMalloc and cudaFree can synchronise the whole device).  They cannot
// create a dt_group, which allocates its window and plan scratch.
// dt_bucket_allreduce_static serves them: the tensor and pointer tables that
// the bucket kernel reads live in a fixed file-scope device array of
// kStaticScratchBytes, staged from a fixed host array, so a call allocates
// nothing on the device or the host.
//
// Costs and rules of the fixed array:
//   - every GPU that loads this library holds the array (1 MiB) until the
//     process exits;
//   - every call shares it and it keeps the last call's contents; a call
//     whose tables differ from the last ones copied to its device overwrites
//     the part it uses before its kernels read it, and a call that repeats
//     them (same device, ranks, dtype, cap, gradients and counts) reuses them
//     without a copy;
//   - calls that overlap on the GPU (issued on different streams without
//     ordering between them) race on the array; calls on one stream are safe;
//   - the copy is from pageable host memory, which CUDA may complete only
//     after the work already queued on the stream: a call that copies can
//     block the host until then, a call that reuses the tables does not;
//   - a call on a stream that is being captured is refused (the copy would
//     be recorded as reading the host array at replay time, after later
//     calls have rewritten it);
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "dt_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)1 << 20;
constexpr int kMaxDevices = 64;

}  // namespace

// The fixed device array: file scope, internal linkage, one copy on every
// device that loads the library.  In host code its name is only a host-side
// stand-in; scratch_address() looks up the device address.
static __device__ __align__(256) unsigned char g_bucket_scratch[kStaticScratchBytes];

namespace {

// Host staging of the same size: copied with a pageable cudaMemcpyAsync,
// which returns once the bytes have left this array.
alignas(256) unsigned char h_bucket_staging[kStaticScratchBytes];
// What the last copy put on the device: its bytes and the arguments they
// encode.  A call that builds the same bytes for the same device, ranks,
// dtype and cap finds them there already.
alignas(256) unsigned char h_last_upload[kStaticScratchBytes];
struct UploadKey {
    int device = -1;
    int P = 0;
    int dtype = -1;
    size_t bytes = 0;
};
UploadKey g_last_key;
// Gradient byte ranges for the overlap check: every range takes at least one
// 8-byte pointer of the table, so the table's limit bounds their number.
struct GradRange {
    uintptr_t lo, hi;
};
GradRange h_ranges[kStaticScratchBytes / sizeof(void *)];

// One launch per bucket of the tables last built.
struct Launch {
    size_t tb, te, start_off;
    uint64_t total, per_block;
    uint32_t blocks;
};
constexpr size_t kMaxBuckets = 4096;
Launch g_launches[kMaxBuckets];

// The arguments of the call whose tables the device array holds (with
// g_last_key): a call that repeats them launches from g_launches without
// building or comparing its tables.
constexpr size_t kMaxTensors = kStaticScratchBytes / (sizeof(void *) + sizeof(dt::BucketTensor));
struct LastCall {
    bool valid = false;
    int device = -1, P = 0, dtype = -1;
    size_t n_tensors = 0, cap = 0, ptr_bytes = 0, tab_bytes = 0, n_launches = 0;
};
LastCall g_last_call;
void *h_last_grads[kStaticScratchBytes / sizeof(void *)];
size_t h_last_counts[kMaxTensors];
std::mutex g_static_mu;
void *g_scratch_addr[kMaxDevices] = {};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Set-up, once per device, with that device current.
cudaError_t scratch_address(int device, void **out)
{
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_bucket_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

// One kernel per bucket of the tables in the device array d, in order on s.
// No signal barrier runs between buckets: with no group there is no window,
// and stream order already orders the buckets.
dt_status launch_all(const unsigned char *d, size_t ptr_bytes, size_t tab_bytes, size_t nl, int P,
                     int dtype, int op, int device, cudaStream_t s)
{
    dt::BucketParams bp;
    memset(&bp, 0, sizeof bp);   // win = nullptr: no barrier block
    bp.ptrs = reinterpret_cast<void *const *>(d);
    bp.P = P;
    bp.avg_pow2 = (P & (P - 1)) == 0;
    bp.avg_scale = bp.avg_pow2 ? 1.0f / (float)P : 0.0f;
    bool kernel_before = false;   // a bucket kernel of this call is already queued
    for (size_t i = 0; i < nl; ++i) {
        const Launch &L = g_launches[i];
        bp.tensors = reinterpret_cast<const dt::BucketTensor *>(d + ptr_bytes) + L.tb;
        bp.block_start = reinterpret_cast<const uint32_t *>(d + ptr_bytes + tab_bytes) + L.start_off;
        bp.ntensors = (uint32_t)(L.te - L.tb);
        bp.total = L.total;
        bp.per_block = L.per_block;
        bp.blocks = L.blocks;
        bp.early = kernel_before ? 1u : 0u;
        bool launched = false;
        if (dt::launch_bucket(bp, dtype, op, device, s, &launched) != cudaSuccess) return DT_ERR_CUDA;
        kernel_before = kernel_before || launched;
    }
    return DT_OK;
}

}  // namespace

extern "C" dt_status dt_bucket_allreduce_static(int world_size, void *const *grads,
                                                const size_t *counts, size_t n_tensors, int dtype,
                                                int op, size_t bucket_cap_bytes, void *stream)
{
    if (world_size < 1 || world_size > DT_MAX_RANKS) return DT_ERR_INVALID;
    if (dtype != DT_BF16 && dtype != DT_F32)
        return dtype == DT_I32 ? DT_ERR_UNSUPPORTED : DT_ERR_INVALID;
    if (op != DT_SUM && op != DT_AVG)
        return (op >= DT_SUM && op <= DT_SUM_STEPWISE) ? DT_ERR_UNSUPPORTED : DT_ERR_INVALID;
    if (n_tensors && (!grads || !counts)) return DT_ERR_INVALID;
    const int P = world_size;
    const size_t es = dtype == DT_BF16 ? 2 : 4;
    const size_t cap = bucket_cap_bytes ? bucket_cap_bytes : DT_DEFAULT_BUCKET_CAP_BYTES;

    // the pointer and tensor tables must fit the fixed array (checked first:
    // nothing below runs on a request that cannot be served)
    if (n_tensors > kStaticScratchBytes / (P * sizeof(void *) + sizeof(dt::BucketTensor)))
        return DT_ERR_TOO_LARGE;
    for (size_t t = 0; t < n_tensors; ++t) {
        if (counts[t] > SIZE_MAX / 16) return DT_ERR_INVALID;
        for (int p = 0; p < P && counts[t]; ++p)
            if (!grads[t * P + p]) return DT_ERR_INVALID;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) return DT_ERR_CUDA;
    if (capture != cudaStreamCaptureStatusNone) return DT_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_static_mu);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return DT_ERR_CUDA;

    const LastCall &lc = g_last_call;
    if (lc.valid && lc.device == device && lc.P == P && lc.dtype == dtype && lc.cap == cap &&
        lc.n_tensors == n_tensors && memcmp(h_last_counts, counts, n_tensors * sizeof(size_t)) == 0 &&
        memcmp(h_last_grads, grads, n_tensors * P * sizeof(void *)) == 0) {
        void *scratch = nullptr;
        if (scratch_address(device, &scratch) != cudaSuccess) return DT_ERR_CUDA;
        return launch_all(static_cast<const unsigned char *>(scratch), lc.ptr_bytes, lc.tab_bytes,
                          lc.n_launches, P, dtype, op, device, s);
    }
    g_last_call.valid = false;   // the tables are rebuilt below

    // plan: [T * P pointers][T tensor entries][block starts of every bucket];
    // buckets are consecutive tensors, greedy in order under the cap (the
    // rule of dt_bucket_plan).  Sizes are checked against the fixed array as
    // the plan grows, before anything is enqueued.
    const size_t ptr_bytes = n_tensors * P * sizeof(void *);
    const size_t tab_bytes = n_tensors * sizeof(dt::BucketTensor);
    if (ptr_bytes + tab_bytes > kStaticScratchBytes) return DT_ERR_TOO_LARGE;
    memcpy(h_bucket_staging, grads, ptr_bytes);
    dt::BucketTensor *tab = reinterpret_cast<dt::BucketTensor *>(h_bucket_staging + ptr_bytes);
    uint32_t *starts = reinterpret_cast<uint32_t *>(h_bucket_staging + ptr_bytes + tab_bytes);
    const size_t max_starts = (kStaticScratchBytes - ptr_bytes - tab_bytes) / sizeof(uint32_t);

    Launch *const launches = g_launches;   // guarded by g_static_mu
    size_t nl = 0, n_starts = 0;
    size_t t = 0;
    while (t < n_tensors) {
        // one bucket: [tb, te)
        const size_t tb = t;
        size_t filled = 0;
        uint64_t first = 0;
        while (t < n_tensors && !(filled > 0 && filled + counts[t] * es > cap)) {
            bool al = true;
            for (int p = 0; p < P; ++p) al = al && aligned16(grads[t * P + p]);
            tab[t].first = first;
            tab[t].count = counts[t];
            tab[t].slot = (uint32_t)t | (al ? 0x80000000u : 0u);
            tab[t].block0 = 0;   // set below, once the bucket's slice length is known
            first += dt::bucket_padded(counts[t], dtype);
            filled += counts[t] * es;
            ++t;
        }
        if (first == 0) continue;   // only empty tensors
        if (nl == kMaxBuckets) return DT_ERR_TOO_LARGE;
        Launch &L = launches[nl++];
        L.tb = tb;
        L.te = t;
        L.total = first;
        if (dt::bucket_grid(dtype, op, P, L.total, device, &L.blocks, &L.per_block) != cudaSuccess)
            return DT_ERR_CUDA;
        // one block per slice of a tensor: the grid's slice length, cut at tensor ends
        uint64_t nblk = 0;
        for (size_t k = L.tb; k < L.te; ++k) nblk += dt::bucket_tensor_blocks(counts[k], dtype, L.per_block);
        if (n_starts + nblk > max_starts) return DT_ERR_TOO_LARGE;
        L.blocks = (uint32_t)nblk;
        L.start_off = n_starts;
        uint32_t block = 0;
        for (size_t k = L.tb; k < L.te; ++k) {
            tab[k].block0 = block;
            const uint64_t nb_k = dt::bucket_tensor_blocks(counts[k], dtype, L.per_block);
            for (uint64_t j = 0; j < nb_k; ++j, ++block) starts[n_starts++] = (uint32_t)(k - L.tb);
        }
    }
    if (nl == 0) return DT_OK;

    const size_t plan_bytes = ptr_bytes + tab_bytes + n_starts * sizeof(uint32_t);
    const bool reuse = g_last_key.device == device && g_last_key.P == P && g_last_key.dtype == dtype &&
                       g_last_key.bytes == plan_bytes &&
                       memcmp(h_last_upload, h_bucket_staging, plan_bytes) == 0;
    if (!reuse) {
        // No two gradient buffers may overlap: sort their byte ranges and
        // compare neighbours (the first overlap in start order is always
        // between neighbours).  A call that repeats the last tables was
        // checked when they were copied.
        size_t nr = 0;
        for (size_t t = 0; t < n_tensors; ++t)
            for (int p = 0; p < P && counts[t]; ++p) {
                const uintptr_t lo = (uintptr_t)grads[t * P + p];
                h_ranges[nr++] = GradRange{lo, lo + counts[t] * es};
            }
        std::sort(h_ranges, h_ranges + nr,
                  [](const GradRange &a, const GradRange &b) { return a.lo < b.lo; });
        for (size_t i = 1; i < nr; ++i)
            if (h_ranges[i].lo < h_ranges[i - 1].hi) return DT_ERR_INVALID;
    }

    void *scratch = nullptr;
    if (scratch_address(device, &scratch) != cudaSuccess) return DT_ERR_CUDA;
    if (!reuse) {
        g_last_key = UploadKey{};   // the device copy is in flux until this copy is queued
        if (cudaMemcpyAsync(scratch, h_bucket_staging, plan_bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return DT_ERR_CUDA;
        memcpy(h_last_upload, h_bucket_staging, plan_bytes);
        g_last_key = UploadKey{device, P, dtype, plan_bytes};
    }

    g_last_call = LastCall{true, device, P, dtype, n_tensors, cap, ptr_bytes, tab_bytes, nl};
    memcpy(h_last_grads, grads, ptr_bytes);
    memcpy(h_last_counts, counts, n_tensors * sizeof(size_t));
    return launch_all(static_cast<const unsigned char *>(scratch), ptr_bytes, tab_bytes, nl, P, dtype,
                      op, device, s);
}
