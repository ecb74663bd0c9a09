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
//   - every call shares it and it keeps the last call's contents; each call
//     overwrites the part it uses before its kernels read it;
//   - calls that overlap on the GPU (issued on different streams without
//     ordering between them) race on the array; calls on one stream are safe;
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture begins.
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

    // no two gradient buffers may overlap: quadratic check, no allocation
    for (size_t t = 0; t < n_tensors; ++t)
        for (int p = 0; p < P && counts[t]; ++p) {
            const uintptr_t lo = (uintptr_t)grads[t * P + p], hi = lo + counts[t] * es;
            for (size_t u = t; u < n_tensors; ++u)
                for (int q = (u == t ? p + 1 : 0); q < P && counts[u]; ++q) {
                    const uintptr_t lo2 = (uintptr_t)grads[u * P + q], hi2 = lo2 + counts[u] * es;
                    if (lo < hi2 && lo2 < hi) return DT_ERR_INVALID;
                }
        }

    std::lock_guard<std::mutex> lock(g_static_mu);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return DT_ERR_CUDA;

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

    struct Launch {
        size_t tb, te, start_off;
        uint64_t total, per_block;
        uint32_t blocks;
    };
    static Launch launches[4096];   // buckets of this call (guarded by g_static_mu)
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
            tab[t].pad = 0;
            first += dt::bucket_padded(counts[t], dtype);
            filled += counts[t] * es;
            ++t;
        }
        if (first == 0) continue;   // only empty tensors
        if (nl == sizeof(launches) / sizeof(launches[0])) return DT_ERR_TOO_LARGE;
        Launch &L = launches[nl++];
        L.tb = tb;
        L.te = t;
        L.total = first;
        if (dt::bucket_grid(dtype, op, P, L.total, device, &L.blocks, &L.per_block) != cudaSuccess)
            return DT_ERR_CUDA;
        if (n_starts + L.blocks > max_starts) return DT_ERR_TOO_LARGE;
        L.start_off = n_starts;
        size_t k = L.tb;
        for (uint32_t j = 0; j < L.blocks; ++j) {
            const uint64_t lo = (uint64_t)j * L.per_block;
            while (k + 1 < L.te && tab[k + 1].first <= lo) ++k;
            starts[n_starts++] = (uint32_t)(k - L.tb);
        }
    }
    if (nl == 0) return DT_OK;

    void *scratch = nullptr;
    if (scratch_address(device, &scratch) != cudaSuccess) return DT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(scratch, h_bucket_staging,
                                    ptr_bytes + tab_bytes + n_starts * sizeof(uint32_t),
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return DT_ERR_CUDA;

    const unsigned char *d = static_cast<const unsigned char *>(scratch);
    dt::BucketParams bp;
    bp.ptrs = reinterpret_cast<void *const *>(d);
    bp.P = P;
    bp.avg_pow2 = (P & (P - 1)) == 0;
    bp.avg_scale = bp.avg_pow2 ? 1.0f / (float)P : 0.0f;
    // one launch per bucket, no signal barrier between buckets: with no group
    // there is no window, and stream order already orders the buckets
    for (size_t i = 0; i < nl; ++i) {
        const Launch &L = launches[i];
        bp.tensors = reinterpret_cast<const dt::BucketTensor *>(d + ptr_bytes) + L.tb;
        bp.block_start = reinterpret_cast<const uint32_t *>(d + ptr_bytes + tab_bytes) + L.start_off;
        bp.ntensors = (uint32_t)(L.te - L.tb);
        bp.total = L.total;
        bp.per_block = L.per_block;
        if (dt::launch_bucket(bp, dtype, op, device, s) != cudaSuccess) return DT_ERR_CUDA;
    }
    return DT_OK;
}
