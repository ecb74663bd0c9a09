// Internal declarations of the same-device collective library shared by the
// kernels and the host code: kernel parameter blocks and launchers.  The host
// side's group object is in dt_group.h.  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <utility>

#include "dt.h"

namespace dt {

constexpr int kThreads = 256;                          // threads per block, all data kernels
constexpr int kMaxSeg = DT_MAX_RANKS * DT_MAX_RANKS;   // all-to-all: P^2 chunk copies

// First device-side failure, written once (atomicCAS on code) by the kernel
// that hit it, mirrored into host-mapped memory so the host can read it
// without synchronising.
struct DevError {
    int32_t code;
    int32_t rank;
    int32_t peer;
    int32_t gen;
};

// Where a kernel with a bounded wait reports that the wait ran out.
struct ErrorSink {
    DevError *err;        // device error word
    DevError *err_host;   // device view of its host-mapped mirror
    uint64_t timeout_ns;
};

// ---- reduction (AllReduce, ReduceScatter) ---------------------------------
// Job j (blockIdx.y) reduces elements [j * job_stride, j * job_stride + n)
// of every input and writes them to out[j * out_per_job + k], k < out_per_job.
// AllReduce: 1 job, out_per_job = P (or 1 shared).  ReduceScatter: P jobs,
// out_per_job = 1, job_stride = n.  The vector kernel takes 16-byte-aligned
// pointers.  Buffers that all lie the same whole number of elements past a
// 16-byte boundary reach it advanced by `head` elements to that boundary
// (and n reduced by head); the kernel then reduces the head elements before
// each job's start on the element path, at negative indices.
struct ReduceParams {
    const void *in[DT_MAX_RANKS];
    void *out[DT_MAX_RANKS];
    uint64_t n;
    uint64_t job_stride;
    float avg_scale;     // AVG with P a power of two: exact 1/P
    int32_t avg_pow2;    // 1: multiply by avg_scale (same rounding as /P); 0: divide by P
    int32_t P;
    int32_t out_per_job;
    uint32_t head;       // elements before the pointers above, 0..15
    uint32_t pad;
#ifdef DT_BOUNDS
    // each input and output buffer as the call's arguments give it
    uint64_t in_lo[DT_MAX_RANKS], in_hi[DT_MAX_RANKS];
    uint64_t out_lo[DT_MAX_RANKS], out_hi[DT_MAX_RANKS];
    ErrorSink sink;
#endif
};

// ---- byte copies (AllGather, AllToAll) ------------------------------------
// Segment s copies `bytes` from src to out[dst_first + k] + dst_off for
// k < dst_count; segments are cut into tiles of tile_bytes and tile t of the
// launch belongs to the segment with tile_begin <= t < next tile_begin.
// Callers leave head and tail at 0.  When a segment's source and
// destinations lie the same distance past a 16-byte boundary, the launcher
// moves the bytes before the source's first boundary and after its last one
// into head and tail: the segment then covers [src - head, src + bytes +
// tail), its 16-byte-aligned middle [src, src + bytes) goes through the
// vector or bulk-copy kernels, and the edges byte by byte.
struct CopySeg {
    const unsigned char *src;
    uint64_t bytes;
    uint64_t dst_off;
    uint64_t tile_begin;
    int16_t dst_first;    // < DT_MAX_RANKS^2
    int16_t dst_count;    // <= DT_MAX_RANKS^2
    uint8_t head;         // < 16
    uint8_t tail;         // < 16
    uint16_t one_pass;    // shifting copy: the destinations share their offset past a
                          // 16-byte boundary, so one pass over the source serves them all
#ifdef DT_BOUNDS
    uint64_t src_lo, src_hi;   // the source buffer the segment lies in
#endif
};
#ifndef DT_BOUNDS
// 40 bytes: an AllToAll's 256 entries take 10 KiB of the kernel's parameter
// block.
static_assert(sizeof(CopySeg) == 40, "segment entries stay 40 bytes");
#endif

#ifdef DT_BOUNDS
// DT_BOUNDS_TRIM=<bytes> in the environment (bounds-checked builds only):
// every destination extent is recorded that many bytes shorter than the call
// gives it.  The kernels then skip stores that lie inside the real buffers
// and report them, which shows the checker at work on correct kernels.
inline uint64_t bounds_trim()
{
    static const uint64_t trim = [] {
        const char *e = getenv("DT_BOUNDS_TRIM");
        return e ? (uint64_t)strtoull(e, nullptr, 10) : 0ull;
    }();
    return trim;
}

inline uint64_t trimmed_end(uint64_t lo, uint64_t bytes)
{
    const uint64_t t = bounds_trim();
    return lo + (bytes > t ? bytes - t : 0);
}
#endif

// The buffers a reduction reads and writes, as the call's arguments give
// them (checked in DT_BOUNDS builds only).
inline void set_reduce_bounds(ReduceParams &p, const void *const *in, uint64_t in_bytes,
                              void *const *out, uint64_t out_bytes, int nin, int nout,
                              const ErrorSink &sink)
{
#ifdef DT_BOUNDS
    for (int r = 0; r < nin; ++r) {
        p.in_lo[r] = reinterpret_cast<uint64_t>(in[r]);
        p.in_hi[r] = p.in_lo[r] + in_bytes;
    }
    for (int q = 0; q < nout; ++q) {
        p.out_lo[q] = reinterpret_cast<uint64_t>(out[q]);
        p.out_hi[q] = trimmed_end(p.out_lo[q], out_bytes);
    }
    p.sink = sink;
#else
    (void)p; (void)in; (void)in_bytes; (void)out; (void)out_bytes; (void)nin; (void)nout; (void)sink;
#endif
}

// The source buffer a segment lies in (checked in DT_BOUNDS builds only).
inline void set_src_bounds(CopySeg &sg, const void *lo, uint64_t bytes)
{
#ifdef DT_BOUNDS
    sg.src_lo = reinterpret_cast<uint64_t>(lo);
    sg.src_hi = sg.src_lo + bytes;
#else
    (void)sg;
    (void)lo;
    (void)bytes;
#endif
}

template <int NSEG, int NOUT = DT_MAX_RANKS>
struct CopyParams {
    void *out[NOUT];
#ifdef DT_BOUNDS
    uint64_t out_lo[NOUT], out_hi[NOUT];   // each destination buffer
#endif
    ErrorSink sink;
    uint64_t tile_bytes;
    uint64_t total_tiles;
    int32_t nseg;
    uint32_t seg_tiles;   // tiles of every segment when they are all equal (and fewer than 2^32
                          // tiles in all): the segment of tile t is t / seg_tiles; else 0
    CopySeg seg[NSEG];
};

// ---- 2-D strided copies (AllToAll along other dims) -----------------------
// Segment s copies `rows` rows of row_bytes from src (row pitch src_pitch) to
// out[dst] + dst_off (row pitch dst_pitch).  Tiles are runs of whole rows.
struct Copy2dSeg {
    const unsigned char *src;
    uint64_t src_pitch;
    uint64_t dst_off;
    uint64_t dst_pitch;
    uint64_t rows;
    uint64_t row_bytes;
    uint64_t rows_per_tile;
    uint64_t tile_begin;
    int32_t dst;
    int32_t pad;
#ifdef DT_BOUNDS
    uint64_t src_lo, src_hi;   // the source buffer the segment lies in
#endif
};

inline void set_src_bounds(Copy2dSeg &sg, const void *lo, uint64_t bytes)
{
#ifdef DT_BOUNDS
    sg.src_lo = reinterpret_cast<uint64_t>(lo);
    sg.src_hi = sg.src_lo + bytes;
#else
    (void)sg;
    (void)lo;
    (void)bytes;
#endif
}

struct Copy2dParams {
    void *out[DT_MAX_RANKS];
#ifdef DT_BOUNDS
    uint64_t out_lo[DT_MAX_RANKS], out_hi[DT_MAX_RANKS];
    ErrorSink sink;
#endif
    uint64_t total_tiles;
    int32_t nseg;
    uint32_t seg_tiles;   // as in CopyParams
    Copy2dSeg seg[DT_MAX_RANKS * DT_MAX_RANKS];
};

// ---- fused bucket all-reduce ----------------------------------------------
// A bucket's tensors laid end to end form its flattened element space, in
// which every tensor occupies its count rounded up to a whole 16-byte vector.
// Each tensor is cut into slices of per_block elements (its last slice
// shorter), one block per slice, so that no block works on two tensors:
// block b works on tensor block_start[b], on its elements [(b - block0) *
// per_block, + per_block) below its count.
struct BucketTensor {
    uint64_t first;   // first element in the bucket's flattened space
    uint64_t count;   // elements of the tensor
    uint32_t slot;    // row of P pointers in `ptrs`; bit 31: all 16-byte aligned
    uint32_t block0;  // the bucket's first block that works on this tensor
};

struct BucketParams {
    const BucketTensor *tensors;     // this bucket's tensors, in order
    const uint32_t *block_start;     // per block: index of its tensor
    void *const *ptrs;               // [n_slots][P]
    uint64_t total;                  // padded elements in the bucket
    uint64_t per_block;              // slice length, a multiple of the vector width
    uint32_t ntensors;
    int32_t P;
    float avg_scale;
    int32_t avg_pow2;
    // 1 in every bucket kernel of a call but the first: its blocks load their
    // first vectors before waiting for the previous kernel (see bucket_kernel)
    uint32_t early;
    uint32_t blocks;                 // data blocks (the barrier block comes after them)
    // The signal-window barrier after this bucket, run by one extra block at
    // the end of the grid (win != nullptr; see bucket_kernel): the group's
    // window [P][P], followed by rank_gen[P] and the counter of finished
    // blocks.
    int32_t *win;
    ErrorSink sink;
};

// Words of a group's barrier state: the window [P][P], the generations of the
// ranks [P], the bucket kernels' finished-block counter, padding.
constexpr size_t win_words(int P) { return (size_t)P * P + P + 4; }

// Elements a tensor occupies in the flattened space, and the grid the bucket
// kernel uses for `total` such elements (blocks the SMs hold at once).
uint64_t bucket_padded(uint64_t count, int dtype);
cudaError_t bucket_grid(int dtype, int op, int P, uint64_t total, int device, uint32_t *blocks,
                        uint64_t *per_block);
// Blocks (slices of per_block elements) of one tensor of `count` elements.
uint64_t bucket_tensor_blocks(uint64_t count, int dtype, uint64_t per_block);

// ---- barrier ----------------------------------------------------------------
struct BarrierParams {
    int32_t *win;        // [P][P]
    int32_t *rank_gen;   // [P]: barriers rank r has passed
    ErrorSink sink;
    int32_t P;
    int32_t extra;       // added to the threshold (failure injection); 0 normally
};

struct RingParams {
    BarrierParams bar;
    const unsigned char *in[DT_MAX_RANKS];
    unsigned char *stage[DT_MAX_RANKS];
    unsigned char *out[DT_MAX_RANKS];
    uint64_t bytes;
};

// ---- launchers (one per kernel family; each counts its launches) ----------
void count_launch();

// Programmatic dependent launch: kernels launched with it may start while the
// previous kernel on the stream finishes; every kernel here waits on its
// prerequisite grid (griddepcontrol.wait) before touching memory.  On by
// default; the environment variable DT_PDL=0 turns it off.
bool pdl_enabled();

// DT_LOG=1 in the environment: every launch prints its kernel, grid, block,
// dynamic shared memory, stream and launch attributes to stderr.
bool log_enabled();

// DT_DEBUG=1 in the environment: every launch is followed by a synchronisation
// of its stream (skipped while the stream is being captured), so a kernel that
// fails is reported by the call that launched it rather than by a later one.
bool debug_enabled();
cudaError_t debug_sync(cudaStream_t s, cudaError_t launched);
void log_launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool cooperative,
                cudaError_t result);

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*fn)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool cooperative, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cooperative) {
        attrs[n].id = cudaLaunchAttributeCooperative;
        attrs[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    count_launch();
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, std::forward<Args>(args)...);
    if (log_enabled()) log_launch(reinterpret_cast<const void *>(fn), grid, block, smem, s, cooperative, e);
    return debug_enabled() ? debug_sync(s, e) : e;
}
int sm_count(int device);
// Bytes of L2 cache on the device (cached per device).
uint64_t l2_bytes(int device);
// SMs x blocks of `fn` one SM holds at once (cached per kernel and device).
cudaError_t resident_blocks(const void *fn, int threads, int device, int *out,
                            size_t dyn_smem = 0);

cudaError_t launch_reduce(const ReduceParams &p, int dtype, int op, int jobs, bool vec,
                          int device, cudaStream_t s);
// nout destinations in `out` (up to DT_MAX_RANKS, or DT_MAX_RANKS^2 for the
// vector form of AllGather)
// out_bytes[k]: the size of destination buffer k (checked in DT_BOUNDS builds)
cudaError_t launch_copy(const CopySeg *segs, int nseg, void *const *out, const uint64_t *out_bytes,
                        int nout, bool vec, const ErrorSink &sink, int device, cudaStream_t s);
cudaError_t launch_copy2d(const Copy2dSeg *segs, int nseg, void *const *out, const uint64_t *out_bytes,
                          bool vec, const ErrorSink &sink, int device, cudaStream_t s);
// *launched (optional) tells whether a kernel went out: a bucket with no
// elements launches nothing, and then runs no barrier either.
cudaError_t launch_bucket(const BucketParams &p, int dtype, int op, int device, cudaStream_t s,
                          bool *launched = nullptr);
cudaError_t launch_barrier(const BarrierParams &p, cudaStream_t s);
cudaError_t launch_ring(const RingParams &p, cudaStream_t s);

}  // namespace dt
