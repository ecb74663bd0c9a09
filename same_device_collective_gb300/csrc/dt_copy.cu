// Byte-copy kernels behind AllGather (equal and uneven shards) and AllToAll.
//
// Both collectives of the DTorch ThreadGroup interface (§2.1) are pure data
// movement: AllGather writes every rank's shard into every rank's output at
// the shard's row offset, AllToAll sends chunk j of rank i to rank j.  The
// host turns a call into a list of segments (source range -> one or more
// destinations at one offset); one launch moves them all.  Each segment is
// cut into tiles and the grid (one to eight waves of blocks, see bulk_grid)
// strides over the tiles of all segments.
//
// 16-byte-aligned segments go through the copy engine (TMA bulk copies): a
// tile is loaded from HBM into shared memory once and stored from there to
// every destination of its segment, so a shard is read once however many
// ranks receive it and no register or load/store-unit traffic is spent on the
// bytes.  Destinations are written once and not read back here, so the
// stores carry an evict-first L2 policy: their dirty lines leave L2 early
// instead of being written back during the next kernel.  Segments whose
// source and destinations share their offset past a 16-byte boundary (views
// that start mid-vector) take the same kernels for their aligned middle and
// copy their few edge bytes alongside; any other layout takes a kernel that
// aligns every store and funnel-shifts the source into place.
#include <atomic>

#include "dt_internal.h"
#include "dt_device.cuh"
#include "dt_shift.cuh"
#include "dt_timeline.cuh"
#include "dt_bounds.cuh"

namespace dt {
namespace {

// The segment tile `tile` belongs to: a binary search over the segments'
// first tiles, which costs log2(segments) dependent parameter-space loads,
// or, in kernels built with kDivide, a division when the launcher set
// seg_tiles (every segment has that many tiles).  The division stays out of
// the other kernels' code altogether: even untaken, its branch slowed the
// single-thread 12-deep AllToAll stream by 4% (8 ranks, 16 MiB-1 GiB per
// rank), and taken by 8-10%, though the tiles and their order are the same.
template <bool kDivide, typename Params>
__device__ __forceinline__ int find_seg(const Params &p, uint64_t tile)
{
    if constexpr (kDivide) {
        if (p.seg_tiles) return (int)((uint32_t)tile / p.seg_tiles);
    }
    int lo = 0, hi = p.nseg - 1;      // last segment with tile_begin <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile_begin <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The head and tail bytes of the launch's segments (see CopySeg), byte by
// byte, in a small launch of their own next to the one that moves the
// segments' aligned middles (folding them into those kernels, on the bulk
// copy's idle lanes, slowed the aligned copies down: the 8-rank AllToAll of
// 512 MiB per rank lost 23%).  Block b takes
// segments b, b + gridDim.x, ...; its threads share each segment's edge bytes
// and destinations.
template <int NSEG, int NOUT>
__global__ void __launch_bounds__(kThreads)
copy_edge_kernel(const __grid_constant__ CopyParams<NSEG, NOUT> p)
{
    pdl_begin();
    for (int s = blockIdx.x; s < p.nseg; s += gridDim.x) {
        const CopySeg &sg = p.seg[s];
        const uint32_t h = sg.head, e = (uint32_t)sg.head + sg.tail;
        if (e == 0) continue;
        for (uint32_t i = threadIdx.x; i < e * (uint32_t)sg.dst_count; i += kThreads) {
            const uint32_t k = i / e, b = i - k * e;
            const int64_t off = b < h ? (int64_t)b - (int64_t)h : (int64_t)(sg.bytes + (b - h));
            const int d = sg.dst_first + (int)k;
            unsigned char *to = static_cast<unsigned char *>(p.out[d]) + (int64_t)sg.dst_off + off;
            if (DT_IN_BOUNDS(span_in(sg.src + off, 1, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyEdge, s,
                             sg.src + off, sg.src_lo) &&
                DT_IN_BOUNDS(span_in(to, 1, p.out_lo[d], p.out_hi[d]), p.sink, kBoundsCopyEdge,
                             kMaxSeg + d, to, p.out_lo[d]))
                *to = sg.src[off];
        }
    }
}

// Bulk-copy (TMA) kernel for 16-byte-aligned segments.  One thread per block
// drives the copy engine: it keeps kBulkStages tiles of
// shared memory in flight (global -> shared bulk loads that complete on one
// mbarrier per stage) and, as each tile lands, issues one shared -> global
// bulk store per destination of its segment.  A stage is refilled once the
// stores of the tile it held have finished reading it (bulk async-groups).
// Every mbarrier wait is bounded: a wait that runs out records DT_ERR_TIMEOUT
// (rank -1, peer = tile), drains the loads still in flight with bounded waits
// and returns.
constexpr int kBulkThreads = 32;

// Tile size and pipeline depth, measured on GB300 per launch layout:
//   kStream: the P^2 single-destination segments of an AllToAll of up to 8
//            ranks whose data does not fit in L2 stream best as 16 KiB tiles
//            12 deep, one block per SM (8 ranks, 64-512 MiB per rank:
//            7.0-7.1 TB/s; every shallower or split shape tried measured
//            6.4-6.6);
//   kSplit:  the other AllToAlls of 8 or more ranks: 16 KiB tiles 4 deep, so
//            three blocks share an SM and three threads issue its copies.
//            A block's single issuing thread bounds the 12-deep shape when
//            the copies come from L2 (8 ranks, 4 MiB per rank: 5.5 -> 9.1
//            TB/s) and when the 256-entry segment table of 16 ranks makes
//            each tile's segment lookup slow (16 ranks, 4-256 MiB per rank:
//            4.7-5.9 -> 6.3-7.7 TB/s);
//   kGather: few segments (equal or uneven shards, shared or per-rank
//            outputs of moderate size, row-block copies): 32 KiB x 6;
//   kGatherSplit: the same launches with at least 3 tiles of 16 KiB per SM
//            and at most 8 destinations per segment: 16 KiB x 4, three
//            blocks per SM (2-rank AllToAll of 64 MiB per rank +3%, 16 MiB
//            +8%; ReplicateToShard of 4 ranks +2%; 2-, 4- and 8-rank gathers
//            of 1-4 MiB shards +5-8%).  With fewer tiles the blocks crowd onto
//            fewer SMs (4-rank gather of 1 MiB shards -12%), and 16-rank
//            gathers, with 16 stores per tile, lost 3-22%;
//   kWide:   large launches whose segments each store to 2..8 destinations
//            (per-rank gathers): every tile is stored several times, so each
//            stage stays busy long enough that two 96 KiB stages beat more,
//            smaller ones when tiles are plentiful (16+ per SM);
//   kWideSplit: the same gathers with 4-16 of those tiles per SM: 32 KiB x 3,
//            two blocks per SM, so two threads per SM issue the stores (the
//            4-rank gather of 16 MiB shards in the RS+AG step 51.0 -> 47.4 us
//            with events around it, the step 98.4 -> 95.8 us; 2 ranks of
//            64 MiB +2%).
// Shared memory: the stages' mbarriers (8 bytes each, area rounded up to 128
// bytes so the tile buffers stay 128-byte aligned), then the tile buffers.
enum BulkKind { kStream = 0, kGather = 1, kWide = 2, kSplit = 3, kWideSplit = 4, kGatherSplit = 5 };

// Blocks per launch.  One block per SM holds a shape's stages; extra blocks
// run in later waves, and the hardware hands each to whichever SM frees up
// first, so SMs that stream slower take fewer tiles.  That balancing pays
// when tiles are plentiful (16+ per SM: 8 waves; the uneven 8-rank gather
// +8%, its shared-output form +6%) and for the wide shape's few large tiles
// (4 waves: the RS+AG step 100.7 -> 98.7 us), but restarting the pipeline
// costs more than it saves for a few thousand small tiles served from L2
// (ReplicateToShard -14% at 4 waves) and for the AllToAll (-1%).
template <int KIND>
uint64_t bulk_grid(uint64_t tiles, int resident)
{
    const bool plenty = tiles >= 16 * (uint64_t)resident;
    const uint64_t waves = KIND == kStream || KIND == kSplit ? 1
                           : plenty ? 8 : KIND == kWide || KIND == kWideSplit ? 4 : 1;
    const uint64_t cap = (uint64_t)resident * waves;
    return tiles < cap ? tiles : cap;
}

template <int KIND>
struct BulkShape {
    static constexpr int kStages = KIND == kStream ? 12 : KIND == kSplit || KIND == kGatherSplit ? 4
                                   : KIND == kGather ? 6 : KIND == kWideSplit ? 3 : 2;
    static constexpr int kTile = KIND == kStream || KIND == kSplit || KIND == kGatherSplit ? 16384
                                 : KIND == kGather || KIND == kWideSplit ? 32768 : 98304;
    static constexpr size_t kBarBytes = ((size_t)kStages * 8 + 127) / 128 * 128;
    static constexpr size_t kSmem = kBarBytes + (size_t)kStages * kTile;
    static_assert(kBarBytes >= (size_t)kStages * 8, "mbarrier area too small");
    static_assert(kTile % 16 == 0 && kTile < (1 << 20), "bulk tile: 16-byte multiple, below the tx limit");
    static_assert(kSmem <= 227 * 1024, "bulk copy shared memory above the per-block limit");
};

template <int NSEG, int NOUT, int KIND>
__global__ void __launch_bounds__(kBulkThreads)
copy_bulk_kernel(const __grid_constant__ CopyParams<NSEG, NOUT> p)
{
    constexpr int kBulkStages = BulkShape<KIND>::kStages;
    constexpr int kBulkTile = BulkShape<KIND>::kTile;
    extern __shared__ __align__(128) unsigned char smem[];
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    if (threadIdx.x != 0) return;
    const uint64_t first = blockIdx.x, step = gridDim.x;
    if (first >= p.total_tiles) return;
    const uint64_t n = (p.total_tiles - first + step - 1) / step;   // tiles of this block
    const uint32_t bar0 = smem_addr(smem);
    const uint32_t buf0 = smem_addr(smem + BulkShape<KIND>::kBarBytes);
    for (int k = 0; k < kBulkStages; ++k) mbar_init(bar0 + 8 * k, 1);
    mbar_init_fence();
    const uint64_t pol = policy_evict_first();

    auto issue_load = [&](uint64_t i) {
        const uint64_t tile = first + i * step;
        const CopySeg &sg = p.seg[find_seg<KIND == kSplit>(p, tile)];
        const uint64_t t0 = (tile - sg.tile_begin) * p.tile_bytes;
        const uint32_t nb = (uint32_t)(sg.bytes - t0 < p.tile_bytes ? sg.bytes - t0 : p.tile_bytes);
        const int k = (int)(i % kBulkStages);
        if (DT_IN_BOUNDS(span_in(sg.src + t0, nb, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyBulk,
                         (int)(&sg - p.seg), sg.src + t0, sg.src_lo)) {
            mbar_expect_tx(bar0 + 8 * k, nb);
            bulk_load(buf0 + k * kBulkTile, sg.src + t0, nb, bar0 + 8 * k);
        } else {
            mbar_expect_tx(bar0 + 8 * k, 0);   // recorded and skipped: the stage completes empty
        }
    };

    const uint64_t pre = n < (uint64_t)kBulkStages ? n : (uint64_t)kBulkStages;
    for (uint64_t i = 0; i < pre; ++i) issue_load(i);
    uint64_t issued = pre;

    for (uint64_t i = 0; i < n; ++i) {
        const int k = (int)(i % kBulkStages);
        if (!mbar_wait_bounded(bar0 + 8 * k, (uint32_t)((i / kBulkStages) & 1), p.sink.timeout_ns)) {
            record_error(p.sink, DT_ERR_TIMEOUT, -1, (int)(first + i * step), 0);
            for (uint64_t j = i + 1; j < issued; ++j)   // let the other loads land (bounded)
                mbar_wait_bounded(bar0 + 8 * (int)(j % kBulkStages),
                                  (uint32_t)((j / kBulkStages) & 1), p.sink.timeout_ns);
            break;
        }
        fence_async_shared();
        const uint64_t tile = first + i * step;
        const CopySeg &sg = p.seg[find_seg<KIND == kSplit>(p, tile)];
        const uint64_t t0 = (tile - sg.tile_begin) * p.tile_bytes;
        const uint32_t nb = (uint32_t)(sg.bytes - t0 < p.tile_bytes ? sg.bytes - t0 : p.tile_bytes);
        for (int d = 0; d < sg.dst_count; ++d) {
            const int q = sg.dst_first + d;
            unsigned char *to = static_cast<unsigned char *>(p.out[q]) + sg.dst_off + t0;
            if (DT_IN_BOUNDS(span_in(to, nb, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsCopyBulk, kMaxSeg + q,
                             to, p.out_lo[q]))
                bulk_store_hint(to, buf0 + k * kBulkTile, nb, pol);
        }
        bulk_commit();
        // refill the stage of tile i-1 once its stores have read it
        if (i >= 1 && issued < n) {
            bulk_wait_read<1>();
            issue_load(issued);
            ++issued;
        }
    }
    bulk_wait_all();
    DT_TL_END_THREAD(DT_TL_COPY_BULK);
}

// Any alignment: the destination is cut into tiles of kShiftChunks 16-byte
// chunks.  Its bytes up to its first 16-byte boundary and after its last one
// go byte by byte; in between, every chunk is one aligned 16-byte store.  The
// chunk's source bytes start `sh` bytes into an aligned source vector and end
// in the next one: lane L of a warp loads aligned source vector c (c its
// chunk), takes vector c + 1 from lane L + 1 (lane 31 loads it), and
// funnel-shifts the pair by sh bytes.  A segment whose destinations share
// their offset past a boundary is shifted once and stored to each of them;
// otherwise each destination takes its own pass.  The first and last vectors
// read may hold bytes just outside the source range (never more than the
// rest of the 16-byte block that holds a source byte); those bytes are
// discarded.
constexpr uint64_t kShiftChunks = 512;                 // 8 KiB of destination per tile
constexpr uint64_t kShiftTile = kShiftChunks * 16;

// Tiles of one (segment, destination) pair: enough for its bytes, at least one.
__host__ __device__ __forceinline__ uint64_t shift_tiles(uint64_t bytes)
{
    const uint64_t t = (bytes + kShiftTile - 1) / kShiftTile;
    return t ? t : 1;
}

template <int NSEG, int NOUT>
__global__ void __launch_bounds__(kThreads)
copy_shift_kernel(const __grid_constant__ CopyParams<NSEG, NOUT> p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const CopySeg &sg = p.seg[find_seg<false>(p, tile)];
        const uint64_t tpp = shift_tiles(sg.bytes);
        const uint64_t idx = tile - sg.tile_begin;
        // one pass for all destinations, or tiles of one destination at a time
        const int k0 = sg.one_pass ? 0 : (int)(idx / tpp);
        const int nk = sg.one_pass ? sg.dst_count : 1;
        const uint64_t t = sg.one_pass ? idx : idx - (uint64_t)k0 * tpp;
        unsigned char *const *outs = reinterpret_cast<unsigned char *const *>(p.out) + sg.dst_first + k0;
        const unsigned char *S = sg.src;
        const uint64_t n = sg.bytes;
        uint64_t dh = (16 - ((reinterpret_cast<uintptr_t>(outs[0]) + sg.dst_off) & 15)) & 15;
        if (dh > n) dh = n;                                // bytes before the boundary
        const uint64_t nch = (n - dh) / 16;
        for (int k = 0; k < nk; ++k) {
            unsigned char *D = outs[k] + sg.dst_off;
            const int q = sg.dst_first + k0 + k;   // for the bounds checks
            (void)q;
            for (uint64_t b = threadIdx.x; t == 0 && b < dh; b += kThreads)
                if (DT_IN_BOUNDS(span_in(S + b, 1, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyShift,
                                 (int)(&sg - p.seg), S + b, sg.src_lo) &&
                    DT_IN_BOUNDS(span_in(D + b, 1, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsCopyShift,
                                 kMaxSeg + q, D + b, p.out_lo[q]))
                    D[b] = S[b];
            for (uint64_t b = dh + nch * 16 + threadIdx.x; t == tpp - 1 && b < n; b += kThreads)
                if (DT_IN_BOUNDS(span_in(S + b, 1, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyShift,
                                 (int)(&sg - p.seg), S + b, sg.src_lo) &&
                    DT_IN_BOUNDS(span_in(D + b, 1, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsCopyShift,
                                 kMaxSeg + q, D + b, p.out_lo[q]))
                    D[b] = S[b];
        }
        const uint64_t c0 = t * kShiftChunks;
        const uint64_t c1 = c0 + kShiftChunks < nch ? c0 + kShiftChunks : nch;
        if (c0 >= c1) continue;
        const unsigned char *sp = S + dh;                  // source of chunk 0
        const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(sp) & 15);
        const uint4 *A = reinterpret_cast<const uint4 *>(sp - sh);    // aligned source vectors
        // warp w takes chunks [base, base + 32); the loop bound is the same
        // for every lane, so the whole warp reaches each shuffle
        for (uint64_t base = c0 + (uint64_t)warp * 32; base < c1; base += kThreads) {
            const uint64_t c = base + lane;
            // vector c is read for chunk c (c < c1) and, when sh > 0, for
            // chunk c - 1 (c <= c1): both hold bytes of the source
            uint4 w = make_uint4(0, 0, 0, 0);
            if ((c < c1 || (sh && c == c1)) &&
                DT_IN_BOUNDS(vector_touches(A + c, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyShift,
                             (int)(&sg - p.seg), A + c, sg.src_lo))
                w = __ldcs(A + c);
            uint4 nx = shfl_down_uint4(w);
            if (lane == 31 && sh && c < c1 &&
                DT_IN_BOUNDS(vector_touches(A + c + 1, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyShift,
                             (int)(&sg - p.seg), A + c + 1, sg.src_lo))
                nx = __ldcs(A + c + 1);
            if (c < c1) {
                const uint4 v = sh ? shift_pair(w, nx, sh) : w;
                for (int k = 0; k < nk; ++k) {
                    uint4 *to = reinterpret_cast<uint4 *>(outs[k] + sg.dst_off + dh) + c;
                    const int q = sg.dst_first + k0 + k;   // for the bounds checks
                    (void)q;
                    if (DT_IN_BOUNDS(span_in(to, 16, p.out_lo[q], p.out_hi[q]), p.sink, kBoundsCopyShift,
                                     kMaxSeg + q, to, p.out_lo[q]))
                        __stcs(to, v);
                }
            }
        }
    }
    DT_TL_END_BLOCK(DT_TL_COPY_SHIFT);
}

// Small aligned launches: plain 16-byte loads and stores, two vectors per
// thread over 8 KiB tiles, up to 8 blocks per resident slot.  For small, mostly
// L2-resident launches the bulk-copy path's fixed costs (barrier set-up, one
// issuing thread per block, a load then a store per tile) dominate; measured
// on GB300 over 4 KiB .. 16 MiB per rank, the register path was up to 2.4x
// faster for gathers of at most 1 MiB of source whose stores total at most
// 4 MiB (slower past 16 MiB of stores, and a 2 MiB P=2 gather lost 12%) and
// for single-destination copies of up to 1 MiB, or up to 16 MiB
// when segments average 64 KiB or more (a P=16 AllToAll of 1 MiB per rank
// 8.9 -> 4.5 us).
constexpr uint64_t kSmallTile = 8192;

bool use_small_copy(uint64_t src_bytes, int nseg, int max_dst)
{
    if (max_dst > 1) return src_bytes <= (1ull << 20) && src_bytes * (uint64_t)max_dst <= (4ull << 20);
    if (src_bytes <= (1ull << 20)) return true;
    return src_bytes <= (16ull << 20) && src_bytes / (uint64_t)nseg >= (64ull << 10);
}

template <int NSEG, int NOUT, bool kDivide>
__global__ void __launch_bounds__(kThreads)
copy_vec_kernel(const __grid_constant__ CopyParams<NSEG, NOUT> p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const CopySeg &sg = p.seg[find_seg<kDivide>(p, tile)];
        const uint64_t t0 = (tile - sg.tile_begin) * p.tile_bytes;
        const uint64_t nv = (sg.bytes - t0 < p.tile_bytes ? sg.bytes - t0 : p.tile_bytes) / 16;
        const uint4 *src = reinterpret_cast<const uint4 *>(sg.src + t0);
        uint4 x[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint64_t v = threadIdx.x + (uint64_t)u * kThreads;
            if (v < nv && DT_IN_BOUNDS(span_in(src + v, 16, sg.src_lo, sg.src_hi), p.sink, kBoundsCopyVec,
                                       (int)(&sg - p.seg), src + v, sg.src_lo))
                x[u] = __ldcs(src + v);
        }
        for (int k = 0; k < sg.dst_count; ++k) {
            const int q = sg.dst_first + k;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(p.out[q]) + sg.dst_off + t0);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint64_t v = threadIdx.x + (uint64_t)u * kThreads;
                if (v < nv && DT_IN_BOUNDS(span_in(dst + v, 16, p.out_lo[q], p.out_hi[q]), p.sink,
                                           kBoundsCopyVec, kMaxSeg + q, dst + v, p.out_lo[q]))
                    __stcs(dst + v, x[u]);
            }
        }
    }
    DT_TL_END_BLOCK(DT_TL_COPY_VEC);
}

template <int NSEG, int NOUT, int KIND>
cudaError_t launch_bulk(const CopyParams<NSEG, NOUT> &p, int device, cudaStream_t s)
{
    using Shape = BulkShape<KIND>;
    void (*fn)(CopyParams<NSEG, NOUT>) = copy_bulk_kernel<NSEG, NOUT, KIND>;
    // The shared-memory opt-in is an attribute of the function on the current
    // device: set it once per device (bit `device` of this instantiation's mask;
    // setting it twice from racing threads is harmless).
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = device >= 0 && device < 64 ? 1ull << device : 0;
    if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Shape::kSmem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit, std::memory_order_release);
    }
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kBulkThreads, device,
                                    &resident, Shape::kSmem);
    if (e != cudaSuccess) return e;
    const uint64_t gx = bulk_grid<KIND>(p.total_tiles, resident);
    return launch_kernel(fn, dim3((unsigned)gx), dim3(kBulkThreads), Shape::kSmem, s, false, p);
}

// Tiles of tile_bytes covering the used segments; records each segment's first tile.
template <int NSEG, int NOUT>
uint64_t cut_tiles(CopyParams<NSEG, NOUT> &p, uint64_t tile_bytes)
{
    p.tile_bytes = tile_bytes;
    uint64_t tiles = 0;
    bool equal = true;
    const uint64_t first = (p.seg[0].bytes + tile_bytes - 1) / tile_bytes;
    for (int i = 0; i < p.nseg; ++i) {
        p.seg[i].tile_begin = tiles;
        const uint64_t t = (p.seg[i].bytes + tile_bytes - 1) / tile_bytes;
        equal = equal && t == first;
        tiles += t;
    }
    p.total_tiles = tiles;
    // Equal segments are found by a division from 8 segments on (AllToAlls of
    // 8 and 16 ranks at 4-256 KiB per rank 1.22-1.45x, 1 MiB 1.18-1.24x;
    // 8- and 16-rank gathers of up to 256 KiB 1.02-1.12x); with fewer the
    // search is as short as the division (2-rank gathers lost 3-4%).
    p.seg_tiles = equal && p.nseg >= 8 && first > 0 && tiles < (1ull << 32) ? (uint32_t)first : 0u;
    return tiles;
}

template <int NSEG, int NOUT>
cudaError_t launch_n(const CopySeg *segs, int nseg, void *const *out, const uint64_t *out_bytes,
                     int nout, bool vec, const ErrorSink &sink, int device, cudaStream_t s)
{
    CopyParams<NSEG, NOUT> p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < nout && r < NOUT; ++r) {
        p.out[r] = out[r];
#ifdef DT_BOUNDS
        p.out_lo[r] = reinterpret_cast<uint64_t>(out[r]);
        p.out_hi[r] = trimmed_end(p.out_lo[r], out_bytes[r]);
#endif
    }
    (void)out_bytes;
    p.sink = sink;
    int max_dst = 0;                    // most destinations of any segment
    int used = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].bytes == 0 || segs[i].dst_count == 0) continue;
        p.seg[used] = segs[i];
        p.seg[used].head = p.seg[used].tail = 0;
        ++used;
        if (segs[i].dst_count > max_dst) max_dst = segs[i].dst_count;
    }
    if (used == 0) return cudaSuccess;   // nothing to move
    p.nseg = used;

    if (!vec) {
        // Does every segment's source lie as far past a 16-byte boundary as
        // each of its destinations?  Then the aligned middle of every segment
        // takes the fast paths below and the edges go byte by byte.
        bool same = true;
        for (int i = 0; i < p.nseg && same; ++i) {
            const CopySeg &sg = p.seg[i];
            const uintptr_t m = reinterpret_cast<uintptr_t>(sg.src) & 15;
            for (int k = 0; k < sg.dst_count && same; ++k)
                same = ((reinterpret_cast<uintptr_t>(p.out[sg.dst_first + k]) + sg.dst_off) & 15) == m;
        }
        if (!same) {
            // otherwise the source is shifted into place: once for all of a
            // segment's destinations when they share their offset past a
            // boundary, else once per destination
            uint64_t tiles = 0;
            for (int i = 0; i < p.nseg; ++i) {
                CopySeg &sg = p.seg[i];
                const uintptr_t m0 = (reinterpret_cast<uintptr_t>(p.out[sg.dst_first]) + sg.dst_off) & 15;
                bool one = true;
                for (int k = 1; k < sg.dst_count && one; ++k)
                    one = ((reinterpret_cast<uintptr_t>(p.out[sg.dst_first + k]) + sg.dst_off) & 15) == m0;
                sg.one_pass = one ? 1 : 0;
                sg.tile_begin = tiles;
                tiles += shift_tiles(sg.bytes) * (one ? 1 : (uint64_t)sg.dst_count);
            }
            p.total_tiles = tiles;
            p.seg_tiles = 0;             // segments of different tile counts: search
            p.tile_bytes = kShiftTile;
            void (*fn)(CopyParams<NSEG, NOUT>) = copy_shift_kernel<NSEG, NOUT>;
            int resident = 0;
            cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
            if (e != cudaSuccess) return e;
            const uint64_t cap = (uint64_t)resident * 4;
            const uint64_t gx = tiles < cap ? tiles : cap;
            return launch_kernel(fn, dim3((unsigned)gx), dim3(kThreads), 0, s, false, p);
        }
        for (int i = 0; i < p.nseg; ++i) {
            CopySeg &sg = p.seg[i];
            uint64_t h = (16 - (reinterpret_cast<uintptr_t>(sg.src) & 15)) & 15;
            if (h > sg.bytes) h = sg.bytes;
            const uint64_t body = (sg.bytes - h) & ~(uint64_t)15;
            sg.head = (uint8_t)h;
            sg.tail = (uint8_t)(sg.bytes - h - body);
            sg.src += h;
            sg.dst_off += h;
            sg.bytes = body;
        }
        const uint64_t gx = (uint64_t)p.nseg;
        cudaError_t e = launch_kernel(copy_edge_kernel<NSEG, NOUT>, dim3((unsigned)gx), dim3(kThreads), 0,
                                      s, false, p);
        if (e != cudaSuccess) return e;
        // the middles: drop segments that are edges only
        int kept = 0;
        for (int i = 0; i < p.nseg; ++i)
            if (p.seg[i].bytes) p.seg[kept++] = p.seg[i];
        if (kept == 0) return cudaSuccess;
        p.nseg = kept;
        max_dst = 0;
        for (int i = 0; i < p.nseg; ++i)
            if (p.seg[i].dst_count > max_dst) max_dst = p.seg[i].dst_count;
    }
    uint64_t src_bytes = 0;
    for (int i = 0; i < p.nseg; ++i) src_bytes += p.seg[i].bytes;
    if (use_small_copy(src_bytes, p.nseg, max_dst)) {
        const uint64_t tiles = cut_tiles(p, kSmallTile);
        void (*fn)(CopyParams<NSEG, NOUT>) =
            p.seg_tiles ? copy_vec_kernel<NSEG, NOUT, true> : copy_vec_kernel<NSEG, NOUT, false>;
        int resident = 0;
        cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
        if (e != cudaSuccess) return e;
        const uint64_t cap = (uint64_t)resident * 8;
        const uint64_t gx = tiles < cap ? tiles : cap;
        return launch_kernel(fn, dim3((unsigned)gx), dim3(kThreads), 0, s, false, p);
    }
    // Wide tiles need enough of them to keep every SM busy to the end (at
    // least 4 per SM; at 2 per SM a 16 MiB-per-rank P=2 gather lost 17%), and
    // they stop paying at 16 destinations, where each tile carries 1.5 MiB of
    // stores and the last wave runs half empty.
    if (max_dst > 1 && max_dst <= 8) {
        const uint64_t sms = (uint64_t)sm_count(device);
        const uint64_t wide = cut_tiles(p, BulkShape<kWide>::kTile);
        if (wide >= 16 * sms) return launch_bulk<NSEG, NOUT, kWide>(p, device, s);
        // smaller gathers keep the 32 KiB x 6 shape below (a 2-rank gather of
        // 16 MiB shards lost 9% on the split shape)
        if (wide >= 4 * sms) {
            cut_tiles(p, BulkShape<kWideSplit>::kTile);
            return launch_bulk<NSEG, NOUT, kWideSplit>(p, device, s);
        }
    }
    if (NSEG > DT_MAX_RANKS) {
        const uint64_t tiles = cut_tiles(p, BulkShape<kStream>::kTile);
        // with a tile or less per SM, one block per SM spreads the copies
        // over every SM's copy engine (8 ranks, 256 KiB per rank: the split
        // shape lost 16%)
        if ((p.nseg <= 64 && 2 * src_bytes > l2_bytes(device)) || tiles <= (uint64_t)sm_count(device))
            return launch_bulk<NSEG, NOUT, kStream>(p, device, s);   // searches (see find_seg)
        return launch_bulk<NSEG, NOUT, kSplit>(p, device, s);
    }
    if (max_dst <= 8 && cut_tiles(p, BulkShape<kGatherSplit>::kTile) >= 3 * (uint64_t)sm_count(device))
        return launch_bulk<NSEG, NOUT, kGatherSplit>(p, device, s);
    cut_tiles(p, BulkShape<kGather>::kTile);
    return launch_bulk<NSEG, NOUT, kGather>(p, device, s);
}

}  // namespace

DT_TL_BINDER(bind_timeline_copy)

cudaError_t launch_copy(const CopySeg *segs, int nseg, void *const *out, const uint64_t *out_bytes,
                        int nout, bool vec,
                        const ErrorSink &sink, int device, cudaStream_t s)
{
    if (nout > DT_MAX_RANKS) {
        if (nseg > DT_MAX_RANKS || nout > kMaxSeg) return cudaErrorInvalidValue;
        return launch_n<DT_MAX_RANKS, kMaxSeg>(segs, nseg, out, out_bytes, nout, vec, sink, device, s);
    }
    if (nseg <= DT_MAX_RANKS)
        return launch_n<DT_MAX_RANKS, DT_MAX_RANKS>(segs, nseg, out, out_bytes, nout, vec, sink, device, s);
    if (nseg <= kMaxSeg)
        return launch_n<kMaxSeg, DT_MAX_RANKS>(segs, nseg, out, out_bytes, nout, vec, sink, device, s);
    return cudaErrorInvalidValue;
}

namespace {

// 2-D copy: a tile is rows_per_tile whole rows of one segment; warp w of the
// block copies rows w, w + 8, ... of the tile, its lanes striding over the
// row in 16-byte vectors (kVec) or bytes.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) copy2d_kernel(const __grid_constant__ Copy2dParams p)
{
    DT_TL_BEGIN();
    pdl_begin();
    DT_TL_WAITED();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const Copy2dSeg &sg = p.seg[find_seg<false>(p, tile)];
        const uint64_t r0 = (tile - sg.tile_begin) * sg.rows_per_tile;
        const uint64_t r1 = r0 + sg.rows_per_tile < sg.rows ? r0 + sg.rows_per_tile : sg.rows;
        unsigned char *dbase = static_cast<unsigned char *>(p.out[sg.dst]) + sg.dst_off;
        for (uint64_t row = r0 + warp; row < r1; row += kThreads / 32) {
            const unsigned char *src = sg.src + row * sg.src_pitch;
            unsigned char *dst = dbase + row * sg.dst_pitch;
            if (kVec) {
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                for (uint64_t v = lane; v < sg.row_bytes / 16; v += 32)
                    if (DT_IN_BOUNDS(span_in(s4 + v, 16, sg.src_lo, sg.src_hi), p.sink, kBoundsCopy2d,
                                     (int)(&sg - p.seg), s4 + v, sg.src_lo) &&
                        DT_IN_BOUNDS(span_in(d4 + v, 16, p.out_lo[sg.dst], p.out_hi[sg.dst]), p.sink,
                                     kBoundsCopy2d, kMaxSeg + sg.dst, d4 + v, p.out_lo[sg.dst]))
                        __stcs(d4 + v, __ldcs(s4 + v));
            } else {
                for (uint64_t b = lane; b < sg.row_bytes; b += 32)
                    if (DT_IN_BOUNDS(span_in(src + b, 1, sg.src_lo, sg.src_hi), p.sink, kBoundsCopy2d,
                                     (int)(&sg - p.seg), src + b, sg.src_lo) &&
                        DT_IN_BOUNDS(span_in(dst + b, 1, p.out_lo[sg.dst], p.out_hi[sg.dst]), p.sink,
                                     kBoundsCopy2d, kMaxSeg + sg.dst, dst + b, p.out_lo[sg.dst]))
                        dst[b] = src[b];
            }
        }
    }
    DT_TL_END_BLOCK(DT_TL_COPY_2D);
}

}  // namespace

cudaError_t launch_copy2d(const Copy2dSeg *segs, int nseg, void *const *out, const uint64_t *out_bytes,
                          bool vec, const ErrorSink &sink, int device, cudaStream_t s)
{
    if (nseg > DT_MAX_RANKS * DT_MAX_RANKS) return cudaErrorInvalidValue;
    Copy2dParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < DT_MAX_RANKS; ++r) {
        p.out[r] = out[r];
#ifdef DT_BOUNDS
        p.out_lo[r] = reinterpret_cast<uint64_t>(out[r]);
        p.out_hi[r] = trimmed_end(p.out_lo[r], out_bytes[r]);
#endif
    }
#ifdef DT_BOUNDS
    p.sink = sink;
#endif
    (void)out_bytes;
    (void)sink;
    uint64_t tiles = 0;
    int used = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].rows == 0 || segs[i].row_bytes == 0) continue;
        p.seg[used] = segs[i];
        uint64_t rpt = 16384 / segs[i].row_bytes;   // about 16 KiB per tile
        if (rpt < 1) rpt = 1;
        p.seg[used].rows_per_tile = rpt;
        p.seg[used].tile_begin = tiles;
        tiles += (segs[i].rows + rpt - 1) / rpt;
        ++used;
    }
    if (used == 0) return cudaSuccess;
    p.nseg = used;
    p.total_tiles = tiles;
    void (*fn)(Copy2dParams) = vec ? copy2d_kernel<true> : copy2d_kernel<false>;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;
    // many short blocks (up to 32 per resident slot, ~13 tiles each for the
    // 8-rank S(0) -> S(1) workload) let the hardware balance the SMs: 6.65 ->
    // 6.88 TB/s against one block per slot
    const uint64_t cap = (uint64_t)resident * 32;
    const uint64_t gx = tiles < cap ? tiles : cap;
    return launch_kernel(fn, dim3((unsigned)gx), dim3(kThreads), 0, s, false, p);
}

}  // namespace dt
