// Byte-copy kernel behind AllGather (equal and uneven shards) and AllToAll.
//
// Both collectives of the DTorch ThreadGroup interface (§2.1) are pure data
// movement: AllGather writes every rank's shard into every rank's output at
// the shard's row offset, AllToAll sends chunk j of rank i to rank j.  The
// host turns a call into a list of segments (source range -> one or more
// destinations at one offset); this kernel moves them in one launch.  Each
// segment is cut into 16 KiB tiles; a resident grid strides over the tiles
// of all segments.  A block loads its tile once into registers (four 16-byte
// vectors per thread, all in flight together) and stores it to every
// destination of the segment, so a shard is read from HBM once however many
// ranks receive it.
#include "dt_internal.h"

namespace dt {
namespace {

constexpr int kVecPerThread = kCopyTileBytes / (16 * kThreads);   // 4

template <int NSEG>
__device__ __forceinline__ int find_seg(const CopyParams<NSEG> &p, uint64_t tile)
{
    int lo = 0, hi = p.nseg - 1;      // last segment with tile_begin <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile_begin <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int NSEG>
__global__ void __launch_bounds__(kThreads)
copy_vec_kernel(const __grid_constant__ CopyParams<NSEG> p)
{
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const CopySeg &sg = p.seg[find_seg(p, tile)];
        const uint64_t t0 = (tile - sg.tile_begin) * p.tile_bytes;   // byte offset in segment
        const uint64_t nv = (sg.bytes - t0 < p.tile_bytes ? sg.bytes - t0 : p.tile_bytes) / 16;
        const uint4 *src = reinterpret_cast<const uint4 *>(sg.src + t0);
        uint4 x[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const uint64_t v = (uint64_t)u * kThreads + threadIdx.x;
            if (v < nv) x[u] = __ldcg(src + v);
        }
        for (int k = 0; k < sg.dst_count; ++k) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                static_cast<unsigned char *>(p.out[sg.dst_first + k]) + sg.dst_off + t0);
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) {
                const uint64_t v = (uint64_t)u * kThreads + threadIdx.x;
                if (v < nv) __stcg(dst + v, x[u]);
            }
        }
    }
}

// Any alignment: byte by byte, same tiling.
template <int NSEG>
__global__ void __launch_bounds__(kThreads)
copy_byte_kernel(const __grid_constant__ CopyParams<NSEG> p)
{
    for (uint64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const CopySeg &sg = p.seg[find_seg(p, tile)];
        const uint64_t t0 = (tile - sg.tile_begin) * p.tile_bytes;
        const uint64_t nb = sg.bytes - t0 < p.tile_bytes ? sg.bytes - t0 : p.tile_bytes;
        for (uint64_t b = threadIdx.x; b < nb; b += kThreads) {
            const unsigned char c = sg.src[t0 + b];
            for (int k = 0; k < sg.dst_count; ++k)
                static_cast<unsigned char *>(p.out[sg.dst_first + k])[sg.dst_off + t0 + b] = c;
        }
    }
}

template <int NSEG>
cudaError_t launch_n(const CopySeg *segs, int nseg, void *const *out, bool vec, int device,
                     cudaStream_t s)
{
    CopyParams<NSEG> p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < DT_MAX_RANKS; ++r) p.out[r] = out[r];
    p.tile_bytes = vec ? kCopyTileBytes : 4096;
    uint64_t tiles = 0;
    int used = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].bytes == 0 || segs[i].dst_count == 0) continue;
        p.seg[used] = segs[i];
        p.seg[used].tile_begin = tiles;
        tiles += (segs[i].bytes + p.tile_bytes - 1) / p.tile_bytes;
        ++used;
    }
    if (used == 0) return cudaSuccess;   // nothing to move
    p.nseg = used;
    p.total_tiles = tiles;

    void (*fn)(CopyParams<NSEG>) = vec ? copy_vec_kernel<NSEG> : copy_byte_kernel<NSEG>;
    int resident = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void *>(fn), kThreads, device, &resident);
    if (e != cudaSuccess) return e;
    const uint64_t gx = tiles < (uint64_t)resident ? tiles : (uint64_t)resident;
    count_launch();
    fn<<<(unsigned)gx, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_copy(const CopySeg *segs, int nseg, void *const *out, bool vec, int device,
                        cudaStream_t s)
{
    if (nseg <= DT_MAX_RANKS) return launch_n<DT_MAX_RANKS>(segs, nseg, out, vec, device, s);
    if (nseg <= kMaxSeg) return launch_n<kMaxSeg>(segs, nseg, out, vec, device, s);
    return cudaErrorInvalidValue;
}

}  // namespace dt
