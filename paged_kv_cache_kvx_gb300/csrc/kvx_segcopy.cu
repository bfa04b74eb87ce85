// Segment copies whose addresses are computed on the fly, with no descriptor
// list in memory:
//   kvx_paged_writes -- the paged write of the TransferEngine API ("RDMA
//       point-to-point communication for LLM systems", API listing): page i
//       of a source page set {indices, stride, offset} goes to page i of a
//       destination page set, page_len bytes each.
//   kvx_seal_blocks  -- seal from template metadata (pegaflow PR #350, the
//       follow-up named after the stage breakdown): segment (b, l) moves from
//       the slab at its rebuilt offset to the receiver's dst_addr[b][l]; the
//       offset comes from the run arithmetic and the group carve, so no
//       per-segment local table is ever written.
//
// HBM-bound copies, one warp per batch of 32 segments (pages longer than 4 KiB
// count as several 4 KiB segments, so that batches stay small and many
// whatever the page size): lane i computes segment i's addresses and checks
// (coalesced metadata loads, the lanes' lookups in parallel), then the batch
// is moved by one of the two engines of kvx_ring.cuh:
//   - with a caller workspace, the SM's bulk-copy engine (k_seg_tma: four
//     warps per SM, each with a ring of 3 x 16 KiB shared-memory stages, the
//     batches claimed from a counter in the workspace);
//   - without one, or for pages under 2 KiB, registers (k_paged_writes /
//     k_seal_blocks below: 16-byte streaming vectors, several loads in flight
//     per lane), which measured faster for short segments.
#include "kvx_ring.cuh"

namespace kvx {
namespace {

using namespace ring;

constexpr int kThreads = 256;
constexpr int kMinBlocks = 3;                // resident blocks per SM (caps registers at 80)

// ---------------------------------------------------------------- paged

struct PagedArgs {
    uint64_t page_len;
    const uint8_t *src;
    uint64_t src_bytes;
    const uint32_t *src_idx;
    uint64_t src_stride, src_offset;
    uint8_t *dst;
    uint64_t dst_bytes;
    const uint32_t *dst_idx;
    uint64_t dst_stride, dst_offset;
    uint64_t n;        // pages
    uint64_t piece;    // bytes per unit of work (a page, or a 4 KiB part of one)
    uint64_t pieces;   // units per page
    uint32_t *status;
};

// Pages longer than this are cut into parts of this size, so that a handful
// of large pages still spreads over every warp of the grid.
constexpr uint64_t kPiece = 4 * 1024;

// Unit u = part u % pieces of page u / pieces: exact (128-bit) page
// addresses; a page outside its buffer is skipped (SPAN on the source side,
// BOUNDS on the destination side).
__device__ __forceinline__ Seg paged_seg(const PagedArgs &a, uint64_t u, uint32_t &bad) {
    const uint64_t i = u / a.pieces, part = u % a.pieces;
    const unsigned __int128 s = (unsigned __int128)a.src_offset + (unsigned __int128)a.src_idx[i] * a.src_stride;
    const unsigned __int128 d = (unsigned __int128)a.dst_offset + (unsigned __int128)a.dst_idx[i] * a.dst_stride;
    const bool ok_s = s + a.page_len <= a.src_bytes;
    const bool ok_d = d + a.page_len <= a.dst_bytes;
    if (!ok_s) bad |= KVX_S_SPAN;
    if (!ok_d) bad |= KVX_S_BOUNDS;
    if (!ok_s || !ok_d) return Seg{nullptr, nullptr, 0, false};
    const uint64_t off = part * a.piece;
    const uint64_t len = a.page_len - off < a.piece ? a.page_len - off : a.piece;
    return Seg{a.src + (uint64_t)s + off, a.dst + (uint64_t)d + off, len, true};
}

__global__ void __launch_bounds__(kThreads, kMinBlocks) k_paged_writes(const __grid_constant__ PagedArgs a) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t units = a.n * a.pieces;
    uint32_t bad = 0;
    for (uint64_t u0 = warp * 32; u0 < units; u0 += nwarps * 32) {
        const uint64_t u = u0 + lane;
        const Seg sg = u < units ? paged_seg(a, u, bad) : Seg{nullptr, nullptr, 0, false};
        warp_copy(sg, lane);
    }
    warp_raise(a.status, bad, lane);
}

// ----------------------------------------------------------------- seal

struct SealArgs {
    const uint32_t *lane_first, *run_block;
    const uint64_t *run_base;
    const int64_t *run_stride;
    const uint32_t *run_group;
    uint64_t run_cap;
    const kvx_group *groups;
    uint64_t group_cap;
    const uint64_t *counts;
    uint32_t B, L;
    const uint32_t *seg_len;
    const uint8_t *slab;
    uint64_t slab_bytes;
    const uint64_t *dst_addr;
    uint8_t *dst;
    uint64_t dst_bytes;
    uint32_t *status;
};

// Segment s = b*L + l: its rebuilt slab offset (the rebuild's arithmetic and
// checks: the run of lane l covering b by binary search, remote(b) from the
// run's base and stride, then local = G.local + (remote(b) - G.base) for a
// dense group or G.local + i*G.chunk + (remote(b) - (G.base + i*G.stride))
// otherwise, exactly; group index valid, b in the group's block range, the
// segment inside block i's slice of the carve, the carve inside the slab)
// and its destination range.
__device__ __forceinline__ Seg seal_seg(const SealArgs &a, uint64_t s, uint64_t ngroups, uint32_t &bad) {
    const uint32_t b = (uint32_t)(s / a.L), l = (uint32_t)(s % a.L);
    const uint64_t len = a.seg_len[l];
    const uint64_t lo = a.lane_first[l], hi = a.lane_first[l + 1];
    bool ok = false;
    uint64_t loc = 0;
    if (lo < hi && hi <= a.run_cap) {
        uint64_t x = lo, z = hi;  // last run with run_block <= b, in [x, z)
        while (z - x > 1) {
            const uint64_t m = (x + z) >> 1;
            if (a.run_block[m] <= b) x = m; else z = m;
        }
        const uint32_t gi = a.run_group[x];
        const uint32_t rb = a.run_block[x];
        if (gi < ngroups && rb <= b) {
            const kvx_group G = a.groups[gi];
            const __int128 g_local = (__int128)G.local, g_chunk = (__int128)G.chunk;
            if (b >= G.block && b - G.block < G.count &&
                g_local + (__int128)G.count * g_chunk <= (__int128)a.slab_bytes) {
                const uint64_t remote = a.run_base[x] + (uint64_t)(b - rb) * (uint64_t)a.run_stride[x];
                const __int128 i = (__int128)(b - G.block);
                const __int128 slice = g_local + i * g_chunk;
                const __int128 v = G.dense ? g_local + ((__int128)remote - (__int128)G.base)
                                           : slice + ((__int128)remote - ((__int128)G.base + i * (__int128)G.stride));
                if (v >= slice && v + (__int128)len <= slice + g_chunk) {
                    ok = true;
                    loc = (uint64_t)v;
                }
            }
        }
    }
    const uint64_t d = a.dst_addr[s];
    if (ok && !(d <= a.dst_bytes && len <= a.dst_bytes - d)) ok = false;
    if (!ok) {
        bad |= KVX_S_BOUNDS;
        return Seg{nullptr, nullptr, 0, false};
    }
    return Seg{a.slab + loc, a.dst + d, len, true};
}

__global__ void __launch_bounds__(kThreads, kMinBlocks) k_seal_blocks(const __grid_constant__ SealArgs a) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t n = (uint64_t)a.B * a.L;
    const uint64_t ngroups = a.counts[0] < a.group_cap ? a.counts[0] : a.group_cap;
    uint32_t bad = 0;
    for (uint64_t s0 = warp * 32; s0 < n; s0 += nwarps * 32) {
        const uint64_t s = s0 + lane;
        const Seg sg = s < n ? seal_seg(a, s, ngroups, bad) : Seg{nullptr, nullptr, 0, false};
        warp_copy(sg, lane);
    }
    warp_raise(a.status, bad, lane);
}

constexpr uint64_t kBulkMinLen = 2048;  // pages shorter than this take the register path

struct PagedGen {
    PagedArgs a;
    __device__ uint64_t units() const { return a.n * a.pieces; }
    __device__ Seg get(uint64_t u, uint32_t &bad) const { return paged_seg(a, u, bad); }
    __device__ uint32_t *status() const { return a.status; }
};

struct SealGen {
    SealArgs a;
    __device__ uint64_t units() const { return (uint64_t)a.B * a.L; }
    __device__ Seg get(uint64_t u, uint32_t &bad) const {
        const uint64_t ngroups = a.counts[0] < a.group_cap ? a.counts[0] : a.group_cap;
        return seal_seg(a, u, ngroups, bad);
    }
    __device__ uint32_t *status() const { return a.status; }
};

// The ring path: the claim counter in ws is cleared, then one launch.
template <class Gen>
kvx_status launch_bulk(const Gen &g, void *ws, cudaStream_t s) {
    SegCtl *ctl = static_cast<SegCtl *>(ws);
    if (cudaMemsetAsync(ctl, 0, sizeof(SegCtl), s) != cudaSuccess) return KVX_ECUDA;
    return launch_ring(g, ctl, s);
}

// Resident blocks of a kernel over the whole device (cached per device).
template <class K>
uint32_t resident_blocks(K kernel, int *cache) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return (uint32_t)cache[dev];
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int n = per_sm * sm_count();
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return (uint32_t)n;
}

// Enough blocks for one batch of 32 segments per warp, at most one full wave.
uint32_t grid_for(uint64_t n, uint32_t resident) {
    const uint64_t batches = ceil_div(n, 32);
    const uint64_t want = ceil_div(batches, kThreads / 32);
    return (uint32_t)(want < resident ? want : resident);
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" size_t kvx_segcopy_workspace_size(void) { return 256; }

extern "C" kvx_status kvx_paged_writes(uint64_t page_len, const uint8_t *src, uint64_t src_bytes,
                                       const uint32_t *src_indices, uint64_t src_stride,
                                       uint64_t src_offset, uint8_t *dst, uint64_t dst_bytes,
                                       const uint32_t *dst_indices, uint64_t dst_stride,
                                       uint64_t dst_offset, uint64_t num_pages, uint32_t *status,
                                       void *ws, size_t ws_bytes, void *stream) {
    if (!status) return KVX_EINVAL;
    if (ws && ws_bytes < kvx_segcopy_workspace_size()) return KVX_EINVAL;
    if (num_pages == 0) return KVX_OK;
    if (!src_indices || !dst_indices || (src_bytes && !src) || (dst_bytes && !dst)) return KVX_EINVAL;
    static int cache[64] = {};
    const uint64_t piece = page_len > kPiece ? kPiece : (page_len ? page_len : 1);
    const uint64_t pieces = page_len > kPiece ? ceil_div(page_len, kPiece) : 1;
    if (num_pages > UINT64_MAX / pieces) return KVX_EINVAL;
    PagedArgs a{page_len, src, src_bytes, src_indices, src_stride, src_offset, dst, dst_bytes,
                dst_indices, dst_stride, dst_offset, num_pages, piece, pieces, status};
    cudaStream_t s = as_stream(stream);
    // the bulk engine wins from 2 KiB pages on; below, batches are too small
    // to cover its per-batch latency and the register path is faster
    if (ws && page_len >= kBulkMinLen) return launch_bulk(PagedGen{a}, ws, s);
    const uint32_t grid = grid_for(num_pages * pieces, resident_blocks(k_paged_writes, cache));
    k_paged_writes<<<grid, kThreads, 0, s>>>(a);
    KVX_LAUNCHED();
    return KVX_OK;
}

extern "C" kvx_status kvx_seal_blocks(const uint32_t *lane_first, const uint32_t *run_block,
                                      const uint64_t *run_base, const int64_t *run_stride,
                                      const uint32_t *run_group, uint64_t run_capacity, const kvx_group *groups,
                                      uint64_t group_capacity, const uint64_t *counts, uint32_t B,
                                      uint32_t L, const uint32_t *seg_len, const uint8_t *slab,
                                      uint64_t slab_bytes, const uint64_t *dst_addr, uint8_t *dst,
                                      uint64_t dst_bytes, uint32_t *status, void *ws,
                                      size_t ws_bytes, void *stream) {
    if (!lane_first || !counts || !status) return KVX_EINVAL;
    if (ws && ws_bytes < kvx_segcopy_workspace_size()) return KVX_EINVAL;
    if ((uint64_t)B * L == 0) return KVX_OK;
    if (!run_block || !run_base || !run_stride || !run_group || !groups || !seg_len || !dst_addr ||
        (slab_bytes && !slab) || (dst_bytes && !dst))
        return KVX_EINVAL;
    static int cache[64] = {};
    SealArgs a{lane_first, run_block, run_base, run_stride, run_group, run_capacity, groups, group_capacity,
               counts, B, L, seg_len, slab, slab_bytes, dst_addr, dst, dst_bytes, status};
    cudaStream_t s = as_stream(stream);
    if (ws) return launch_bulk(SealGen{a}, ws, s);
    const uint32_t grid = grid_for((uint64_t)B * L, resident_blocks(k_seal_blocks, cache));
    k_seal_blocks<<<grid, kThreads, 0, s>>>(a);
    KVX_LAUNCHED();
    return KVX_OK;
}
