// Segment copies whose addresses are computed on the fly, with no descriptor
// list in memory:
//   kvx_paged_writes -- the paged write of the TransferEngine API ("RDMA
//       point-to-point communication for LLM systems", API listing): page i
//       of a source page set {indices, stride, offset} goes to page i of a
//       destination page set, page_len bytes each.
//   kvx_seal_blocks  -- seal from template metadata (pegaflow PR #350, the
//       follow-up named after the stage breakdown): segment (b, l) moves from
//       the slab at its rebuilt offset to the receiver's dst_addr[b][l]; the
//       offset comes from the group carve and run_off, so no per-segment
//       local table is ever written.
//
// HBM-bound copies.  One warp takes 32 segments at a time (pages longer than
// 4 KiB count as several 4 KiB segments, so that the batches of a copy stay
// small and many against the grid's warps whatever the page size): lane i computes
// segment i's addresses and checks (coalesced metadata loads, the lanes'
// lookups in parallel), then the whole warp moves the 32 segments.  Aligned
// segments of up to 64 KiB form one index space of 16-byte vectors, walked
// four vectors per lane per step (loads first, then stores), so short and
// long segments alike keep several loads in flight per lane and every
// access of a warp instruction stays inside one or two segments (coalesced).
// Longer aligned segments go one at a time in 4-vector steps; unaligned ones
// byte by byte.  Streaming cache hints: neither side is read again.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kThreads = 256;
constexpr int kMinBlocks = 3;                // resident blocks per SM (caps registers at 80)
constexpr int kFlatU = 4;                    // vectors per lane per flat step
constexpr int kLongU = 4;                    // vectors per lane per long-segment step
constexpr uint64_t kFlatMaxLen = 64 * 1024;  // longer segments go one at a time
constexpr unsigned kFull = 0xFFFFFFFFu;

struct Seg {
    const uint8_t *src;
    uint8_t *dst;
    uint64_t len;
    bool ok;
};

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(uint8_t *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ const uint8_t *shfl_ptr(const uint8_t *p, int src) {
    return reinterpret_cast<const uint8_t *>(
        __shfl_sync(kFull, reinterpret_cast<unsigned long long>(p), src));
}
__device__ __forceinline__ uint8_t *shfl_ptr(uint8_t *p, int src) {
    return reinterpret_cast<uint8_t *>(__shfl_sync(kFull, reinterpret_cast<unsigned long long>(p), src));
}

// Moves the 32 segments of a warp (lane i holds segment i; !ok = skip).
__device__ void warp_copy(const Seg &sg, uint32_t lane) {
    const uintptr_t align = reinterpret_cast<uintptr_t>(sg.src) | reinterpret_cast<uintptr_t>(sg.dst) | sg.len;
    const bool vec = sg.ok && sg.len > 0 && (align & 15) == 0;
    const bool flat = vec && sg.len <= kFlatMaxLen;

    // 1. aligned segments up to 64 KiB: one index space of 16-byte vectors
    const uint32_t n16 = flat ? (uint32_t)(sg.len >> 4) : 0u;
    const uint32_t incl = warp_incl_sum(n16);
    const uint32_t excl = incl - n16;
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    // every lane the same length: the segment of vector k is k / n16
    const bool uniform = __all_sync(kFull, n16 == __shfl_sync(kFull, n16, 0)) && n16 > 0;
    for (uint32_t k0 = 0; k0 < total; k0 += 32 * kFlatU) {
        uint4 v[kFlatU];
        uint8_t *d[kFlatU];
#pragma unroll
        for (int u = 0; u < kFlatU; u++) {
            const uint32_t k = k0 + (uint32_t)u * 32 + lane;
            uint32_t i, e;
            if (uniform) {
                i = k / n16;
                e = i * n16;
                i &= 31;
            } else {  // the last segment whose first vector is <= k
                i = 0;
#pragma unroll
                for (uint32_t step = 16; step > 0; step >>= 1) {
                    const uint32_t x = __shfl_sync(kFull, excl, (i + step) & 31);
                    if (i + step < 32 && x <= k) i += step;
                }
                e = __shfl_sync(kFull, excl, i);
            }
            const uint8_t *s = shfl_ptr(sg.src, i);
            uint8_t *dd = shfl_ptr(sg.dst, i);
            const uint64_t off = (uint64_t)(k - e) * 16;
            d[u] = nullptr;
            if (k < total) {
                v[u] = ld_stream(s + off);
                d[u] = dd + off;
            }
        }
#pragma unroll
        for (int u = 0; u < kFlatU; u++)
            if (d[u]) st_stream(d[u], v[u]);
    }

    // 2. longer aligned segments, one at a time
    uint32_t mask = __ballot_sync(kFull, vec && !flat);
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1;
        const uint8_t *s = shfl_ptr(sg.src, i);
        uint8_t *dd = shfl_ptr(sg.dst, i);
        const uint64_t len = __shfl_sync(kFull, (unsigned long long)sg.len, i);
        for (uint64_t o0 = (uint64_t)lane * 16; o0 < len; o0 += 32 * 16 * kLongU) {
            uint4 v[kLongU];
#pragma unroll
            for (int u = 0; u < kLongU; u++) {
                const uint64_t o = o0 + (uint64_t)u * 32 * 16;
                if (o < len) v[u] = ld_stream(s + o);
            }
#pragma unroll
            for (int u = 0; u < kLongU; u++) {
                const uint64_t o = o0 + (uint64_t)u * 32 * 16;
                if (o < len) st_stream(dd + o, v[u]);
            }
        }
    }

    // 3. unaligned segments, byte by byte
    mask = __ballot_sync(kFull, sg.ok && sg.len > 0 && !vec);
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1;
        const uint8_t *s = shfl_ptr(sg.src, i);
        uint8_t *dd = shfl_ptr(sg.dst, i);
        const uint64_t len = __shfl_sync(kFull, (unsigned long long)sg.len, i);
        for (uint64_t o = lane; o < len; o += 32) dd[o] = s[o];
    }
}

__device__ __forceinline__ void warp_raise(uint32_t *status, uint32_t bits, uint32_t lane) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) bits |= __shfl_xor_sync(kFull, bits, d);
    if (lane == 0 && bits) atomicOr(status, bits);
}

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
    const uint32_t *lane_first, *run_block, *run_group;
    const uint64_t *run_off;
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
// checks: run of lane l covering b by binary search, group index valid, b in
// the group's block range, the segment inside block i's slice of the carve,
// the carve inside the slab) and its destination range.
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
        if (gi < ngroups && a.run_block[x] <= b) {
            const kvx_group G = a.groups[gi];
            const __int128 g_local = (__int128)G.local, g_chunk = (__int128)G.chunk;
            if (b >= G.block && b - G.block < G.count &&
                g_local + (__int128)G.count * g_chunk <= (__int128)a.slab_bytes) {
                const __int128 i = (__int128)(b - G.block);
                const __int128 step = G.dense ? (__int128)G.stride : g_chunk;
                const __int128 v = g_local + i * step + (__int128)a.run_off[x];
                const __int128 slice = g_local + i * g_chunk;
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

// ------------------------------------------------------- bulk-copy path

// The same copies through the SM's bulk-copy engine, as the descriptor-driven
// pack does, so no byte is staged in registers: four warps per SM, each
// driving its own ring of three 16 KiB shared-memory stages (cp.async.bulk
// global->shared completing on an mbarrier, then cp.async.bulk
// shared->global), 192 KiB of loads per SM in flight.  Four independent rings
// rather than one: a warp stalls while it claims a batch and resolves its
// addresses, and one ring per SM left the copy engine idle then (measured on
// GB300: 5745 GB/s for 4 KiB pages with one 3 x 64 KiB ring, 6773 with four).
// Warps claim batches of 32 segments from a counter in the caller's
// workspace and resolve the next batch's addresses while the current one
// copies.  A batch moves in rounds of at most 16 KiB per segment; each round's
// pieces are packed in lane order into stage groups of at most 16 KiB, and
// each lane issues the bulk copies of its own piece.  Unaligned segments are
// copied by the warp's registers on the spot.
constexpr uint32_t kStageBytes = 16 * 1024;
constexpr uint64_t kBulkMinLen = 2048;  // pages shorter than this take the register path
constexpr int kRing = 3;
constexpr int kRingWarps = 4;  // independent rings per SM, so one warp's stalls hide behind the others

struct SegCtl {
    uint32_t next;  // next unclaimed batch
};

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

template <class Gen>
__global__ void __launch_bounds__(32 * kRingWarps, 1) k_seg_tma(const __grid_constant__ Gen g, SegCtl *ctl) {
    extern __shared__ __align__(128) uint8_t ring_all[];
    __shared__ __align__(8) uint64_t bars_all[kRingWarps][kRing];
    __shared__ uint8_t *s_dst_all[kRingWarps][kRing][32];
    __shared__ uint32_t s_off_all[kRingWarps][kRing][32], s_len_all[kRingWarps][kRing][32];
    const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint8_t *ring = ring_all + (uint64_t)wid * kRing * kStageBytes;
    uint64_t *bars = bars_all[wid];
    auto &s_dst = s_dst_all[wid];
    auto &s_off = s_off_all[wid];
    auto &s_len = s_len_all[wid];
    const uint64_t units = g.units();
    const uint64_t nb = ceil_div(units, 32);
    if (lane == 0) {
        for (int k = 0; k < kRing; k++) mbar_init(&bars[k], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    uint32_t bad = 0;
    bool ok = true;
    uint32_t issued = 0, stored = 0;  // stage groups loaded / stored (warp-uniform)

    auto claim = [&](uint64_t &b, Seg &sg) {
        uint32_t x = 0;
        if (lane == 0) x = atomicAdd(&ctl->next, 1u);
        b = __shfl_sync(kFull, x, 0);
        const uint64_t u = b * 32 + lane;
        sg = (b < nb && u < units) ? g.get(u, bad) : Seg{nullptr, nullptr, 0, false};
    };
    auto store_oldest = [&]() -> bool {
        const int k = stored % kRing;
        bool w = true;
        if (lane == 0) w = mbar_wait(&bars[k], (stored / kRing) & 1u);
        w = __shfl_sync(kFull, w, 0);
        if (!w) return false;
        const uint32_t len = s_len[k][lane];
        if (len) bulk_s2g(s_dst[k][lane], ring + (uint64_t)k * kStageBytes + s_off[k][lane], len);
        bulk_commit();
        stored++;
        return true;
    };

    uint64_t bcur, bnxt;
    Seg cur, nxt;
    claim(bcur, cur);
    while (bcur < nb) {
        claim(bnxt, nxt);  // the next batch's addresses resolve while this one copies
        const uintptr_t al = reinterpret_cast<uintptr_t>(cur.src) | reinterpret_cast<uintptr_t>(cur.dst) | cur.len;
        const bool tma = cur.ok && cur.len > 0 && (al & 15) == 0;
        warp_copy(tma ? Seg{nullptr, nullptr, 0, false} : cur, lane);
        for (uint64_t r0 = 0;; r0 += kStageBytes) {  // rounds of at most one stage per segment
            const uint64_t left = tma && r0 < cur.len ? cur.len - r0 : 0;
            const uint32_t my_len = (uint32_t)(left < kStageBytes ? left : kStageBytes);
            if (!__any_sync(kFull, my_len != 0)) break;
            // stage groups in lane order, each at most one stage
            uint32_t grp = 0, off = 0, ngrp = 0, fill = 0;
            for (int i = 0; i < 32; i++) {
                const uint32_t li = __shfl_sync(kFull, my_len, i);
                if (li == 0) continue;
                if (ngrp == 0 || fill + li > kStageBytes) {
                    ngrp++;
                    fill = 0;
                }
                if (lane == (uint32_t)i) {
                    grp = ngrp - 1;
                    off = fill;
                }
                fill += li;
            }
            for (uint32_t k = 0; k < ngrp && ok; k++) {
                if (issued - stored == (uint32_t)kRing && !store_oldest()) {
                    ok = false;
                    break;
                }
                const int st = issued % kRing;
                if (issued >= (uint32_t)kRing) bulk_wait_read_all();  // its last store has read the stage
                const bool mine = my_len != 0 && grp == k;
                const uint32_t bytes = __reduce_add_sync(kFull, mine ? my_len : 0u);
                s_len[st][lane] = mine ? my_len : 0u;
                s_off[st][lane] = off;
                s_dst[st][lane] = cur.dst + r0;
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&bars[st], bytes);
                __syncwarp();
                if (mine) bulk_g2s(ring + (uint64_t)st * kStageBytes + off, cur.src + r0, my_len, &bars[st]);
                issued++;
            }
            if (!ok) break;
        }
        if (!ok) break;
        bcur = bnxt;
        cur = nxt;
    }
    while (ok && stored < issued) ok = store_oldest();
    if (!ok) {
        if (lane == 0) {
            atomicOr(g.status(), KVX_S_TIMEOUT);
            // let the loads still in flight land before the ring is released
            for (uint32_t k = stored; k < issued; k++) mbar_wait(&bars[k % kRing], (k / kRing) & 1u);
        }
        __syncwarp();
    }
    bulk_wait_all();
    warp_raise(g.status(), bad, lane);
}

template <class Gen>
cudaError_t set_ring_smem() {
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(k_seg_tma<Gen>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(kRingWarps * kRing * kStageBytes));
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

// Bulk-copy launch: one warp per SM; the claim counter is zeroed first.
template <class Gen>
kvx_status launch_tma(const Gen &g, void *ws, cudaStream_t s) {
    if (set_ring_smem<Gen>() != cudaSuccess) return KVX_ECUDA;
    SegCtl *ctl = static_cast<SegCtl *>(ws);
    if (cudaMemsetAsync(ctl, 0, sizeof(SegCtl), s) != cudaSuccess) return KVX_ECUDA;
    k_seg_tma<Gen><<<sm_count(), 32 * kRingWarps, kRingWarps * kRing * kStageBytes, s>>>(g, ctl);
    KVX_LAUNCHED();
    return KVX_OK;
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
    if (ws && page_len >= kBulkMinLen) return launch_tma(PagedGen{a}, ws, s);
    const uint32_t grid = grid_for(num_pages * pieces, resident_blocks(k_paged_writes, cache));
    k_paged_writes<<<grid, kThreads, 0, s>>>(a);
    KVX_LAUNCHED();
    return KVX_OK;
}

extern "C" kvx_status kvx_seal_blocks(const uint32_t *lane_first, const uint32_t *run_block,
                                      const uint32_t *run_group, const uint64_t *run_off,
                                      uint64_t run_capacity, const kvx_group *groups,
                                      uint64_t group_capacity, const uint64_t *counts, uint32_t B,
                                      uint32_t L, const uint32_t *seg_len, const uint8_t *slab,
                                      uint64_t slab_bytes, const uint64_t *dst_addr, uint8_t *dst,
                                      uint64_t dst_bytes, uint32_t *status, void *ws,
                                      size_t ws_bytes, void *stream) {
    if (!lane_first || !counts || !status) return KVX_EINVAL;
    if (ws && ws_bytes < kvx_segcopy_workspace_size()) return KVX_EINVAL;
    if ((uint64_t)B * L == 0) return KVX_OK;
    if (!run_block || !run_group || !run_off || !groups || !seg_len || !dst_addr ||
        (slab_bytes && !slab) || (dst_bytes && !dst))
        return KVX_EINVAL;
    static int cache[64] = {};
    SealArgs a{lane_first, run_block, run_group, run_off, run_capacity, groups, group_capacity,
               counts, B, L, seg_len, slab, slab_bytes, dst_addr, dst, dst_bytes, status};
    cudaStream_t s = as_stream(stream);
    if (ws) return launch_tma(SealGen{a}, ws, s);
    const uint32_t grid = grid_for((uint64_t)B * L, resident_blocks(k_seal_blocks, cache));
    k_seal_blocks<<<grid, kThreads, 0, s>>>(a);
    KVX_LAUNCHED();
    return KVX_OK;
}
