// Segment copies shared by the copy kernels (sm_103a): a batch of 32
// segments per warp, each lane holding one segment's source, destination and
// length, moved either through registers (warp_copy) or through the SM's
// bulk-copy engine (k_seg_tma, a ring of shared-memory stages per warp).
#pragma once

#include "kvx_common.cuh"

namespace kvx {
namespace ring {
namespace {

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
constexpr int kRing = 3;
constexpr int kRingWarps = 4;  // independent rings per SM, so one warp's stalls hide behind the others

struct SegCtl {
    uint32_t next;  // next unclaimed batch
};

// A ring's bookkeeping in shared memory: one mbarrier per stage, and per
// stage the store each lane owes (destination, offset in the stage, length).
struct RingSmem {
    uint64_t bars[kRing];
    uint8_t *s_dst[kRing][32];
    uint32_t s_off[kRing][32], s_len[kRing][32];
};

// One warp drives one ring: ring points at its kRing * kStageBytes bytes of
// shared memory.  Batches of 32 segments are claimed from ctl until g has
// none left.
template <class Gen>
__device__ void ring_warp(const Gen &g, SegCtl *ctl, uint8_t *ring, RingSmem &rs, uint32_t lane) {
    uint64_t *bars = rs.bars;
    auto &s_dst = rs.s_dst;
    auto &s_off = rs.s_off;
    auto &s_len = rs.s_len;
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
__global__ void __launch_bounds__(32 * kRingWarps, 1) k_seg_tma(const __grid_constant__ Gen g, SegCtl *ctl) {
    extern __shared__ __align__(128) uint8_t ring_all[];
    __shared__ RingSmem rs[kRingWarps];
    const uint32_t wid = threadIdx.x >> 5;
    ring_warp(g, ctl, ring_all + (uint64_t)wid * kRing * kStageBytes, rs[wid], threadIdx.x & 31);
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

// Bulk-copy launch: one CTA of kRingWarps rings per SM.  The claim counter
// *ctl must be zero when the kernel starts (the caller clears it on s).
template <class Gen>
kvx_status launch_ring(const Gen &g, SegCtl *ctl, cudaStream_t s) {
    if (set_ring_smem<Gen>() != cudaSuccess) return KVX_ECUDA;
    k_seg_tma<Gen><<<sm_count(), 32 * kRingWarps, kRingWarps * kRing * kStageBytes, s>>>(g, ctl);
    KVX_LAUNCHED();
    return KVX_OK;
}

}  // namespace
}  // namespace ring
}  // namespace kvx
