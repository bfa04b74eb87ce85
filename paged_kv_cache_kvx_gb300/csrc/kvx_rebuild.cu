// Arithmetic rebuild of every segment's slab pointer (pegaflow PR #350,
// Requester step 5: local(b) = group_local + (remote(b) - group_remote),
// every pointer bounds-checked).
//
// With run r of lane l covering block b, G = its group and i = b - G.block:
//   dense group:     local = G.local + (remote(b) - G.base)
//                          = G.local + i * G.stride + run_off[r]
//   non-dense group: local = G.local + i * G.chunk + run_off[r]
// (the page's formula, and its dense local mirror of each remote block).
// The checks: the group index is valid, b is inside the group's block range,
// [local, local + len) lies inside block i's slice [G.local + i*chunk,
// G.local + (i+1)*chunk) of the carve, and the carve ends inside the slab.
//
// Thread layout as in the encoder: a CTA is 8 warps; lane t of warp w handles
// lane l0 + t over K consecutive blocks, so each warp store is one coalesced
// row segment of the block-major output.  A thread finds the run covering its
// first block by binary search in the lane's run_block list, then walks.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kRows = 8;
constexpr int kThreads = 32 * kRows;
constexpr uint32_t kTargetCtas = 2048;

struct Geometry {
    uint32_t K, ntl, ntr;
};

Geometry geometry(uint32_t B, uint32_t L) {
    Geometry g;
    g.ntl = (uint32_t)ceil_div(L ? L : 1, 32);
    g.K = 4;
    while (g.K < 64 && (uint64_t)g.ntl * ceil_div(B ? B : 1, (uint64_t)kRows * g.K) > kTargetCtas)
        g.K *= 2;
    g.ntr = (uint32_t)ceil_div(B ? B : 1, (uint64_t)kRows * g.K);
    return g;
}

__global__ void __launch_bounds__(kThreads)
k_rebuild(const uint32_t *__restrict__ lane_first, const uint32_t *__restrict__ run_block,
          const uint32_t *__restrict__ run_group, const uint64_t *__restrict__ run_off,
          uint64_t run_cap, const kvx_group *__restrict__ groups, uint64_t group_cap,
          const uint64_t *__restrict__ counts, uint32_t B, uint32_t L,
          const uint32_t *__restrict__ seg_len, uint64_t slab_bytes, uint64_t *__restrict__ local,
          uint32_t *status, Geometry g) {
    const uint32_t tl = blockIdx.x % g.ntl, tr = blockIdx.x / g.ntl;
    const uint32_t t = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t l = tl * 32 + t;
    const uint64_t b0 = (uint64_t)tr * kRows * g.K + (uint64_t)w * g.K;
    if (l >= L || b0 >= B) return;
    const uint64_t b1 = b0 + g.K < B ? b0 + g.K : B;
    const uint64_t ngroups = counts[0] < group_cap ? counts[0] : group_cap;
    const uint64_t len = seg_len[l];

    uint64_t lo = lane_first[l], hi = lane_first[l + 1];
    bool lane_ok = lo < hi && hi <= run_cap;
    uint64_t r = lo;
    if (lane_ok) {
        // last run of the lane whose first block is <= b0
        uint64_t a = lo, z = hi;  // answer in [a, z)
        while (z - a > 1) {
            const uint64_t m = (a + z) >> 1;
            if (run_block[m] <= b0) a = m; else z = m;
        }
        r = a;
    }
    uint32_t bad = 0;
    // cached per run: its group's fields and its offset inside the group
    uint64_t cur_r = ~0ull, off = 0, g_block = 0, g_count = 0;
    __int128 g_local = 0, g_chunk = 0, g_step = 0;
    bool run_ok = false;
    for (uint64_t b = b0; b < b1; b++) {
        uint64_t out = ~0ull;
        if (lane_ok) {
            while (r + 1 < hi && run_block[r + 1] <= b) r++;
            if (r != cur_r) {
                cur_r = r;
                const uint32_t gi = run_group[r];
                run_ok = gi < ngroups;
                if (run_ok) {
                    const kvx_group G = groups[gi];
                    g_local = (__int128)G.local;
                    g_chunk = (__int128)G.chunk;
                    // dense: remote(b) - group_remote advances by the stride;
                    // non-dense: the dense local mirror advances by the chunk
                    g_step = G.dense ? (__int128)G.stride : (__int128)G.chunk;
                    g_block = G.block;
                    g_count = G.count;
                    off = run_off[r];
                    run_ok = g_local + (__int128)G.count * g_chunk <= (__int128)slab_bytes;
                }
            }
            if (run_ok && b >= g_block && b - g_block < g_count && run_block[r] <= b) {
                const __int128 i = (__int128)(b - g_block);
                const __int128 loc = g_local + i * g_step + (__int128)off;
                const __int128 slice = g_local + i * g_chunk;  // this block's part of the carve
                if (loc >= slice && loc + (__int128)len <= slice + g_chunk) out = (uint64_t)loc;
            }
        }
        if (out == ~0ull) bad = KVX_S_BOUNDS;
        local[b * L + l] = out;
    }
    if (bad) atomicOr(status, bad);
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" kvx_status kvx_rebuild(const uint32_t *lane_first, const uint32_t *run_block,
                                  const uint32_t *run_group, const uint64_t *run_off,
                                  uint64_t run_capacity, const kvx_group *groups,
                                  uint64_t group_capacity, const uint64_t *counts, uint32_t B,
                                  uint32_t L, const uint32_t *seg_len, uint64_t slab_bytes,
                                  uint64_t *local, uint32_t *status, void *stream) {
    if (!lane_first || !counts || !status) return KVX_EINVAL;
    if ((uint64_t)B * L == 0) return KVX_OK;
    if (!run_block || !run_group || !run_off || !groups || !seg_len || !local) return KVX_EINVAL;
    const Geometry g = geometry(B, L);
    k_rebuild<<<g.ntl * g.ntr, kThreads, 0, as_stream(stream)>>>(
        lane_first, run_block, run_group, run_off, run_capacity, groups, group_capacity, counts, B,
        L, seg_len, slab_bytes, local, status, g);
    KVX_LAUNCHED();
    return KVX_OK;
}
