// Arithmetic rebuild of every segment's slab pointer (pegaflow PR #350,
// Requester step 5: local(b) = group_local + (remote(b) - group_remote),
// every pointer bounds-checked).
//
// With run r of lane l covering block b, G = its group and i = b - G.block:
//   dense group:     local = G.local + (remote(b) - G.base)
//                          = G.local + i * G.stride + run_off[r]
//   non-dense group: local = G.local + i * G.chunk + run_off[r]
// (the page's formula, and its dense local mirror of each remote block).
// The checks: the group index is valid, the run starts at the group's first
// block, b is inside the group's block range, [local, local + len) lies
// inside block i's slice [G.local + i*chunk, G.local + (i+1)*chunk) of the
// carve, and the carve ends inside the slab.  The call is not given the runs'
// strides: a dense group's stride stands for them.
//
// Thread layout as in the encoder: a CTA is 8 warps; lane t of warp w handles
// lane l0 + t over K consecutive blocks, so each warp store is one coalesced
// row segment of the block-major output.  K grows with the table until the
// grid fits on the device at once (a second wave would repeat the whole
// latency chain).  A thread finds the run covering its first block by an
// interpolation-guided search of the lane's run_block list (exact when the
// lane's runs have equal lengths), then walks, loading each next run's group
// index together with its first block.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kRows = 8;
constexpr int kThreads = 32 * kRows;
constexpr int kCtasPerSm = 5;

struct Geometry {
    uint32_t K, ntl, ntr;
};

Geometry geometry(uint32_t B, uint32_t L, uint64_t max_ctas) {
    Geometry g;
    g.ntl = (uint32_t)ceil_div(L ? L : 1, 32);
    const uint64_t rows = max_ctas / g.ntl ? max_ctas / g.ntl : 1;  // row tiles that fit beside ntl lane tiles
    const uint64_t K = ceil_div(B ? B : 1, (uint64_t)kRows * rows);
    g.K = K < 4 ? 4 : (uint32_t)K;
    g.ntr = (uint32_t)ceil_div(B ? B : 1, (uint64_t)kRows * g.K);
    return g;
}

// Last index m in [lo, hi) with run_block[m] <= b, for a list that starts at
// block 0 and increases up to B.  Each probe loads two neighbours (one round
// trip) and stops when they bracket b; probes alternate between an
// interpolation guess and bisection, so any list takes O(log n) probes.  An
// unordered list only makes the answer meaningless; it stays in [lo, hi).
__device__ __forceinline__ uint64_t find_run(const uint32_t *__restrict__ run_block, uint64_t lo, uint64_t hi,
                                             uint64_t b, uint64_t B) {
    uint64_t a = lo, z = hi;    // answer in [a, z)
    uint64_t ba = 0, bz = B;    // run_block[a], and run_block[z] (B for z = hi)
    bool guess = true;
    while (z - a > 1) {
        uint64_t m = (a + z) >> 1;
        if (guess && ba <= b && b < bz) {
            // single precision on purpose: the guess only steers the search
            // (double precision is a slow path on this part)
            const float f = __fdividef((float)(b - ba), (float)(bz - ba));
            const uint64_t q = a + (uint64_t)(f * (float)(z - a));
            m = q < a ? a : (q > z - 1 ? z - 1 : q);
        }
        guess = !guess;
        const uint64_t b0 = run_block[m];
        const uint64_t b1 = m + 1 < z ? run_block[m + 1] : bz;
        if (b0 <= b) {
            if (b < b1) return m;
            a = m + 1;
            ba = b1;
        } else {
            z = m;
            bz = b0;
        }
    }
    return a < hi ? a : hi - 1;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
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
    uint64_t r = lane_ok ? find_run(run_block, lo, hi, b0, B) : lo;
    uint32_t bad = 0;
    // Per run, everything that does not depend on the block is settled once.
    // Every valid group advances its local pointer by the chunk per block (a
    // dense group's stride equals its chunk, and a one-block group has no
    // step), so local(b) = G.local + (b - G.block)*chunk + off on the run's
    // window [vs, ve) of blocks inside the group, when off + len <= chunk and
    // the carve ends inside the slab; the loop then only compares and adds,
    // and all lanes still store row b together.  A dense group whose stride
    // differs from its chunk is checked block by block (general).
    uint64_t vs = 0, ve = 0, v = 0, g_chunk = 0, g_local = 0, g_block = 0, g_count = 0, off = 0, rb = 0;
    int64_t g_stride = 0;
    bool general = false;
    // the run after r: its first block and group index, loaded together
    uint64_t nb = ~0ull;
    uint32_t ngi = 0, gi = lane_ok ? run_group[r] : 0;
    if (lane_ok && r + 1 < hi) {
        nb = run_block[r + 1];
        ngi = run_group[r + 1];
    }
    auto enter = [&](uint64_t b) {  // run r from block b on
        vs = ve = 0;
        general = false;
        if (!lane_ok || gi >= ngroups) return;
        const kvx_group G = groups[gi];
        g_local = G.local;
        g_chunk = G.chunk;
        g_stride = G.stride;
        g_block = G.block;
        g_count = G.count;
        off = run_off[r];
        rb = run_block[r];
        // the carve of the group ends inside the slab, and the run starts at
        // the group's first block (every run of a group does)
        if ((__int128)g_local + (__int128)G.count * (__int128)g_chunk > (__int128)slab_bytes) return;
        if (rb != g_block) return;
        if (G.dense && G.count > 1 && (__int128)g_stride != (__int128)g_chunk) {
            general = true;
            return;
        }
        if (!(off <= g_chunk && len <= g_chunk - off)) return;  // the segment overruns its slice
        vs = g_block > b ? g_block : b;
        ve = g_block + g_count;
        if (vs < ve) v = g_local + (vs - g_block) * g_chunk + off;
    };
    enter(b0);
    uint64_t *dst = local + b0 * L + l;
    for (uint64_t b = b0; b < b1; b++, dst += L) {
        if (nb <= b) {  // the next run starts at or before b
            do {
                r++;
                gi = ngi;
                nb = ~0ull;
                if (r + 1 < hi) {
                    nb = run_block[r + 1];
                    ngi = run_group[r + 1];
                }
            } while (nb <= b);
            enter(b);
        }
        uint64_t out = ~0ull;
        if (b >= vs && b < ve) {
            out = v;
            v += g_chunk;
        } else if (general && b >= g_block && b - g_block < g_count) {
            // dense: remote(b) - group_remote advances by the stride
            const uint64_t i = b - g_block;
            const __int128 loc = (__int128)g_local + (__int128)i * g_stride + (__int128)off;
            const __int128 slice = (__int128)g_local + (__int128)i * g_chunk;  // block i's part of the carve
            if (loc >= slice && loc + (__int128)len <= slice + (__int128)g_chunk) out = (uint64_t)loc;
        }
        if (out == ~0ull) bad = KVX_S_BOUNDS;
        *dst = out;
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
    const Geometry g = geometry(B, L, (uint64_t)sm_count() * kCtasPerSm);
    k_rebuild<<<g.ntl * g.ntr, kThreads, 0, as_stream(stream)>>>(
        lane_first, run_block, run_group, run_off, run_capacity, groups, group_capacity, counts, B,
        L, seg_len, slab_bytes, local, status, g);
    KVX_LAUNCHED();
    return KVX_OK;
}
