// Arithmetic rebuild of every segment's slab pointer (pegaflow PR #350,
// Requester step 5: local(b) = group_local + (remote(b) - group_remote),
// every pointer bounds-checked).
//
// With run r of lane l covering block b, G = its group and i = b - G.block,
// remote(b) = run_base[r] + (b - run_block[r]) * run_stride[r] (the run
// arithmetic, wrapping in 64 bits) and
//   dense group:     local = G.local + (remote(b) - G.base)
//   non-dense group: local = G.local + i * G.chunk + (remote(b) - (G.base + i * G.stride))
// (the page's formula, and its dense local mirror of each remote block),
// evaluated exactly.  The checks: the group index is valid, b is inside the
// group's block range, [local, local + len) lies inside block i's slice
// [G.local + i*chunk, G.local + (i+1)*chunk) of the carve, and the carve ends
// inside the slab.
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
constexpr int kCtasPerSm = 4;  // 56 registers: the run entry's gathers and checks fit without spilling

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
          const uint64_t *__restrict__ run_base, const int64_t *__restrict__ run_stride,
          const uint32_t *__restrict__ run_group, uint64_t run_cap, const kvx_group *__restrict__ groups, uint64_t group_cap,
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
    // Per run, everything that does not depend on the block is settled once
    // (enter).  When the run starts at its group's first block, its stride
    // equals the remote step of the group's blocks (a dense group's chunk, a
    // non-dense group's stride: true of every run of a planned group) and
    // its addresses do not wrap, local - slice is the same constant for
    // every block, so local(b) = G.local + (b - G.block)*chunk + c on the
    // window [vs, ve) of blocks in both the run and the group, and the loop
    // only compares and adds while all lanes still store row b together.
    // Any other run (a one-block group, a corrupt record) is evaluated one
    // block at a time with the exact formula: enter then covers block b
    // alone and asks to be called again at b + 1 (re).
    uint64_t vs = 0, ve = 0, v = 0, g_chunk = 0, re = b0;
    // the run after r: its first block and group index, loaded together
    uint64_t nb = ~0ull, rb = lane_ok ? run_block[r] : 0;  // rb: run r's first block
    uint32_t ngi = 0, gi = lane_ok ? run_group[r] : 0;
    if (lane_ok && r + 1 < hi) {
        nb = run_block[r + 1];
        ngi = run_group[r + 1];
    }
    auto enter = [&](uint64_t b) {  // run r from block b on
        vs = ve = 0;
        re = nb;
        if (!lane_ok || gi >= ngroups) return;
        // all loads first, and no branch before every check has used them
        // (a load sunk past an early return would cost a second round trip
        // to L2); the run's first block is known from the walk, so each run
        // costs three gathers besides the group record
        const kvx_group G = groups[gi];
        const uint64_t rbase = run_base[r];
        const int64_t rstr = run_stride[r];
        g_chunk = G.chunk;
        // the carve of the group ends inside the slab
        const bool carve_ok =
            (__int128)G.local + (__int128)G.count * (__int128)G.chunk <= (__int128)slab_bytes;
        // the run's blocks from b on that lie in the group: [lo, we)
        uint64_t lo = b > G.block ? b : G.block;
        lo = lo < rb ? rb : lo;
        uint64_t we = (uint64_t)G.block + G.count;
        we = nb < we ? nb : we;
        we = b1 < we ? b1 : we;
        // the fast case: the run starts at the group's first block, its
        // stride is the group's remote step, and its addresses do not wrap
        // over the window (moving monotonically, only the far end, block
        // we - 1, can leave [0, 2^64)); then local - slice = run_base - G.base
        const bool step_ok = G.dense ? (rstr >= 0 && (uint64_t)rstr == G.chunk) : rstr == G.stride;
        const uint64_t n = we - 1 - rb, m = rstr < 0 ? 0ull - (uint64_t)rstr : (uint64_t)rstr;
        const uint64_t span = n * m;
        const bool no_wrap = __umul64hi(n, m) == 0 && (rstr < 0 ? span <= rbase : span <= ~rbase);
        const uint64_t c = rbase - G.base;
        const bool c_ok = rbase >= G.base && c <= G.chunk && len <= G.chunk - c;
        if (!carve_ok || lo >= we) return;  // no block of the run is inside the group
        if (rb == G.block && step_ok && no_wrap) {
            if (c_ok) {  // otherwise every block overruns its slice
                vs = lo;
                ve = we;
                v = G.local + (vs - G.block) * G.chunk + c;
            }
            return;
        }
        // The exact formula for block b alone.  The carve ends inside the
        // slab, so for a block inside the group every offset below G.count *
        // G.chunk fits in 64 bits; only a non-dense group's G.base + i *
        // G.stride needs 128.
        re = b + 1;
        const uint64_t i = b - G.block;
        if (b < rb || b < G.block || i >= G.count) return;
        const uint64_t remote = rbase + (b - rb) * (uint64_t)rstr;
        const uint64_t slice = i * G.chunk;  // block i's part of the carve, from G.local
        bool ok;
        uint64_t off;  // the segment's offset inside its slice
        if (G.dense) {  // local = G.local + (remote - G.base)
            ok = remote >= G.base && remote - G.base >= slice;
            off = remote - G.base - slice;
        } else {        // local = G.local + slice + (remote - (G.base + i * G.stride))
            const __int128 e = (__int128)remote - ((__int128)G.base + (__int128)i * (__int128)G.stride);
            ok = e >= 0 && e <= (__int128)G.chunk;
            off = (uint64_t)e;
        }
        if (ok && off <= G.chunk && len <= G.chunk - off) {
            vs = b;
            ve = b + 1;
            v = G.local + slice + off;
        }
    };
    uint64_t *dst = local + b0 * L + l;
    for (uint64_t b = b0; b < b1; b++, dst += L) {
        if (re <= b) {
            while (nb <= b) {  // the next run starts at or before b
                r++;
                gi = ngi;
                rb = nb;
                nb = ~0ull;
                if (r + 1 < hi) {
                    nb = run_block[r + 1];
                    ngi = run_group[r + 1];
                }
            }
            enter(b);
        }
        uint64_t out = ~0ull;
        if (b >= vs && b < ve) {
            out = v;
            v += g_chunk;
        } else {
            bad = KVX_S_BOUNDS;
        }
        *dst = out;
    }
    if (bad) atomicOr(status, bad);
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" kvx_status kvx_rebuild(const uint32_t *lane_first, const uint32_t *run_block,
                                  const uint64_t *run_base, const int64_t *run_stride,
                                  const uint32_t *run_group, uint64_t run_capacity, const kvx_group *groups,
                                  uint64_t group_capacity, const uint64_t *counts, uint32_t B,
                                  uint32_t L, const uint32_t *seg_len, uint64_t slab_bytes,
                                  uint64_t *local, uint32_t *status, void *stream) {
    if (!lane_first || !counts || !status) return KVX_EINVAL;
    if ((uint64_t)B * L == 0) return KVX_OK;
    if (!run_block || !run_base || !run_stride || !run_group || !groups || !seg_len || !local)
        return KVX_EINVAL;
    const Geometry g = geometry(B, L, (uint64_t)sm_count() * kCtasPerSm);
    k_rebuild<<<g.ntl * g.ntr, kThreads, 0, as_stream(stream)>>>(
        lane_first, run_block, run_base, run_stride, run_group, run_capacity, groups, group_capacity, counts, B,
        L, seg_len, slab_bytes, local, status, g);
    KVX_LAUNCHED();
    return KVX_OK;
}
