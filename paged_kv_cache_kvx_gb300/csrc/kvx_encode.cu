// Run encoding of the block prefix's per-segment address table
// (pegaflow PR #350, Holder paragraph: per-lane greedy run accumulators;
// Wire format paragraph: runs_per_lane / run_base / run_stride / run_count).
//
// The greedy rule as a state machine per lane: S_0 = START; for i >= 1,
// S_i = IN when S_{i-1} = START or d[i-1] == d[i-2] (d[j] = a[j+1] - a[j]),
// otherwise S_i = START.  So each position's transition is either "constant
// IN" (i == 1, or two equal consecutive differences) or "NOT".  A thread
// runs its slice of a lane under both possible entry states at once; the
// slices are combined by an associative operator into per-lane prefixes
// (entry state, runs before, last start before), and an emit pass writes
// each run at its lane-major index.
//
// One cooperative kernel, three phases separated by bounded grid barriers:
//   1. per tile (32 lanes x 8K blocks): the tile's effect on each lane;
//   2. one warp per lane: a warp-shuffle scan of its tiles' effects gives
//      every tile's entry prefix and the lane's run count, which is also
//      added atomically to its 32-lane tile's total (for tall tables, one
//      warp per lane and chunk of 32 row tiles, with one more barrier
//      between the chunks' own scans and the fold of earlier chunks);
//   3. per tile: lane offsets (totals of earlier lane tiles plus a warp
//      scan), then every thread re-walks its slice from its entry prefix
//      and writes its runs.
// Thread layout: a CTA is 8 warps; lane t of warp w handles table lane
// l0 + t over blocks [tile_b0 + w*K, +K), so every warp load is one
// coalesced 256-byte row segment of the block-major table.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kRows = 8;           // warps per CTA = row slices per tile
constexpr int kThreads = 32 * kRows;

// Effect of a slice on the greedy state, for entry state 0 (START) or 1 (IN).
struct Xfer {
    uint32_t cnt[2];   // run starts inside the slice
    uint32_t last[2];  // block of the last start inside the slice, or kNone
    uint32_t fin[2];   // state at the slice's last block
};

__device__ __forceinline__ Xfer xfer_identity() {
    Xfer x;
    x.cnt[0] = x.cnt[1] = 0;
    x.last[0] = x.last[1] = kNone;
    x.fin[0] = 0;
    x.fin[1] = 1;
    return x;
}

// Entry e of a two-entry field, by select (keeps Xfer in registers).
__device__ __forceinline__ uint32_t pick(const uint32_t (&v)[2], uint32_t e) {
    return e ? v[1] : v[0];
}

// a then b
__device__ __forceinline__ Xfer xfer_then(const Xfer &a, const Xfer &b) {
    Xfer c;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const uint32_t e1 = a.fin[e];
        const uint32_t bl = pick(b.last, e1);
        c.cnt[e] = a.cnt[e] + pick(b.cnt, e1);
        c.last[e] = bl != kNone ? bl : a.last[e];
        c.fin[e] = pick(b.fin, e1);
    }
    return c;
}

// Resolved prefix at a slice boundary: state of the block before the slice,
// runs started before it, and the block of the last start before it.
struct Prefix {
    uint32_t state;
    uint32_t runs;
    uint32_t prev;
};

__device__ __forceinline__ Prefix prefix_then(const Prefix &p, const Xfer &x) {
    Prefix q;
    const uint32_t xl = pick(x.last, p.state);
    q.state = pick(x.fin, p.state);
    q.runs = p.runs + pick(x.cnt, p.state);
    q.prev = xl != kNone ? xl : p.prev;
    return q;
}

// Per-lane tile records in the workspace: first the tile's Xfer, then (after
// the per-lane scan) the tile's entry Prefix.
struct TileRec {
    uint32_t a, b, c, d;
};

__device__ __forceinline__ TileRec pack_xfer(const Xfer &x) {
    return TileRec{x.cnt[0] | (x.fin[0] << 31), x.cnt[1] | (x.fin[1] << 31), x.last[0], x.last[1]};
}
__device__ __forceinline__ Xfer unpack_xfer(const TileRec &t) {
    Xfer x;
    x.cnt[0] = t.a & 0x7FFFFFFFu;
    x.fin[0] = t.a >> 31;
    x.cnt[1] = t.b & 0x7FFFFFFFu;
    x.fin[1] = t.b >> 31;
    x.last[0] = t.c;
    x.last[1] = t.d;
    return x;
}

struct EncodeCtl {
    GridSync gs;
    uint32_t cut;  // template check: B - (first failing block), 0 when every block passes
};

__device__ __forceinline__ uint64_t ld_addr(const uint64_t *addr, uint64_t b, uint32_t L, uint32_t l) {
    return __ldg(addr + b * L + l);
}

// Position of the j-th set bit (from 0) of m; m has more than j set bits.
__device__ __forceinline__ uint32_t nth_bit(uint64_t m, uint32_t j) {
    uint32_t x = (uint32_t)m, pos = 0;
    const uint32_t c = __popc(x);
    if (j >= c) {
        x = (uint32_t)(m >> 32);
        j -= c;
        pos = 32;
    }
#pragma unroll
    for (uint32_t s = 16; s > 0; s >>= 1) {
        const uint32_t below = __popc(x & ((1u << s) - 1u));
        if (j >= below) {
            x >>= s;
            j -= below;
            pos += s;
        }
    }
    return pos;
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, uint32_t src) {
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src);
    return (uint64_t)hi << 32 | lo;
}

// Slice [b0, b1) of lane l under both entry states; m0 / m1 get a bit per
// block of the slice (bit i - b0) where a run starts under entry state 0 /
// 1 (slices are at most 64 blocks).
__device__ Xfer slice_xfer(const uint64_t *addr, uint32_t L, uint32_t l, uint64_t b0, uint64_t b1,
                           uint64_t &m0, uint64_t &m1) {
    Xfer x = xfer_identity();
    m0 = m1 = 0;
    if (b0 >= b1) return x;
    uint64_t p2 = b0 >= 2 ? ld_addr(addr, b0 - 2, L, l) : 0;
    uint64_t p1 = b0 >= 1 ? ld_addr(addr, b0 - 1, L, l) : 0;
    uint32_t s0 = 0, s1 = 1;
#pragma unroll 4
    for (uint64_t i = b0; i < b1; i++) {
        const uint64_t a = ld_addr(addr, i, L, l);
        uint32_t n0, n1;
        if (i == 0) {
            n0 = n1 = 0;
        } else if (i == 1 || a - p1 == p1 - p2) {
            n0 = n1 = 1;
        } else {
            n0 = s0 ^ 1u;
            n1 = s1 ^ 1u;
        }
        const uint64_t bit = 1ull << (i - b0);
        if (n0 == 0) { x.cnt[0]++; x.last[0] = (uint32_t)i; m0 |= bit; }
        if (n1 == 0) { x.cnt[1]++; x.last[1] = (uint32_t)i; m1 |= bit; }
        s0 = n0;
        s1 = n1;
        p2 = p1;
        p1 = a;
    }
    x.fin[0] = s0;
    x.fin[1] = s1;
    return x;
}

struct Geometry {
    uint32_t K;     // blocks per thread
    uint32_t ntl;   // lane tiles (32 lanes each)
    uint32_t ntr;   // row tiles (kRows * K blocks each)
};

// The launch geometry: slices of K blocks, K chosen so that the tiles fill at
// most kTilesPerSm blocks on every SM (phases 1 and 3 then end together on
// every SM; an SM with one block more than the others sets the pace), K at
// least kMinK and at most 64 (a slice's run starts fit one 64-bit mask).
constexpr uint32_t kMinK = 8;
constexpr uint32_t kTilesPerSm = 5;

Geometry geometry(uint32_t B, uint32_t L, uint32_t sms, uint32_t k_min = kMinK) {
    Geometry g;
    g.ntl = (uint32_t)ceil_div(L ? L : 1, 32);
    const uint64_t target = (uint64_t)kTilesPerSm * (sms ? sms : 1);
    const uint64_t rows = target / g.ntl ? target / g.ntl : 1;  // row tiles that fit beside ntl lane tiles
    const uint64_t K = ceil_div(B ? B : 1, (uint64_t)kRows * rows);
    g.K = K < k_min ? k_min : (K > 64 ? 64 : (uint32_t)K);
    g.ntr = (uint32_t)ceil_div(B ? B : 1, (uint64_t)kRows * g.K);
    return g;
}

// The workspace holds the tile records of the tallest geometry any device
// can choose (K = kMinK), so its size does not depend on the device.
Geometry ws_geometry(uint32_t B, uint32_t L) {
    Geometry g;
    g.ntl = (uint32_t)ceil_div(L ? L : 1, 32);
    g.K = kMinK;
    g.ntr = (uint32_t)ceil_div(B ? B : 1, (uint64_t)kRows * kMinK);
    return g;
}

// Row tiles per lane above which the lane scan is spread over every warp of
// the grid, one warp per (lane, chunk of 32 row tiles).
constexpr uint32_t kTallRows = 64;

__host__ __device__ __forceinline__ uint32_t lane_chunks(const Geometry &g) {
    return g.ntr > kTallRows ? (g.ntr + 31) / 32 : 0;
}

struct Ws {
    EncodeCtl *ctl;
    TileRec *tiles;       // [ntr][L]
    uint64_t *tile_runs;  // [ntl]
    TileRec *chunks;      // [L][lane_chunks]: each chunk's combined effect (tall tables)
};

Ws carve(void *base, uint32_t B, uint32_t L, size_t *bytes) {
    Geometry g = ws_geometry(B, L);
    Carver c(base);
    Ws w;
    w.ctl = c.take<EncodeCtl>(1);
    w.tile_runs = c.take<uint64_t>(g.ntl);
    w.tiles = c.take<TileRec>((size_t)g.ntr * L);
    w.chunks = c.take<TileRec>((size_t)L * lane_chunks(g));
    *bytes = c.off;
    return w;
}

__device__ __forceinline__ Xfer shfl_up_xfer(const Xfer &v, int d) {
    Xfer o;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        o.cnt[e] = __shfl_up_sync(0xFFFFFFFFu, v.cnt[e], d);
        o.last[e] = __shfl_up_sync(0xFFFFFFFFu, v.last[e], d);
        o.fin[e] = __shfl_up_sync(0xFFFFFFFFu, v.fin[e], d);
    }
    return o;
}

__device__ __forceinline__ Xfer shfl_xfer(const Xfer &v, int src) {
    Xfer o;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        o.cnt[e] = __shfl_sync(0xFFFFFFFFu, v.cnt[e], src);
        o.last[e] = __shfl_sync(0xFFFFFFFFu, v.last[e], src);
        o.fin[e] = __shfl_sync(0xFFFFFFFFu, v.fin[e], src);
    }
    return o;
}

// Sum of v[0..n) by the whole block (every thread gets the result).
__device__ uint64_t block_sum_tiles(const uint64_t *v, uint32_t n, uint64_t *s_red) {
    const uint32_t t = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint64_t sum = 0;
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) sum += __ldcg(v + i);
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_down_sync(0xFFFFFFFFu, sum, d);
    __syncthreads();  // s_red may still be read from the previous call
    if (t == 0) s_red[w] = sum;
    __syncthreads();
    uint64_t tot = 0;
    for (int i = 0; i < kRows; i++) tot += s_red[i];
    return tot;
}

struct EncodeArgs {
    const uint64_t *addr;
    const uint32_t *seg_size;  // optional [B][L]: observed segment sizes (template check)
    const uint32_t *tmpl_len;  // [L] template segment lengths (with seg_size)
    uint32_t *prefix;          // [1] out: blocks that pass (with seg_size)
    uint32_t B, L;
    Geometry g;
    TileRec *tiles;
    TileRec *chunks;
    uint32_t *runs_per_lane;
    uint64_t *tile_runs;
    uint64_t *num_runs;
    uint64_t *run_base;
    int64_t *run_stride;
    uint32_t *run_count;
    uint64_t run_cap;
    EncodeCtl *ctl;
    uint32_t *status;
};

// Scans the effects of row tiles [r_lo, r_hi) of lane l in chunks of 32 (one
// per lane of the warp), from entry prefix carry: every tile's record is
// replaced by its entry prefix.  Returns the prefix after r_hi.
__device__ Prefix scan_tile_range(TileRec *tiles, uint32_t L, uint32_t l, uint32_t r_lo, uint32_t r_hi,
                                  Prefix carry, uint32_t t) {
    for (uint32_t c0 = r_lo; c0 < r_hi; c0 += 32) {
        const uint32_t r = c0 + t;
        TileRec *slot = tiles + (uint64_t)r * L + l;
        Xfer x = xfer_identity();
        if (r < r_hi) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(slot));
            x = unpack_xfer(TileRec{v.x, v.y, v.z, v.w});
        }
        Xfer incl = x;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Xfer o = shfl_up_xfer(incl, d);
            if ((int)t >= d) incl = xfer_then(o, incl);
        }
        Xfer excl = shfl_up_xfer(incl, 1);
        if (t == 0) excl = xfer_identity();
        const Prefix mine = prefix_then(carry, excl);
        if (r < r_hi) *slot = TileRec{mine.state, mine.runs, mine.prev, 0u};
        carry = prefix_then(carry, shfl_xfer(incl, 31));
    }
    return carry;
}

// A lane's run count, and its share of its 32-lane tile's total (zeroed with
// the control block).
__device__ __forceinline__ void lane_done(const EncodeArgs &a, uint32_t l, uint32_t runs) {
    a.runs_per_lane[l] = runs;
    atomicAdd(reinterpret_cast<unsigned long long *>(a.tile_runs + l / 32), (unsigned long long)runs);
}

// Six blocks per SM fit (40 registers); the geometry fills at most five per
// SM with tiles (758 tiles of a 100,000 x 64 table on 152 SMs), so tables
// up to that height run one tile per block, and taller ones loop.
__global__ void __launch_bounds__(kThreads, 6) k_encode(const __grid_constant__ EncodeArgs a) {
    __shared__ Xfer sx[kRows][32];     // slice effects; kept from phase 1 to 3 when one_tile
    __shared__ uint64_t sm0[kRows][32], sm1[kRows][32];  // slice run starts (one_tile)
    __shared__ Prefix sp[kRows][32];
    __shared__ uint64_t s_lb[32];
    __shared__ uint64_t s_red[kRows];
    const uint32_t B = a.B, L = a.L;
    const Geometry g = a.g;
    const uint32_t t = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t ntiles = g.ntl * g.ntr;
    const uint32_t G = gridDim.x;

    // ---- phase 0 (holder prefix scan): the first block whose segment sizes
    // differ from the template ends the prefix; blocks from it on add nothing
    uint32_t Bv = B;
    if (a.prefix) {
        uint32_t cut = 0;
        for (uint32_t tile = blockIdx.x; tile < ntiles; tile += G) {
            const uint32_t tl = tile % g.ntl, tr = tile / g.ntl;
            const uint32_t l = tl * 32 + t;
            const uint64_t b0 = (uint64_t)tr * kRows * g.K + (uint64_t)w * g.K;
            const uint64_t b1 = b0 + g.K < B ? b0 + g.K : B;
            if (l < L) {
                const uint32_t want = __ldg(a.tmpl_len + l);
                for (uint64_t b = b0; b < b1; b++)
                    if (__ldg(a.seg_size + b * L + l) != want) {
                        cut = max(cut, (uint32_t)(B - b));
                        break;
                    }
            }
        }
        for (int d = 16; d > 0; d >>= 1) cut = max(cut, __shfl_xor_sync(0xFFFFFFFFu, cut, d));
        if (t == 0 && cut) atomicMax(&a.ctl->cut, cut);
        if (!grid_barrier(&a.ctl->gs, G)) {
            if (threadIdx.x == 0) atomicOr(a.status, KVX_S_TIMEOUT);
            return;
        }
        Bv = B - *(volatile uint32_t *)&a.ctl->cut;
        if (blockIdx.x == 0 && threadIdx.x == 0) *a.prefix = Bv;
    }

    // ---- phase 1: each tile's effect on each of its lanes
    const bool one_tile = ntiles <= G;  // every block has at most one tile in phases 1 and 3
    for (uint32_t tile = blockIdx.x; tile < ntiles; tile += G) {
        const uint32_t tl = tile % g.ntl, tr = tile / g.ntl;
        const uint32_t l = tl * 32 + t;
        const uint64_t b0 = (uint64_t)tr * kRows * g.K + (uint64_t)w * g.K;
        const uint64_t b1 = b0 + g.K < Bv ? b0 + g.K : Bv;
        uint64_t m0 = 0, m1 = 0;
        sx[w][t] = (l < L && b0 < Bv) ? slice_xfer(a.addr, L, l, b0, b1, m0, m1) : xfer_identity();
        sm0[w][t] = m0;
        sm1[w][t] = m1;
        __syncthreads();
        if (w == 0 && l < L) {
            Xfer acc = sx[0][t];
            for (int r = 1; r < kRows; r++) acc = xfer_then(acc, sx[r][t]);
            a.tiles[(uint64_t)tr * L + l] = pack_xfer(acc);
        }
        __syncthreads();
    }
    if (!grid_barrier(&a.ctl->gs, G)) {
        if (threadIdx.x == 0) atomicOr(a.status, KVX_S_TIMEOUT);
        return;
    }

    // ---- phase 2: per lane, a warp-shuffle scan over its tiles' effects.  One
    // warp per lane; for tall tables (many row tiles, few lanes) one warp
    // per (lane, chunk of 32 row tiles) over the whole grid: each chunk is
    // scanned on its own and its total published, then, after a barrier,
    // every chunk folds the totals of the lane's earlier chunks into its
    // tiles' entry prefixes.
    // Work items are numbered warp-major over the blocks (item i to warp i / G
    // of block i % G): numbered block-major, the few hundred items landed on
    // the first blocks, eight warps each, and ran several times slower.
    if (g.ntr <= kTallRows) {
        for (uint32_t l = w * G + blockIdx.x; l < L; l += G * kRows) {
            const Prefix carry = scan_tile_range(a.tiles, L, l, 0, g.ntr, Prefix{0u, 0u, kNone}, t);
            if (t == 0) lane_done(a, l, carry.runs);
        }
    } else {
        const uint32_t C = lane_chunks(g);
        const uint64_t tasks = (uint64_t)L * C;
        const uint64_t gw = (uint64_t)w * G + blockIdx.x, nw = (uint64_t)G * kRows;
        for (uint64_t q = gw; q < tasks; q += nw) {  // each chunk's own scan
            const uint32_t l = (uint32_t)(q / C), c = (uint32_t)(q % C);
            const uint32_t r = c * 32 + t;
            TileRec *slot = a.tiles + (uint64_t)r * L + l;
            Xfer x = xfer_identity();
            if (r < g.ntr) {
                const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(slot));
                x = unpack_xfer(TileRec{v.x, v.y, v.z, v.w});
            }
            Xfer incl = x;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const Xfer o = shfl_up_xfer(incl, d);
                if ((int)t >= d) incl = xfer_then(o, incl);
            }
            Xfer excl = shfl_up_xfer(incl, 1);
            if (t == 0) excl = xfer_identity();
            if (r < g.ntr) *slot = pack_xfer(excl);  // the tile's effect-before within its chunk
            if (t == 31) a.chunks[(uint64_t)l * C + c] = pack_xfer(incl);
        }
        if (!grid_barrier(&a.ctl->gs, G)) {
            if (threadIdx.x == 0) atomicOr(a.status, KVX_S_TIMEOUT);
            return;
        }
        for (uint64_t q = gw; q < tasks; q += nw) {  // fold the earlier chunks in
            const uint32_t l = (uint32_t)(q / C), c = (uint32_t)(q % C);
            const uint32_t r = c * 32 + t;
            TileRec *slot = a.tiles + (uint64_t)r * L + l;
            const TileRec *tot = a.chunks + (uint64_t)l * C;
            Xfer e = xfer_identity();
            if (r < g.ntr) {
                const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(slot));
                e = unpack_xfer(TileRec{v.x, v.y, v.z, v.w});
            }
            // carry = the lane's prefix before chunk c; end = after chunk c
            Prefix carry{0u, 0u, kNone}, end{0u, 0u, kNone};
            for (uint32_t c0 = 0; c0 <= c; c0 += 32) {
                Xfer x = xfer_identity();
                if (c0 + t <= c) {
                    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(tot + c0 + t));
                    x = unpack_xfer(TileRec{v.x, v.y, v.z, v.w});
                }
                Xfer incl = x;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const Xfer o = shfl_up_xfer(incl, d);
                    if ((int)t >= d) incl = xfer_then(o, incl);
                }
                const uint32_t last = c - c0 < 32 ? c - c0 : 31;  // chunk c, or this group's last
                end = prefix_then(carry, shfl_xfer(incl, (int)last));
                if (c - c0 < 32) {
                    // chunk c is in this group: the prefix before it
                    const Xfer before = shfl_xfer(incl, last ? (int)last - 1 : 0);
                    if (last) carry = prefix_then(carry, before);
                } else {
                    carry = end;
                }
            }
            if (r < g.ntr) {
                const Prefix mine = prefix_then(carry, e);
                *slot = TileRec{mine.state, mine.runs, mine.prev, 0u};
            }
            if (c == C - 1 && t == 0) lane_done(a, l, end.runs);
        }
    }
    if (!grid_barrier(&a.ctl->gs, G)) {
        if (threadIdx.x == 0) atomicOr(a.status, KVX_S_TIMEOUT);
        return;
    }

    // ---- phase 3: lane offsets, then every slice writes its runs
    if (blockIdx.x == 0) {  // total runs
        const uint64_t tot = block_sum_tiles(a.tile_runs, g.ntl, s_red);
        if (threadIdx.x == 0) *a.num_runs = tot;
    }
    for (uint32_t tile = blockIdx.x; tile < ntiles; tile += G) {
        const uint32_t tl = tile % g.ntl, tr = tile / g.ntl;
        const uint32_t l0 = tl * 32, l = l0 + t;
        {   // runs of every lane tile before tl, then a warp scan over the tile's lanes
            const uint64_t base0 = block_sum_tiles(a.tile_runs, tl, s_red);
            if (w == 0) {
                const uint64_t mine = l < L ? __ldcg(a.runs_per_lane + l) : 0;
                uint64_t incl = mine;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if ((int)t >= d) incl += o;
                }
                s_lb[t] = base0 + incl - mine;
            }
        }
        const uint64_t b0 = (uint64_t)tr * kRows * g.K + (uint64_t)w * g.K;
        const uint64_t b1 = b0 + g.K < Bv ? b0 + g.K : Bv;
        const bool active = l < L && b0 < Bv;
        // a block with one tile kept its slice's effect from phase 1
        if (!one_tile) {  // a block with one tile kept its slices' effects and starts from phase 1
            uint64_t m0, m1;
            sx[w][t] = active ? slice_xfer(a.addr, L, l, b0, b1, m0, m1) : xfer_identity();
        }
        __syncthreads();
        if (w == 0 && l < L) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(a.tiles + (uint64_t)tr * L + l));
            Prefix p{v.x, v.y, v.z};
            for (int r = 0; r < kRows; r++) {
                sp[r][t] = p;
                p = prefix_then(p, sx[r][t]);
            }
        }
        __syncthreads();
        if (one_tile) {
            // Runs in table order: warp w writes those of lanes 4w .. 4w+3 of the
            // tile, 32 consecutive runs at a time, so that its stores are
            // contiguous.  Its 32 (lane, slice) pairs are its lanes' slices,
            // one per thread; a run's pair is found by a search over the
            // pairs' run offsets, its block from the pair's start mask.
            static_assert(kRows * 4 == 32, "four lanes of eight slices per warp");
            const uint32_t tt = w * 4 + (t >> 3), r = t & 7;  // this thread's pair
            const uint64_t rb0 = (uint64_t)tr * kRows * g.K + (uint64_t)r * g.K;
            const bool act = l0 + tt < L && rb0 < Bv;
            const Prefix pr = sp[r][tt];
            const uint64_t m = act ? (pr.state ? sm1[r][tt] : sm0[r][tt]) : 0;
            const uint32_t c = (uint32_t)__popcll(m);
            uint32_t incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if ((int)t >= d) incl += o;
            }
            const uint32_t off = incl - c;  // the warp's runs before this pair's
            const uint32_t T = __shfl_sync(0xFFFFFFFFu, incl, 31);
            for (uint32_t q0 = 0; q0 < T; q0 += 32) {
                const uint32_t q = q0 + t;
                uint32_t v = 0;  // the last pair whose runs start at or before run q
#pragma unroll
                for (uint32_t s = 16; s > 0; s >>= 1)
                    if (__shfl_sync(0xFFFFFFFFu, off, v + s) <= q) v += s;
                const uint32_t j = q - __shfl_sync(0xFFFFFFFFu, off, v);
                const uint32_t lane_run0 = __shfl_sync(0xFFFFFFFFu, off, v & ~7u);  // offset of its lane's first pair
                const uint64_t mv = shfl_u64(m, v);
                if (q < T) {
                    const uint32_t tv = w * 4 + (v >> 3), rv = v & 7, lv = l0 + tv;
                    const uint64_t b0v = (uint64_t)tr * kRows * g.K + (uint64_t)rv * g.K;
                    const uint64_t i = b0v + nth_bit(mv, j);
                    const uint64_t av = ld_addr(a.addr, i, L, lv);
                    const uint64_t nx = i + 1 < Bv ? ld_addr(a.addr, i + 1, L, lv) : 0;
                    const uint64_t idx = s_lb[tv] + sp[0][tv].runs + (q - lane_run0);
                    if (idx < a.run_cap) {  // always true: runs per lane <= ceil(B/2)
                        a.run_base[idx] = av;
                        a.run_stride[idx] = i + 1 < Bv ? (int64_t)(nx - av) : 0;
                    }
                    // the run before it in its lane ends here
                    const uint32_t pv = j ? (uint32_t)(b0v + nth_bit(mv, j - 1)) : sp[rv][tv].prev;
                    if (pv != kNone && idx - 1 < a.run_cap) a.run_count[idx - 1] = (uint32_t)(i - pv);
                }
            }
            // the lane's last run, in the slice where the table ends
            if (act && rb0 + g.K >= Bv) {
                const uint32_t last = c ? (uint32_t)(rb0 + 63 - __clzll((long long)m)) : pr.prev;
                const uint64_t li = s_lb[tt] + pr.runs + c - 1;
                if (li < a.run_cap) a.run_count[li] = (uint32_t)(Bv - last);
            }
        } else if (active) {
            const Prefix p = sp[w][t];
            const uint64_t lb = s_lb[t];
            uint32_t runs = p.runs;
            uint32_t prev = p.prev;
            // a run starting at block i: its base and stride, and the block
            // count of the run before it
            auto emit = [&](uint64_t i, uint64_t av, uint64_t nx) {
                const uint64_t idx = lb + runs;
                if (idx < a.run_cap) {  // always true: runs per lane <= ceil(B/2)
                    a.run_base[idx] = av;
                    a.run_stride[idx] = i + 1 < Bv ? (int64_t)(nx - av) : 0;
                }
                if (prev != kNone && idx - 1 < a.run_cap) a.run_count[idx - 1] = (uint32_t)(i - prev);
                prev = (uint32_t)i;
                runs++;
            };
            {
                uint64_t p2 = b0 >= 2 ? ld_addr(a.addr, b0 - 2, L, l) : 0;
                uint64_t p1 = b0 >= 1 ? ld_addr(a.addr, b0 - 1, L, l) : 0;
                uint64_t av = ld_addr(a.addr, b0, L, l);
                uint32_t s = p.state;
                for (uint64_t i = b0; i < b1; i++) {
                    const uint64_t nx = i + 1 < Bv ? ld_addr(a.addr, i + 1, L, l) : 0;
                    uint32_t n;
                    if (i == 0)
                        n = 0;
                    else if (i == 1 || av - p1 == p1 - p2)
                        n = 1;
                    else
                        n = s ^ 1u;
                    if (n == 0) emit(i, av, nx);
                    s = n;
                    p2 = p1;
                    p1 = av;
                    av = nx;
                }
            }
            if (b1 == Bv && lb + runs - 1 < a.run_cap) a.run_count[lb + runs - 1] = (uint32_t)(Bv - prev);
        }
        __syncthreads();
    }
}

// Blocks of k_encode that can be resident at once (cooperative launch limit).
uint32_t encode_max_blocks() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return (uint32_t)cached[dev];
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_encode, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int n = per_sm * sm_count();
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return (uint32_t)n;
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" uint64_t kvx_run_capacity(uint32_t B, uint32_t L) {
    return (uint64_t)L * (((uint64_t)B + 1) / 2);
}

extern "C" size_t kvx_encode_workspace_size(uint32_t B, uint32_t L) {
    size_t bytes = 0;
    carve(nullptr, B, L, &bytes);
    return bytes;
}

namespace kvx {
namespace {

kvx_status launch_encode(const uint64_t *addr, const uint32_t *seg_size, const uint32_t *tmpl_len,
                         uint32_t *prefix, uint32_t B, uint32_t L, uint32_t *runs_per_lane,
                         uint64_t *run_base, int64_t *run_stride, uint32_t *run_count,
                         uint64_t run_capacity, uint64_t *num_runs, uint32_t *status, void *ws,
                         size_t ws_bytes, void *stream) {
    if (!num_runs || !status || !ws || (L && !runs_per_lane) || ((uint64_t)B * L && !addr))
        return KVX_EINVAL;
    if (kvx_run_capacity(B, L) && (!run_base || !run_stride || !run_count)) return KVX_EINVAL;
    if (run_capacity < kvx_run_capacity(B, L)) return KVX_ECAPACITY;
    size_t need = 0;
    Ws w = carve(ws, B, L, &need);
    if (ws_bytes < need) return KVX_EINVAL;
    const Geometry g = geometry(B, L, (uint32_t)sm_count());
    cudaStream_t s = as_stream(stream);
    // the control block and the lane-tile totals (carved right after it) start at zero
    const size_t zero_bytes = reinterpret_cast<char *>(w.tile_runs + g.ntl) - reinterpret_cast<char *>(w.ctl);
    if (cudaMemsetAsync(w.ctl, 0, zero_bytes, s) != cudaSuccess) return KVX_ECUDA;
    EncodeArgs a;
    a.addr = addr;
    a.seg_size = seg_size;
    a.tmpl_len = tmpl_len;
    a.prefix = prefix;
    a.B = B;
    a.L = L;
    a.g = g;
    a.tiles = w.tiles;
    a.chunks = w.chunks;
    a.runs_per_lane = runs_per_lane;
    a.tile_runs = w.tile_runs;
    a.num_runs = num_runs;
    a.run_base = run_base;
    a.run_stride = run_stride;
    a.run_count = run_count;
    a.run_cap = run_capacity;
    a.ctl = w.ctl;
    a.status = status;
    const uint32_t ntiles = g.ntl * g.ntr;
    const uint32_t maxb = encode_max_blocks();
    const uint32_t grid = ntiles < maxb ? ntiles : maxb;
    void *args[] = {&a};
    if (cudaLaunchCooperativeKernel((const void *)k_encode, dim3(grid), dim3(kThreads), args, 0, s) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return KVX_ECUDA;
    }
    note_launch();
    return KVX_OK;
}

}  // namespace
}  // namespace kvx

extern "C" kvx_status kvx_encode_runs(const uint64_t *addr, uint32_t B, uint32_t L,
                                      uint32_t *runs_per_lane, uint64_t *run_base,
                                      int64_t *run_stride, uint32_t *run_count,
                                      uint64_t run_capacity, uint64_t *num_runs,
                                      uint32_t *status, void *ws, size_t ws_bytes,
                                      void *stream) {
    return launch_encode(addr, nullptr, nullptr, nullptr, B, L, runs_per_lane, run_base,
                         run_stride, run_count, run_capacity, num_runs, status, ws, ws_bytes,
                         stream);
}

extern "C" kvx_status kvx_verify_encode(const uint64_t *addr, const uint32_t *seg_size,
                                        const uint32_t *seg_len, uint32_t B, uint32_t L,
                                        uint32_t *prefix_blocks, uint32_t *runs_per_lane,
                                        uint64_t *run_base, int64_t *run_stride,
                                        uint32_t *run_count, uint64_t run_capacity,
                                        uint64_t *num_runs, uint32_t *status, void *ws,
                                        size_t ws_bytes, void *stream) {
    if (!prefix_blocks || (L && !seg_len) || ((uint64_t)B * L && !seg_size)) return KVX_EINVAL;
    return launch_encode(addr, seg_size, seg_len, prefix_blocks, B, L, runs_per_lane, run_base,
                         run_stride, run_count, run_capacity, num_runs, status, ws, ws_bytes,
                         stream);
}
