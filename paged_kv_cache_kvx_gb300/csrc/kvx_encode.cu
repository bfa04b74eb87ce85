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
// Thread layout: a CTA is 8 warps; lane t of warp w handles table lane
// l0 + t over blocks [tile_b0 + w*K, +K), so every warp load is one
// coalesced 256-byte row segment of the block-major table.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kRows = 8;           // warps per CTA = row slices per tile
constexpr int kThreads = 32 * kRows;
constexpr uint32_t kTargetCtas = 1024;

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

// a then b
__device__ __forceinline__ Xfer xfer_then(const Xfer &a, const Xfer &b) {
    Xfer c;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const uint32_t e1 = a.fin[e];
        c.cnt[e] = a.cnt[e] + b.cnt[e1];
        c.last[e] = b.last[e1] != kNone ? b.last[e1] : a.last[e];
        c.fin[e] = b.fin[e1];
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
    q.state = x.fin[p.state];
    q.runs = p.runs + x.cnt[p.state];
    q.prev = x.last[p.state] != kNone ? x.last[p.state] : p.prev;
    return q;
}

// Per-lane tile records in the workspace: first the tile's Xfer, then (after
// the last block's scan) the tile's entry Prefix.
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
    uint32_t ticket;
};

__device__ __forceinline__ uint64_t ld_addr(const uint64_t *addr, uint64_t b, uint32_t L, uint32_t l) {
    return __ldg(addr + b * L + l);
}

// Slice [b0, b1) of lane l under both entry states.
__device__ Xfer slice_xfer(const uint64_t *addr, uint32_t L, uint32_t l, uint64_t b0, uint64_t b1) {
    Xfer x = xfer_identity();
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
        if (n0 == 0) { x.cnt[0]++; x.last[0] = (uint32_t)i; }
        if (n1 == 0) { x.cnt[1]++; x.last[1] = (uint32_t)i; }
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

Geometry geometry(uint32_t B, uint32_t L) {
    Geometry g;
    g.ntl = (uint32_t)ceil_div(L ? L : 1, 32);
    g.K = 8;
    while (g.K < 64 && (uint64_t)g.ntl * ceil_div(B ? B : 1, (uint64_t)kRows * g.K) > kTargetCtas)
        g.K *= 2;
    g.ntr = (uint32_t)ceil_div(B ? B : 1, (uint64_t)kRows * g.K);
    return g;
}

struct Ws {
    EncodeCtl *ctl;
    TileRec *tiles;       // [ntr][L]
    uint64_t *lane_base;  // [L]
};

Ws carve(void *base, uint32_t B, uint32_t L, size_t *bytes) {
    Geometry g = geometry(B, L);
    Carver c(base);
    Ws w;
    w.ctl = c.take<EncodeCtl>(1);
    w.tiles = c.take<TileRec>((size_t)g.ntr * L);
    w.lane_base = c.take<uint64_t>(L);
    *bytes = c.off;
    return w;
}

// Pass 1: per-(tile, lane) Xfer; the last block scans tiles per lane into
// entry prefixes, writes runs_per_lane, scans lanes into run offsets.
__global__ void __launch_bounds__(kThreads)
k_encode_tiles(const uint64_t *__restrict__ addr, uint32_t B, uint32_t L, Geometry g,
               TileRec *__restrict__ tiles, uint64_t *__restrict__ lane_base,
               uint32_t *__restrict__ runs_per_lane, uint64_t *__restrict__ num_runs,
               EncodeCtl *ctl) {
    __shared__ Xfer sx[kRows][32];
    const uint32_t tl = blockIdx.x % g.ntl, tr = blockIdx.x / g.ntl;
    const uint32_t t = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t l = tl * 32 + t;
    const uint64_t tb0 = (uint64_t)tr * kRows * g.K;
    const uint64_t b0 = tb0 + (uint64_t)w * g.K;
    const uint64_t b1 = b0 + g.K < B ? b0 + g.K : B;
    Xfer x = xfer_identity();
    if (l < L && b0 < B) x = slice_xfer(addr, L, l, b0, b1);
    sx[w][t] = x;
    __syncthreads();
    if (w == 0 && l < L) {
        Xfer acc = sx[0][t];
        for (int r = 1; r < kRows; r++) acc = xfer_then(acc, sx[r][t]);
        tiles[(uint64_t)tr * L + l] = pack_xfer(acc);
    }
    if (!last_block(&ctl->ticket)) return;

    // Last block: per lane, tiles in order -> entry prefixes.  Records are
    // loaded in batches before they are combined and overwritten, so the
    // loads of a batch are in flight together.
    constexpr uint32_t kBatch = 8;
    for (uint32_t lane = threadIdx.x; lane < L; lane += blockDim.x) {
        Prefix p{0u, 0u, kNone};
        for (uint32_t r0 = 0; r0 < g.ntr; r0 += kBatch) {
            uint4 v[kBatch];
#pragma unroll
            for (uint32_t j = 0; j < kBatch; j++)
                if (r0 + j < g.ntr)
                    v[j] = __ldcg(reinterpret_cast<const uint4 *>(tiles + (uint64_t)(r0 + j) * L + lane));
#pragma unroll
            for (uint32_t j = 0; j < kBatch; j++) {
                if (r0 + j >= g.ntr) break;
                const Xfer xr = unpack_xfer(TileRec{v[j].x, v[j].y, v[j].z, v[j].w});
                tiles[(uint64_t)(r0 + j) * L + lane] = TileRec{p.state, p.runs, p.prev, 0u};
                p = prefix_then(p, xr);
            }
        }
        runs_per_lane[lane] = p.runs;
        lane_base[lane] = p.runs;
    }
    __syncthreads();
    const uint64_t total = block_scan_inplace_u64(lane_base, L);
    if (threadIdx.x == 0) *num_runs = total;
}

// Pass 2: recompute each thread's slice, resolve its entry prefix from the
// tile prefix, and write the runs that start inside the slice.  The count of
// a run is written by the thread that meets the next start (or the lane's
// end).
__global__ void __launch_bounds__(kThreads)
k_encode_emit(const uint64_t *__restrict__ addr, uint32_t B, uint32_t L, Geometry g,
              const TileRec *__restrict__ tiles, const uint64_t *__restrict__ lane_base,
              uint64_t *__restrict__ run_base, int64_t *__restrict__ run_stride,
              uint32_t *__restrict__ run_count, uint64_t run_cap) {
    __shared__ Xfer sx[kRows][32];
    __shared__ Prefix sp[kRows][32];
    const uint32_t tl = blockIdx.x % g.ntl, tr = blockIdx.x / g.ntl;
    const uint32_t t = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t l = tl * 32 + t;
    const uint64_t tb0 = (uint64_t)tr * kRows * g.K;
    const uint64_t b0 = tb0 + (uint64_t)w * g.K;
    const uint64_t b1 = b0 + g.K < B ? b0 + g.K : B;
    const bool active = l < L && b0 < B;
    sx[w][t] = active ? slice_xfer(addr, L, l, b0, b1) : xfer_identity();
    __syncthreads();
    if (w == 0 && l < L) {
        const TileRec tp = tiles[(uint64_t)tr * L + l];
        Prefix p{tp.a, tp.b, tp.c};
        for (int r = 0; r < kRows; r++) {
            sp[r][t] = p;
            p = prefix_then(p, sx[r][t]);
        }
    }
    __syncthreads();
    if (!active) return;

    Prefix p = sp[w][t];
    const uint64_t lb = lane_base[l];
    uint64_t p2 = b0 >= 2 ? ld_addr(addr, b0 - 2, L, l) : 0;
    uint64_t p1 = b0 >= 1 ? ld_addr(addr, b0 - 1, L, l) : 0;
    uint64_t a = ld_addr(addr, b0, L, l);
    uint32_t s = p.state;
    uint32_t runs = p.runs;
    uint32_t prev = p.prev;
    for (uint64_t i = b0; i < b1; i++) {
        const uint64_t nx = i + 1 < B ? ld_addr(addr, i + 1, L, l) : 0;
        uint32_t n;
        if (i == 0)
            n = 0;
        else if (i == 1 || a - p1 == p1 - p2)
            n = 1;
        else
            n = s ^ 1u;
        if (n == 0) {
            const uint64_t idx = lb + runs;
            if (idx < run_cap) {  // always true: runs per lane <= ceil(B/2)
                run_base[idx] = a;
                run_stride[idx] = i + 1 < B ? (int64_t)(nx - a) : 0;
            }
            if (prev != kNone && idx - 1 < run_cap) run_count[idx - 1] = (uint32_t)(i - prev);
            prev = (uint32_t)i;
            runs++;
        }
        s = n;
        p2 = p1;
        p1 = a;
        a = nx;
    }
    if (b1 == B && lb + runs - 1 < run_cap) run_count[lb + runs - 1] = (uint32_t)(B - prev);
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

extern "C" kvx_status kvx_encode_runs(const uint64_t *addr, uint32_t B, uint32_t L,
                                      uint32_t *runs_per_lane, uint64_t *run_base,
                                      int64_t *run_stride, uint32_t *run_count,
                                      uint64_t run_capacity, uint64_t *num_runs, void *ws,
                                      size_t ws_bytes, void *stream) {
    if (!num_runs || !ws || (L && !runs_per_lane) || ((uint64_t)B * L && !addr))
        return KVX_EINVAL;
    if (kvx_run_capacity(B, L) && (!run_base || !run_stride || !run_count)) return KVX_EINVAL;
    if (run_capacity < kvx_run_capacity(B, L)) return KVX_ECAPACITY;
    size_t need = 0;
    Ws w = carve(ws, B, L, &need);
    if (ws_bytes < need) return KVX_EINVAL;
    const Geometry g = geometry(B, L);
    cudaStream_t s = as_stream(stream);
    if (cudaMemsetAsync(w.ctl, 0, sizeof(EncodeCtl), s) != cudaSuccess) return KVX_ECUDA;
    const uint32_t grid = g.ntl * g.ntr;
    k_encode_tiles<<<grid, kThreads, 0, s>>>(addr, B, L, g, w.tiles, w.lane_base, runs_per_lane,
                                             num_runs, w.ctl);
    KVX_LAUNCHED();
    if (B && L) {
        k_encode_emit<<<grid, kThreads, 0, s>>>(addr, B, L, g, w.tiles, w.lane_base, run_base,
                                                run_stride, run_count, run_capacity);
        KVX_LAUNCHED();
    }
    return KVX_OK;
}
