// Transfer planning (pegaflow PR #350, Requester plan_transfer steps 1-4 and
// the READ splitting paragraph) as one cooperative kernel whose phases are
// separated by a bounded grid barrier:
//
//   init      step 1, table level: lane count, zero-size slots, empty lanes,
//             lane_first = prefix of runs_per_lane, arrays in sync, slab size
//   decode    step 1 per run (zero count, one-block stride, span); the lane of
//             each run; per-tile sums for the per-lane block prefix; the key
//             bits that differ (which radix digits are active)
//   keys      step 2: first block of each run (segmented prefix of counts in
//             its lane), per-lane coverage, sort items, first radix histogram
//   hist      (2048-run tiles) before every radix pass but the first: the
//             pass's per-tile histograms, counted in shared memory
//   sort      step 2: stable LSD radix passes on (node, base) over the active
//             digits, one barrier each; equal keys keep run order = (lane,
//             first block) order.  The smaller tile bodies count the next
//             pass's histograms with atomics as they scatter
//   post-sort step 3: sorted records; compat(p) = same node, first block,
//             count and stride as p-1 and base-adjacent to it; group starts,
//             with the "grown chunk still fits the stride" cut inside a
//             compatible stretch.  With 2048-run tiles the same phase goes on
//             to the groups and the carve: each tile publishes its group
//             count, then its bytes and reads, behind flags, and takes the
//             earlier tiles' totals by looking back at theirs
//   cut,      only when some stretch outgrows its stride: the cut again with
//   count     walks along such stretches in order, then the counts again
//   groups    (smaller tiles, or after the walks) group records, run_group /
//             run_off, bytes and read pieces
//   emit      step 4: slab carve (groups back to back) and descriptors (one
//             per dense group / per block, split at 32 MiB)
//
// Runs are cut into tiles of 512, 1024 or 2048 (2, 4 or 8 per thread of a
// 256-thread block): the smallest whose tiles all get a block.  Only as many
// blocks as there are tiles take part, each owning tiles b, b+P, ...; when the
// grid has two blocks per SM and there is at most a tile per SM, the first
// block to start on each SM takes part, so no two working blocks share one.
// A block gets the carry for its tile by an ordered reduction of the earlier
// tiles' aggregates, so scans cost no extra barrier.  Every read of data
// another block wrote in this kernel bypasses L1.  Tables of up to 2048 runs
// (every bump-allocated holder of up to 1024 slots) go to k_plan_small, one
// block with the table in shared memory, and this kernel returns at once.
#include <atomic>

#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kT = 256;
// Runs per thread: 8 (2048-run tiles) in general; 4 or 2 (1024- or 512-run
// tiles) for tables small enough that every such tile still has a block of
// its own: each phase's per-thread chains shrink, and no block takes a second
// tile.  The smaller tiles serve at most kSmallTiles tiles, which bounds the
// per-tile workspace.
constexpr int kIPT = 8;
constexpr uint32_t kTile = kT * kIPT;

// Where a radix pass after the first gets its histograms.  2048-run tiles:
// from a phase of their own before the pass (each block counts its own tiles
// in shared memory, a grid barrier, then the pass), where the previous pass's
// scatter would pay two global atomics per run (tile and tile-group rows).
// Smaller tiles (tables of a few dozen): from those atomics during the
// previous pass's scatter, which cost less there than the extra barrier.
template <int IPT>
constexpr bool kLocalHist = IPT == kIPT;

constexpr uint64_t kSmallTiles = 256;
constexpr uint32_t kDigits = 256;
// Radix histograms are also kept summed over groups of this many tiles, so a
// tile's digit offsets take the groups before its own plus at most
// kHistGroup - 1 tiles of its own group, instead of every earlier tile.
constexpr uint32_t kHistGroup = 8;

struct PlanCtl {
    GridSync gs;
    uint32_t fail;
    uint32_t st;
    uint32_t walked;  // a stretch walker of the cut phase set flags beyond its own position
    unsigned long long or_base, and_base;
    uint32_t or_node, and_node;
    uint32_t or_empty, and_empty;  // some / every run has a zero-size segment
    uint32_t primaries;            // blocks that came first on their SM (two blocks per SM, small tables)
    uint32_t sm_rank[256];         // per SM id: planner blocks that have started there
};

// Sort record; r holds the run index in its low 31 bits and, in the top bit,
// whether the run's segments are empty (zero-size V lane).
struct __align__(16) SortItem {
    uint64_t base;
    uint32_t node;
    uint32_t r;
};

constexpr uint32_t kEmptyBit = 1u << 31;
constexpr uint32_t kEmptyDigit = 12;  // radix digit of the empty flag

__device__ __forceinline__ uint32_t item_run(const SortItem &it) { return it.r & ~kEmptyBit; }

struct __align__(16) Rec {
    uint64_t base;
    int64_t stride;
    uint32_t len, block, count, node, r, pad;
};

// Segmented sum: value since the last segment head, and whether a head was seen.
struct __align__(16) Seg {
    uint64_t sum;
    uint32_t head;
    uint32_t pad;
};
struct SegOp {
    __device__ Seg operator()(const Seg &a, const Seg &b) const {
        return Seg{b.head ? b.sum : a.sum + b.sum, a.head | b.head, 0};
    }
};
struct MaxOp {
    __device__ int64_t operator()(int64_t a, int64_t b) const { return a > b ? a : b; }
};
// Group numbering: starts so far and position of the last start.
struct __align__(16) GAgg {
    uint64_t n;
    int64_t last;
};
struct GOp {
    __device__ GAgg operator()(const GAgg &a, const GAgg &b) const {
        return GAgg{a.n + b.n, a.last > b.last ? a.last : b.last};
    }
};
// Carve: slab bytes and descriptor count so far.
struct __align__(16) CAgg {
    uint64_t bytes;
    uint64_t descs;
};
struct COp {
    __device__ CAgg operator()(const CAgg &a, const CAgg &b) const {
        return CAgg{a.bytes + b.bytes, a.descs + b.descs};
    }
};

struct PlanArgs {
    const uint32_t *rpl;
    uint32_t table_lanes;
    uint32_t template_lanes;
    const uint64_t *run_base;
    const int64_t *run_stride;
    const uint32_t *run_count;
    const uint64_t *num_runs;
    uint64_t run_cap;
    uint32_t B;
    const uint32_t *seg_len;
    const uint32_t *numa;
    uint64_t pool_bytes;
    kvx_group *groups;
    uint64_t group_cap;
    kvx_desc *descs;
    uint64_t desc_cap;
    uint32_t *lane_first;
    uint32_t *run_block;
    uint32_t *run_group;
    uint64_t *run_off;
    uint64_t *counts;
    uint32_t *status;
    uint32_t out16;  // groups and descs start on 16-byte boundaries: records move in 16-byte pieces
    uint32_t sms;    // the device's SMs
    // workspace
    PlanCtl *ctl;
    uint32_t *run_lane;
    Seg *seg;
    SortItem *items0, *items1;
    uint32_t *hist[3];   // [tile][digit]
    uint32_t *ghist[3];  // [tile group][digit]: the same counts summed over groups of kHistGroup tiles
    uint64_t *run_bl;  // per run: its first block (low word), its lane's segment length (high word)
    uint8_t *compat;
    uint8_t *gflag;
    int64_t *segmax;
    GAgg *gagg;
    CAgg *cagg;
    GAgg *gthr;  // per tile and thread: groups before the thread's first run
    CAgg *cthr;  // per tile and thread: carve prefix inside the tile
    uint32_t *ready_g;  // per tile: gagg (and the tile's first group flag) published, 2 = abandoned
    uint32_t *ready_c;  // per tile: cagg published, 2 = abandoned
};

// The block's index among the planner's working blocks, which every phase
// takes as vb: blockIdx.x, except that with two blocks per SM a table of at
// most one tile per SM takes one block per distinct SM (the first to start
// there, numbered in arrival order).
__shared__ uint32_t g_vb;

union ScanSmem {
    Seg seg[kT];
    int64_t i64[kT];
    GAgg g[kT];
    CAgg c[kT];
};

// Shuffle of any 4-byte-multiple value, one 32-bit word at a time.
template <class T>
__device__ __forceinline__ T shfl_up_words(const T &v, int d) {
    static_assert(sizeof(T) % 4 == 0, "4-byte multiple");
    T o;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(&v);
    uint32_t *dst = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); i++) dst[i] = __shfl_up_sync(0xFFFFFFFFu, src[i], d);
    return o;
}

// Block scan (blockDim a multiple of 32, at most 1024): warp-shuffle scans,
// then one warp scans the warp totals through shared memory -- three block
// barriers.  Returns the inclusive value; *excl gets the exclusive one,
// *total the block total.  sh holds at least 32 elements.
template <class T, class Op>
__device__ T block_scan(T v, Op op, T identity, T *sh, T *excl, T *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    T x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T o = shfl_up_words(x, d);
        if (lane >= d) x = op(o, x);
    }
    __syncthreads();  // sh may still be read from a previous scan
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        T t = lane < nw ? sh[lane] : identity;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const T o = shfl_up_words(t, d);
            if (lane >= d) t = op(o, t);
        }
        sh[lane] = t;
    }
    __syncthreads();
    const T before = w > 0 ? sh[w - 1] : identity;
    const T in_warp = shfl_up_words(x, 1);
    *excl = lane > 0 ? op(before, in_warp) : before;
    *total = sh[nw - 1];
    return op(before, x);
}

// Seg over a warp in lane order: the fold of all 32 values (every lane gets
// it), and each lane's inclusive prefix.
__device__ __forceinline__ Seg shfl_seg(const Seg &v, int src, bool down, int d) {
    Seg o;
    const uint32_t lo = (uint32_t)v.sum, hi = (uint32_t)(v.sum >> 32);
    const uint32_t l2 = down ? __shfl_down_sync(0xFFFFFFFFu, lo, d) : __shfl_sync(0xFFFFFFFFu, lo, src);
    const uint32_t h2 = down ? __shfl_down_sync(0xFFFFFFFFu, hi, d) : __shfl_sync(0xFFFFFFFFu, hi, src);
    o.head = down ? __shfl_down_sync(0xFFFFFFFFu, v.head, d) : __shfl_sync(0xFFFFFFFFu, v.head, src);
    o.sum = (uint64_t)h2 << 32 | l2;
    o.pad = 0;
    return o;
}
__device__ __forceinline__ Seg warp_fold_seg(Seg v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Seg o = shfl_seg(v, 0, true, d);
        if (lane + d < 32) v = SegOp()(v, o);
    }
    return shfl_seg(v, 0, false, 0);
}
__device__ __forceinline__ Seg warp_scan_seg(Seg v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Seg o = shfl_up_words(v, d);
        if (lane >= d) v = SegOp()(o, v);
    }
    return v;
}

// Ordered reduction of agg[0, t) by the whole block (the carry into tile t).
template <class T, class Op>
__device__ T reduce_prefix(const T *agg, uint64_t t, Op op, T identity, T *sh) {
    const uint64_t per = (t + blockDim.x - 1) / blockDim.x;
    const uint64_t lo = per * threadIdx.x;
    const uint64_t hi = lo + per < t ? lo + per : t;
    T v = identity;
    for (uint64_t i = lo; i < hi; i++) v = op(v, ld_cg(agg + i));
    T ex, tot;
    block_scan(v, op, identity, sh, &ex, &tot);
    return tot;
}

// Radix digits of the sort key (node, empty, base), empty = the run's segments
// have length 0 (such runs come after the others of their node).
//
// Packed form (the usual one): only the bit ranges in which the keys differ
// matter, so the key is re-packed as node bits | empty bit | base bits, each
// field cut to its differing range (every key agrees outside it, so the order
// is unchanged), and sorted 8 bits at a time.  A digit descriptor then holds
// kPacked, the digit index (bits 0-2) and the layout: base shift (3-8) and
// width (9-15), empty width (16), node shift (17-21) and width (22-27).
// Byte form (keys wider than 64 bits once packed): 0-7 base bytes, 8-11 node
// bytes, kEmptyDigit the empty flag.
constexpr uint32_t kPacked = 1u << 31;

__device__ __forceinline__ uint64_t low_mask(uint32_t w) { return w >= 64 ? ~0ull : (1ull << w) - 1; }

__device__ __forceinline__ uint32_t digit_of(uint64_t base, uint32_t node, uint32_t empty, uint32_t dig) {
    if (dig & kPacked) {
        const uint32_t k = dig & 7u, lo_b = (dig >> 3) & 63u, wb = (dig >> 9) & 127u;
        const uint32_t we = (dig >> 16) & 1u, lo_n = (dig >> 17) & 31u, wn = (dig >> 22) & 63u;
        uint64_t key = wb ? (base >> lo_b) & low_mask(wb) : 0;
        if (we) key |= (uint64_t)empty << wb;  // wb < 64 whenever we = 1
        if (wn) key |= (uint64_t)((node >> lo_n) & low_mask(wn)) << (wb + we);
        return (uint32_t)(key >> (8 * k)) & 0xFFu;
    }
    if (dig < 8) return (uint32_t)(base >> (8 * dig)) & 0xFFu;
    if (dig == kEmptyDigit) return empty;
    return (node >> (8 * (dig - 8))) & 0xFFu;
}

// Lanes of the warp whose digit equals this lane's (digits below kDigits;
// a lane holding kDigits or more matches nobody and gets no meaningful
// mask): one ballot per digit bit, so the cost does not grow with the number
// of distinct digits in the warp (random keys have nearly 32).
__device__ __forceinline__ uint32_t digit_peers(uint32_t d) {
    uint32_t m = __ballot_sync(0xFFFFFFFFu, d < kDigits);
#pragma unroll
    for (int b = 0; b < 8; b++) {
        const uint32_t bit = (d >> b) & 1u;
        const uint32_t bb = __ballot_sync(0xFFFFFFFFu, bit);
        m &= bit ? bb : ~bb;
    }
    return m;
}

// H[key] += 1 for every lane whose key is not ~0u, with one atomic per run of
// equal keys in consecutive lanes (sorted or structured keys come in runs;
// random ones cost one atomic each, without a matching step).
__device__ __forceinline__ void add_key_runs(uint32_t *H, uint32_t key, uint32_t lane) {
    const uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, key, 1);
    const uint32_t bnd = __ballot_sync(0xFFFFFFFFu, lane == 0 || prev != key);
    if (key != ~0u && (bnd >> lane & 1u)) {
        const uint32_t after = bnd & ~((2u << lane) - 1u);  // run boundaries after this lane
        const uint32_t next = after ? (uint32_t)__ffs((int)after) - 1u : 32u;
        atomicAdd(&H[key], next - lane);
    }
}

// The radix passes for keys whose bits differ as in db (base), de (empty), dn
// (node): least significant digit first.  Returns the number of passes.
__device__ __forceinline__ uint32_t plan_digits(uint64_t db, uint32_t de, uint32_t dn, uint32_t *act) {
    const uint32_t lo_b = db ? __ffsll((long long)db) - 1 : 0;
    const uint32_t wb = db ? 64 - __clzll((long long)db) - lo_b : 0;
    const uint32_t we = de ? 1 : 0;
    const uint32_t lo_n = dn ? __ffs((int)dn) - 1 : 0;
    const uint32_t wn = dn ? 32 - __clz((int)dn) - lo_n : 0;
    const uint32_t W = wb + we + wn;
    uint32_t n = 0;
    if (W <= 64) {
        const uint32_t layout = kPacked | lo_b << 3 | wb << 9 | we << 16 | lo_n << 17 | wn << 22;
        for (uint32_t k = 0; k * 8 < W; k++) act[n++] = layout | k;
    } else {
        for (uint32_t d = 0; d < 8; d++)
            if ((db >> (8 * d)) & 0xFFu) act[n++] = d;
        if (de) act[n++] = kEmptyDigit;
        for (uint32_t d = 0; d < 4; d++)
            if ((dn >> (8 * d)) & 0xFFu) act[n++] = 8 + d;
    }
    return n;
}

// Largest l with lane_first[l] <= r (lane_first has L + 1 entries).
template <class Get>
__device__ __forceinline__ uint32_t lane_of(Get lane_first, uint32_t L, uint64_t r) {
    uint32_t lo = 0, hi = L;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if ((uint64_t)lane_first(mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// lane_first is staged in shared memory when it fits (every template with up
// to 4095 lanes); larger tables search it in global memory.
constexpr uint32_t kLaneSmem = 4096;

__device__ __forceinline__ bool group_dense(uint32_t count, int64_t stride, uint64_t chunk) {
    return count == 1 || (stride > 0 && chunk == (uint64_t)stride);
}

__device__ __forceinline__ uint64_t group_pieces(const kvx_group &g) {
    if (g.dense) return ceil_div((uint64_t)g.count * g.chunk, KVX_MAX_READ_BYTES);
    return (uint64_t)g.count * ceil_div(g.chunk, KVX_MAX_READ_BYTES);
}

__device__ __forceinline__ bool compatible(const Rec &prev, const Rec &x) {
    return x.node == prev.node && x.block == prev.block && x.count == prev.count &&
           x.stride == prev.stride && x.base == prev.base + prev.len;
}

__device__ __forceinline__ void raise_plan(const PlanArgs &a, uint32_t bits) {
    if (bits) {
        atomicOr(a.status, bits);
        atomicOr(&a.ctl->st, bits);
    }
}

// Group and descriptor records in the caller's arrays: three or two 16-byte
// pieces when the arrays are 16-byte aligned (fewer, wider stores), else the
// plain struct copy.
__device__ __forceinline__ uint4 u4(uint64_t x, uint64_t y) {
    return make_uint4((uint32_t)x, (uint32_t)(x >> 32), (uint32_t)y, (uint32_t)(y >> 32));
}
__device__ __forceinline__ void st_group(const PlanArgs &a, uint64_t gid, const kvx_group &G) {
    if (a.out16) {
        uint4 *dst = reinterpret_cast<uint4 *>(a.groups + gid);
        dst[0] = u4(G.base, (uint64_t)G.stride);
        dst[1] = u4(G.chunk, G.local);
        dst[2] = make_uint4(G.block, G.count, G.node, G.dense);
    } else {
        a.groups[gid] = G;
    }
}
__device__ __forceinline__ kvx_group ld_group(const PlanArgs &a, uint64_t gid) {
    if (!a.out16) return ld_cg(a.groups + gid);
    const uint4 *src = reinterpret_cast<const uint4 *>(a.groups + gid);
    const uint4 p0 = __ldcg(src), p1 = __ldcg(src + 1), p2 = __ldcg(src + 2);
    kvx_group G;
    G.base = (uint64_t)p0.x | (uint64_t)p0.y << 32;
    G.stride = (int64_t)((uint64_t)p0.z | (uint64_t)p0.w << 32);
    G.chunk = (uint64_t)p1.x | (uint64_t)p1.y << 32;
    G.local = (uint64_t)p1.z | (uint64_t)p1.w << 32;
    G.block = p2.x;
    G.count = p2.y;
    G.node = p2.z;
    G.dense = p2.w;
    return G;
}
__device__ __forceinline__ void st_desc(const PlanArgs &a, uint64_t d, uint64_t remote, uint64_t local,
                                        uint64_t len, uint32_t gid) {
    if (a.out16) {
        uint4 *dst = reinterpret_cast<uint4 *>(a.descs + d);
        dst[0] = u4(remote, local);
        dst[1] = make_uint4((uint32_t)len, (uint32_t)(len >> 32), gid, 0u);
    } else {
        a.descs[d] = kvx_desc{remote, local, len, gid, 0};
    }
}

// ------------------------------------------------------------------ phases

// Step 1, table level (one block).
__device__ void phase_init(const PlanArgs &a, uint64_t R) {
    __shared__ uint64_t sh[33];
    __shared__ uint32_t s_bits;
    const uint32_t tid = threadIdx.x;
    PlanCtl *ctl = a.ctl;
    if (tid == 0) {
        s_bits = 0;
        ctl->or_base = 0;
        ctl->and_base = ~0ull;
        ctl->or_node = 0;
        ctl->and_node = ~0u;
        ctl->or_empty = 0;
        ctl->and_empty = 1;
        a.counts[0] = a.counts[1] = a.counts[2] = 0;
    }
    __syncthreads();
    uint32_t fail = 0, bits = 0;
    if (a.table_lanes != a.template_lanes) {
        bits = KVX_S_LANES;
        fail = 1;
    } else {
        const uint32_t L = a.table_lanes;
        uint64_t carry = 0, lensum = 0;
        uint32_t mybits = 0;
        for (uint32_t base = 0; base < L; base += blockDim.x) {
            const uint32_t i = base + tid;
            uint64_t v = 0;
            if (i < L) {
                v = a.rpl[i];
                const uint32_t len = a.seg_len[i];
                if (len == 0 && (i & 1u) == 0) mybits |= KVX_S_ZERO_LEN;  // zero-size K slot
                if (v == 0 && a.B > 0) mybits |= KVX_S_COVERAGE;
                lensum += len;
            }
            uint64_t tot;
            const uint64_t ex = block_excl_sum<uint64_t>(v, sh, &tot);
            if (i < L) a.lane_first[i] = (uint32_t)(carry + ex);
            carry += tot;
        }
        mybits = __reduce_or_sync(0xFFFFFFFFu, mybits);
        if ((tid & 31) == 0 && mybits) atomicOr(&s_bits, mybits);
        uint64_t lentot;
        block_excl_sum<uint64_t>(lensum, sh, &lentot);
        __syncthreads();
        if (tid == 0) a.lane_first[L] = (uint32_t)carry;
        bits = s_bits;
        if (carry != R || R > a.run_cap) {
            bits |= KVX_S_ARRAYS;
            fail = 1;
        } else {
            const unsigned __int128 slab = (unsigned __int128)a.B * (unsigned __int128)lentot;
            if (slab >= ((unsigned __int128)1 << 63)) {
                bits |= KVX_S_CAPACITY;
                fail = 1;
            }
        }
    }
    if (tid == 0) {
        if (bits) atomicOr(a.status, bits);
        ctl->st = bits;
        ctl->fail = fail;
    }
}

// Step 1 per run; lanes; per-tile segmented count sums; key bits.
template <int IPT>
__device__ void phase_decode(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb, ScanSmem &sm,
                             uint32_t *s_lf) {
    __shared__ uint32_t s_bits;
    __shared__ unsigned long long s_or, s_and;
    __shared__ uint32_t s_orn, s_andn;
    const uint32_t L = a.table_lanes;
    const bool lf_smem = L + 1 <= kLaneSmem;
    if (lf_smem)
        for (uint32_t i = threadIdx.x; i <= L; i += blockDim.x) s_lf[i] = __ldcg(a.lane_first + i);
    if (threadIdx.x == 0) {
        s_bits = 0;
        s_or = 0;
        s_and = ~0ull;
        s_orn = 0;
        s_andn = ~0u;
    }
    __syncthreads();
    {   // the keys phase sums its first histogram into ghist[0]; the post-sort
        // phase publishes per-tile totals behind these flags
        const uint64_t n = (uint64_t)kDigits * ceil_div((uint64_t)nt, (uint64_t)kHistGroup);
        for (uint64_t i = (uint64_t)vb * blockDim.x + threadIdx.x; i < n;
             i += (uint64_t)P * blockDim.x)
            a.ghist[0][i] = 0;
        for (uint64_t i = (uint64_t)vb * blockDim.x + threadIdx.x; i < nt;
             i += (uint64_t)P * blockDim.x) {
            a.ready_g[i] = 0;
            a.ready_c[i] = 0;
        }
    }
    uint32_t bits = 0;
    unsigned long long o = 0, an = ~0ull;
    uint32_t on = 0, ann = ~0u, oe = 0, ae = 1;
    // Each warp takes 32 * IPT consecutive runs of the tile, run j * 32 + lane
    // for its lane (coalesced loads and stores); the tile's segmented count
    // total is folded in run order, warp by warp.
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (uint32_t tile = vb; tile < nt; tile += P) {
        const uint64_t r0 = (uint64_t)tile * (kT * IPT) + (uint64_t)w * (32 * IPT) + lane;
        // all loads of this thread's runs first, then the checks
        uint32_t lanes[IPT], cnts[IPT], lens[IPT], nodes[IPT];
        uint64_t bases[IPT];
        int64_t strides[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t r = r0 + (uint64_t)j * 32;
            lanes[j] = 0;
            if (r < R) {
                lanes[j] = lf_smem ? lane_of([&](uint32_t i) { return s_lf[i]; }, L, r)
                                   : lane_of([&](uint32_t i) { return __ldcg(a.lane_first + i); }, L, r);
                bases[j] = a.run_base[r];
                strides[j] = a.run_stride[r];
                cnts[j] = a.run_count[r];
            }
        }
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            if (r0 + (uint64_t)j * 32 < R) {
                lens[j] = __ldg(a.seg_len + lanes[j]);
                nodes[j] = __ldg(a.numa + lanes[j]);
            }
        }
        Seg wagg{0, 0, 0};  // this warp's runs so far, in order
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t r = r0 + (uint64_t)j * 32;
            Seg s{0, 0, 0};
            if (r < R) {
                const uint32_t l = lanes[j];
                a.run_lane[r] = l;
                const uint64_t base = bases[j];
                const int64_t stride = strides[j];
                const uint32_t cnt = cnts[j];
                const uint32_t len = lens[j];
                const uint32_t node = nodes[j];
                if (cnt == 0) bits |= KVX_S_ZERO_COUNT;
                if (cnt == 1 && stride != 0) bits |= KVX_S_STRIDE1;
                if (cnt >= 1) {
                    const __int128 first = (__int128)base;
                    const __int128 last = first + (__int128)(cnt - 1) * (__int128)stride;
                    const __int128 hi = last > first ? last : first;
                    if (last < 0 || hi + (__int128)len > (__int128)a.pool_bytes) bits |= KVX_S_SPAN;
                }
                const bool head = r == (lf_smem ? s_lf[l] : __ldcg(a.lane_first + l));
                s = Seg{cnt, head ? 1u : 0u, 0};
                o |= base;
                an &= base;
                on |= node;
                ann &= node;
                oe |= len == 0;
                ae &= len == 0;
            }
            wagg = SegOp()(wagg, warp_fold_seg(s));
        }
        __syncthreads();  // sm.seg may still be read from the previous tile
        if (lane == 0) sm.seg[w] = wagg;
        __syncthreads();
        if (threadIdx.x == 0) {
            Seg tot{0, 0, 0};
            for (uint32_t i = 0; i < kT / 32; i++) tot = SegOp()(tot, sm.seg[i]);
            a.seg[tile] = tot;
        }
    }
    // one shared atomic per warp, one global atomic per block
    bits = __reduce_or_sync(0xFFFFFFFFu, bits);
    on = __reduce_or_sync(0xFFFFFFFFu, on);
    ann = __reduce_and_sync(0xFFFFFFFFu, ann);
    oe = __reduce_or_sync(0xFFFFFFFFu, oe);
    ae = __reduce_and_sync(0xFFFFFFFFu, ae);
    const uint32_t o_lo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)o);
    const uint32_t o_hi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(o >> 32));
    const uint32_t a_lo = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)an);
    const uint32_t a_hi = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)(an >> 32));
    if ((threadIdx.x & 31) == 0) {
        if (bits) atomicOr(&s_bits, bits);
        atomicOr(&s_or, ((unsigned long long)o_hi << 32) | o_lo);
        atomicAnd(&s_and, ((unsigned long long)a_hi << 32) | a_lo);
        atomicOr(&s_orn, on);
        atomicAnd(&s_andn, ann);
        if (oe) atomicOr(&a.ctl->or_empty, 1u);
        if (!ae) atomicAnd(&a.ctl->and_empty, 0u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        raise_plan(a, s_bits);
        atomicOr(&a.ctl->or_base, s_or);
        atomicAnd(&a.ctl->and_base, s_and);
        atomicOr(&a.ctl->or_node, s_orn);
        atomicAnd(&a.ctl->and_node, s_andn);
    }
}

// The radix passes over the bits in which not all keys agree.  Fewer than two
// runs need no sort.
__device__ uint32_t active_digits(const PlanArgs &a, uint64_t R, uint32_t *act) {
    const unsigned long long db = __ldcg(&a.ctl->or_base) ^ __ldcg(&a.ctl->and_base);
    const uint32_t dn = __ldcg(&a.ctl->or_node) ^ __ldcg(&a.ctl->and_node);
    const uint32_t de = __ldcg(&a.ctl->or_empty) ^ __ldcg(&a.ctl->and_empty);
    return R > 1 ? plan_digits(db, de, dn, act) : 0;
}

// Step 2: first block of each run, coverage, sort items, first histogram.
template <int IPT>
__device__ void phase_keys(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb, uint32_t nact,
                           uint32_t dig0, ScanSmem &sm, const uint32_t *s_lf, uint32_t *s_hist) {
    const bool lf_smem = a.table_lanes + 1 <= kLaneSmem;
    __shared__ uint32_t s_bits;
    if (threadIdx.x == 0) s_bits = 0;
    __syncthreads();
    uint32_t bits = 0;
    // Runs as in the decode phase: each warp takes 32 * IPT consecutive runs,
    // run j * 32 + lane for its lane.  A run's first block is the segmented
    // count sum before it: warp scans per j in run order, the warps' totals
    // through shared memory (the scans run twice rather than hold IPT
    // prefixes in registers).
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (uint32_t tile = vb; tile < nt; tile += P) {
        for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x) s_hist[d] = 0;
        const Seg carry = reduce_prefix(a.seg, tile, SegOp(), Seg{0, 0, 0}, sm.seg);
        const uint64_t r0 = (uint64_t)tile * (kT * IPT) + (uint64_t)w * (32 * IPT) + lane;
        uint32_t cnts[IPT], lanes[IPT], nodes[IPT], lens[IPT];
        uint64_t bases[IPT];
        uint32_t heads = 0;
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t r = r0 + (uint64_t)j * 32;
            cnts[j] = 0;
            lanes[j] = 0;
            if (r < R) {
                lanes[j] = __ldcg(a.run_lane + r);
                cnts[j] = a.run_count[r];
                bases[j] = a.run_base[r];
            }
        }
        Seg wagg{0, 0, 0};
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t r = r0 + (uint64_t)j * 32;
            if (r < R) {
                nodes[j] = __ldg(a.numa + lanes[j]);
                lens[j] = __ldg(a.seg_len + lanes[j]);
                const bool head = r == (lf_smem ? s_lf[lanes[j]] : __ldcg(a.lane_first + lanes[j]));
                if (head) heads |= 1u << j;
            }
            const Seg incl = warp_scan_seg(Seg{cnts[j], heads >> j & 1u, 0});
            wagg = SegOp()(wagg, shfl_seg(incl, 31, false, 0));
        }
        __syncthreads();  // reduce_prefix's scan has read sm.seg
        if (lane == 0) sm.seg[w] = wagg;
        __syncthreads();
        Seg run = carry;  // every run before this warp's j-th group of 32
        for (uint32_t i = 0; i < w; i++) run = SegOp()(run, sm.seg[i]);
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t r = r0 + (uint64_t)j * 32;
            const Seg incl = warp_scan_seg(Seg{cnts[j], heads >> j & 1u, 0});
            Seg ex = shfl_up_words(incl, 1);
            if (lane == 0) ex = Seg{0, 0, 0};
            const Seg before = SegOp()(run, ex);
            run = SegOp()(run, shfl_seg(incl, 31, false, 0));
            if (r >= R) continue;
            const uint64_t blk = (heads >> j & 1u) ? 0 : before.sum;  // blocks of the lane before this run
            const uint32_t l = lanes[j];
            a.run_block[r] = (uint32_t)blk;
            a.run_bl[r] = blk | (uint64_t)lens[j] << 32;
            const uint32_t next_first = lf_smem ? s_lf[l + 1] : __ldcg(a.lane_first + l + 1);
            if (r + 1 == (uint64_t)next_first && blk + cnts[j] != a.B) bits |= KVX_S_COVERAGE;
            a.items0[r] = SortItem{bases[j], nodes[j], (uint32_t)r | (lens[j] == 0 ? kEmptyBit : 0u)};
        }
        if (nact) {
            // histogram of the first active digit; one shared atomic per run of
            // equal digits in consecutive lanes
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                const uint64_t r = r0 + (uint64_t)j * 32;
                const uint32_t d = r < R ? digit_of(bases[j], nodes[j], lens[j] == 0 ? 1u : 0u, dig0) : ~0u;
                add_key_runs(s_hist, d, lane);
            }
            __syncthreads();
            for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x) {
                const uint32_t c = s_hist[d];
                a.hist[0][(uint64_t)tile * kDigits + d] = c;
                if (c) atomicAdd(&a.ghist[0][(uint64_t)(tile / kHistGroup) * kDigits + d], c);
            }
        }
        __syncthreads();
    }
    if (nact > 1) {  // pass 1's histograms sum into hist[1] (small tiles) and ghist[1]
        const uint64_t ng = (uint64_t)kDigits * ceil_div((uint64_t)nt, (uint64_t)kHistGroup);
        const uint64_t n = kLocalHist<IPT> ? ng : (uint64_t)kDigits * nt;
        for (uint64_t i = (uint64_t)vb * blockDim.x + threadIdx.x; i < n;
             i += (uint64_t)P * blockDim.x) {
            if (!kLocalHist<IPT>) a.hist[1][i] = 0;
            if (i < ng) a.ghist[1][i] = 0;
        }
    }
    bits = __reduce_or_sync(0xFFFFFFFFu, bits);
    if ((threadIdx.x & 31) == 0 && bits) atomicOr(&s_bits, bits);
    __syncthreads();
    if (threadIdx.x == 0) raise_plan(a, s_bits);
}

// One radix pass (one barrier).  Histograms are tile-major, H[t][d] = items
// of tile t with digit d.  Every block sweeps H once, one thread per digit
// (coalesced rows): the digit totals, and the count before each of its own
// tiles; the digit bases follow by a scan of the totals.  Then per tile: a
// stable rank inside the tile (warp match + per-warp digit counters), the
// scatter, and the next digit's histogram per output tile (atomics into Hn,
// cleared one pass earlier).  Hz is cleared here for the pass after next.
constexpr uint32_t kOwnChunk = 8;  // own tiles whose offsets are held at once

// Per-block counters of a radix pass.
struct SortCounters {
    uint32_t wcnt[kT / 32][kDigits];  // per warp and digit
    uint32_t s_off[kOwnChunk][kDigits];
    uint32_t s_base[kDigits];
};
constexpr int kSweep = 32;         // histogram rows loaded at once in the offset sweep


template <int IPT>
__device__ void phase_sort_pass(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb,
                                const SortItem *in, SortItem *out, const uint32_t *H, uint32_t *Hn,
                                uint32_t *Hz, const uint32_t *G, uint32_t *Gn, uint32_t *Gz, uint32_t dig,
                                bool has_next, uint32_t ndig, bool clear_z, SortCounters &sc) {
    uint32_t (*wcnt)[kDigits] = sc.wcnt;
    uint32_t (*s_off)[kDigits] = sc.s_off;
    uint32_t *s_base = sc.s_base;
    __shared__ uint64_t sh[33];
    static_assert(kT == kDigits, "one thread per digit");
    const uint32_t ng = (nt + kHistGroup - 1) / kHistGroup;
    if (clear_z) {  // the histograms of the pass after next sum into Hz and Gz
        const uint64_t n = (uint64_t)kDigits * (kLocalHist<IPT> ? ng : nt);
        for (uint64_t i = (uint64_t)vb * blockDim.x + threadIdx.x; i < n;
             i += (uint64_t)P * blockDim.x) {
            if (!kLocalHist<IPT>) Hz[i] = 0;
            if (i < (uint64_t)kDigits * ng) Gz[i] = 0;
        }
    }
    const uint32_t d_me = threadIdx.x;
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const uint32_t own = nt > vb ? (nt - vb + P - 1) / P : 0;
    for (uint32_t c0 = 0; c0 < own; c0 += kOwnChunk) {
        const uint32_t nslot = own - c0 < kOwnChunk ? own - c0 : kOwnChunk;
        // the count of digit d_me in the tile groups before each own tile's
        // group (and, after the sweep, its total): kSweep group rows in
        // flight per thread
        uint64_t run = 0;
        uint32_t next_slot = 0;
        for (uint32_t g0 = 0; g0 < ng; g0 += kSweep) {
            uint32_t v[kSweep];
#pragma unroll
            for (int u = 0; u < kSweep; u++)
                v[u] = g0 + u < ng ? __ldcg(G + (uint64_t)(g0 + u) * kDigits + d_me) : 0;
#pragma unroll
            for (int u = 0; u < kSweep; u++) {
                while (next_slot < nslot && (vb + (c0 + next_slot) * P) / kHistGroup == g0 + u) {
                    s_off[next_slot][d_me] = (uint32_t)run;
                    next_slot++;
                }
                run += v[u];
            }
        }
        // plus the tiles of each own tile's group that come before it
        for (uint32_t slot = 0; slot < nslot; slot++) {
            const uint32_t tile = vb + (c0 + slot) * P;
            const uint32_t t0 = tile - tile % kHistGroup;
            uint32_t v[kHistGroup - 1];
#pragma unroll
            for (int u = 0; u < (int)kHistGroup - 1; u++)
                v[u] = t0 + u < tile ? __ldcg(H + (uint64_t)(t0 + u) * kDigits + d_me) : 0;
            uint32_t sum = 0;
#pragma unroll
            for (int u = 0; u < (int)kHistGroup - 1; u++) sum += v[u];
            s_off[slot][d_me] += sum;
        }
        {   // digit bases = exclusive scan of the digit totals
            uint64_t tot;
            const uint64_t ex = block_excl_sum<uint64_t>(run, sh, &tot);
            s_base[d_me] = (uint32_t)ex;
        }
        __syncthreads();
        for (uint32_t slot = 0; slot < kOwnChunk && c0 + slot < own; slot++) {
            const uint32_t tile = vb + (c0 + slot) * P;
            for (uint32_t i = threadIdx.x; i < (kT / 32) * kDigits; i += blockDim.x) (&wcnt[0][0])[i] = 0;
            __syncthreads();
            SortItem it[IPT];
            uint32_t d[IPT], pos[IPT];
            const uint64_t t0 = (uint64_t)tile * (kT * IPT) + (uint64_t)w * (32 * IPT);
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                const uint64_t idx = t0 + (uint64_t)j * 32 + lane;
                if (idx < R) {
                    it[j] = ld_cg(in + idx);
                    d[j] = digit_of(it[j].base, it[j].node, it[j].r >> 31, dig);
                } else {
                    d[j] = kDigits;  // past the end: matches only other past-the-end lanes
                }
            }
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                const uint32_t peers = digit_peers(d[j]);
                const uint32_t rank = __popc(peers & lt_mask);
                const uint32_t before = d[j] < kDigits ? wcnt[w][d[j]] : 0;
                __syncwarp();
                if (d[j] < kDigits && rank == 0) wcnt[w][d[j]] = before + __popc(peers);
                __syncwarp();
                pos[j] = before + rank;
            }
            __syncthreads();
            {
                uint32_t acc = 0;
                for (int ww = 0; ww < kT / 32; ww++) {
                    const uint32_t c = wcnt[ww][d_me];
                    wcnt[ww][d_me] = acc;
                    acc += c;
                }
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                uint32_t key = ~0u;  // next-histogram bin of this item (output tile, next digit)
                if (d[j] < kDigits) {
                    const uint64_t dst = (uint64_t)s_base[d[j]] + s_off[slot][d[j]] + wcnt[w][d[j]] + pos[j];
                    if (dst < R) {  // always: the offsets are a permutation of [0, R)
                        out[dst] = it[j];
                        if (!kLocalHist<IPT> && has_next)
                            key = (uint32_t)(dst / (kT * IPT)) * kDigits +
                                  digit_of(it[j].base, it[j].node, it[j].r >> 31, ndig);
                    }
                }
                if (!kLocalHist<IPT> && has_next) {  // per tile, and per group of kHistGroup tiles
                    add_key_runs(Hn, key, lane);
                    add_key_runs(Gn, key == ~0u ? ~0u : (key / kDigits / kHistGroup) * kDigits + key % kDigits,
                                 lane);
                }
            }
            __syncthreads();
        }
    }
}

// The histograms of a radix pass after the first, from the previous pass's
// output: each block counts its own tiles' digits in shared memory (one
// atomic per run of equal digits in consecutive lanes), writes the tile rows
// of H and adds them into the group rows of G (cleared two phases earlier).
// A grid barrier follows, then the pass.  Out of line: inlined, it made the
// whole kernel spill.
template <int IPT>
__device__ __noinline__ void phase_hist(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb,
                                        const SortItem *in, uint32_t *H, uint32_t *G, uint32_t dig,
                                        uint32_t *s_hist) {
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (uint32_t tile = vb; tile < nt; tile += P) {
        for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x) s_hist[d] = 0;
        __syncthreads();
        const uint64_t t0 = (uint64_t)tile * (kT * IPT) + (uint64_t)w * (32 * IPT) + lane;
        SortItem it[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++)
            if (t0 + (uint64_t)j * 32 < R) it[j] = ld_cg(in + t0 + (uint64_t)j * 32);
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const bool in_range = t0 + (uint64_t)j * 32 < R;
            add_key_runs(s_hist, in_range ? digit_of(it[j].base, it[j].node, it[j].r >> 31, dig) : ~0u, lane);
        }
        __syncthreads();
        for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x) {
            const uint32_t c = s_hist[d];
            H[(uint64_t)tile * kDigits + d] = c;
            if (c) atomicAdd(&G[(uint64_t)(tile / kHistGroup) * kDigits + d], c);
        }
        __syncthreads();
    }
}

__device__ __forceinline__ Rec make_rec(const PlanArgs &a, SortItem it, uint64_t R) {
    it.r = item_run(it);
    if (it.r >= R) it.r = 0;  // never taken: sorted items are a permutation of the runs
    Rec x;
    x.base = it.base;
    x.node = it.node;
    x.r = it.r;
    x.stride = __ldg(a.run_stride + it.r);
    x.count = __ldg(a.run_count + it.r);
    const uint64_t bl = __ldcg(a.run_bl + it.r);
    x.block = (uint32_t)bl;
    x.len = (uint32_t)(bl >> 32);
    x.pad = 0;
    return x;
}

// The record of the run at sorted position p.
__device__ __forceinline__ Rec rec_at(const PlanArgs &a, const SortItem *sorted, uint64_t p, uint64_t R) {
    return make_rec(a, ld_cg(sorted + p), R);
}

// The base of the run that starts the compatible stretch holding sorted
// position p (known to be compatible with p - 1), by the whole block: it
// walks back over the sorted order kT positions at a time, each thread
// testing one position against its predecessor, to the last position that
// is not compatible with its predecessor.  A stretch joins runs of one block
// range and stride at adjacent bases, so it is a few rounds long at most.
__device__ uint64_t stretch_base(const PlanArgs &a, uint64_t R, const SortItem *sorted, uint64_t p,
                                 int64_t *s_max, uint64_t *s_found) {
    for (uint64_t hi = p; hi > 0; hi = hi > kT ? hi - kT : 0) {
        const int64_t q = (int64_t)hi - (int64_t)kT + (int64_t)threadIdx.x;
        bool start = false;
        uint64_t base = 0;
        if (q >= 0) {
            const Rec x = make_rec(a, ld_cg(sorted + q), R);
            base = x.base;
            start = q == 0 || !compatible(make_rec(a, ld_cg(sorted + q - 1), R), x);
        }
        if (threadIdx.x == 0) *s_max = -1;
        __syncthreads();
        if (start) atomicMax(reinterpret_cast<long long *>(s_max), (long long)q);
        __syncthreads();
        const int64_t last = *s_max;
        if (last >= 0) {
            if (q == last) *s_found = base;
            __syncthreads();
            return *s_found;
        }
    }
    return 0;  // never reached: position 0 starts a stretch
}

// Per-tile totals passed between blocks inside one phase: a tile publishes
// its total behind a flag (after a fence), and a later tile waits for the
// flags of the tiles before it.  Every tile publishes before it waits for
// anything, waits go only to tiles that publish first (earlier tiles, and
// the first flag of the next tile), and all blocks are resident, so the
// waits end; each is bounded in time all the same.
__device__ __forceinline__ void publish(uint32_t *flag, uint32_t v) {
    __syncthreads();  // the block's writes of this tile are done
    if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(v) : "memory");
    }
}
// The flag's value once set (1 = published, 2 = the tile was abandoned), or 0
// if the wait gave up after about a second.
__device__ __forceinline__ uint32_t wait_ready(const uint32_t *flag) {
    uint64_t t0 = 0;
    for (uint32_t polls = 0;; polls++) {
        const uint32_t v = ld_acquire_gpu(flag);
        if (v) return v;
        if (polls >= 64) {
            if (polls == 64) t0 = global_ns();
            if (polls >= kBarrierPolls || global_ns() - t0 > kWaitNs) return 0;
            __nanosleep(64);
        }
    }
}

// Diagnostic (kvx_selftest_timeouts): the flag wait gives up on a flag that
// nothing ever sets.
__device__ uint32_t g_selftest_flag;  // never written: stays 0

__global__ void k_selftest_flag(uint32_t *status) {
    if (threadIdx.x == 0 && wait_ready(&g_selftest_flag) == 0) atomicOr(status, KVX_S_TIMEOUT);
}

// Steps 3 and 4 after the sort, one phase per tile with no grid barrier:
//   - adjacency: the sorted records and compat flags;
//   - the group starts: the "grown chunk still fits the stride" cut from the
//     bases of each stretch's first run (shared memory inside the tile, a
//     look-back for the stretch open at the tile's start);
//   - group numbering: the tile publishes its group count, then sums the
//     counts of the tiles before it;
//   - groups: run_group / run_off, and the tile's slab bytes and reads, which
//     it publishes, then sums those of the tiles before it;
//   - the carve and the reads: group records with their slab offsets and the
//     read descriptors, replayed from registers;
//   - the last tile writes the counts.
// Runs whose stretch outgrows its stride need a walk in order across
// positions other tiles own: such a tile is marked walked and abandoned, so
// are the tiles after it, and the barrier-separated phases (cut with the
// walks, count, groups, emit) redo everything after the grid barrier.  The
// records, compat flags and per-tile stretch starts every tile writes here
// are what those phases read.
template <int IPT, bool kFuse>
__device__ void phase_post_sort(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb,
                                const SortItem *sorted, ScanSmem &sm, uint64_t *s_tbase) {
    __shared__ uint64_t s_open;  // base of the first run of the stretch open at the tile's start
    __shared__ uint32_t s_need;
    __shared__ int64_t s_lmax;
    __shared__ uint64_t s_lbase;
    __shared__ uint8_t s_first[kT];  // each thread's first position starts a group
    __shared__ uint32_t s_next;      // the position after the tile starts a group (or is the end)
    __shared__ uint32_t s_bad;
    const uint64_t T = (uint64_t)kT * IPT;
    for (uint32_t tile = vb; tile < nt; tile += P) {
        const uint64_t p0 = (uint64_t)tile * T + (uint64_t)threadIdx.x * IPT;
        Rec prev;
        bool have_prev = false;
        if (p0 > 0 && p0 < R) {
            prev = make_rec(a, ld_cg(sorted + p0 - 1), R);
            have_prev = true;
        }
        SortItem its[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            its[j].r = 0;
            if (p0 + j < R) {
                its[j] = ld_cg(sorted + p0 + j);
                its[j].r = item_run(its[j]);
                if (its[j].r >= R) its[j].r = 0;  // never taken: a permutation of the runs
            }
        }
        int64_t xs[IPT];
        uint32_t xc[IPT], blocks[IPT], xl[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            if (p0 + j >= R) continue;
            const uint32_t r = its[j].r;
            xs[j] = __ldg(a.run_stride + r);
            xc[j] = __ldg(a.run_count + r);
            const uint64_t bl = __ldcg(a.run_bl + r);
            blocks[j] = (uint32_t)bl;
            xl[j] = (uint32_t)(bl >> 32);
        }
        int64_t mx = -1;
        uint32_t cm = 0;  // bit j: position p0 + j is compatible with its predecessor
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) continue;
            Rec x;
            x.base = its[j].base;
            x.node = its[j].node;
            x.r = its[j].r;
            x.stride = xs[j];
            x.count = xc[j];
            x.block = blocks[j];
            x.len = xl[j];
            x.pad = 0;
            s_tbase[p - (uint64_t)tile * T] = x.base;
            const bool c = have_prev && compatible(prev, x);
            a.compat[p] = c ? 1 : 0;
            if (c) cm |= 1u << j;
            else mx = (int64_t)p;
            prev = x;
            have_prev = true;
        }
        int64_t ex, tot;
        block_scan(mx, MaxOp(), (int64_t)-1, sm.i64, &ex, &tot);
        if (threadIdx.x == 0) a.segmax[tile] = tot;
        // The stretch open at the tile's first position, if it began in an
        // earlier tile: its first run's base is needed only when its runs
        // could share a group (more than one block and a positive stride;
        // every run of a stretch has the same count and stride).
        if (threadIdx.x == 0)
            s_need = p0 < R && (cm & 1u) && xc[0] > 1 && xs[0] > 0 ? 1u : 0u;
        __syncthreads();  // s_tbase complete, s_need set
        if (s_need) {
            const uint64_t b = stretch_base(a, R, sorted, (uint64_t)tile * T, &s_lmax, &s_lbase);
            if (threadIdx.x == 0) s_open = b;
            __syncthreads();
        }
        uint64_t s_base = 0;  // base of the current stretch's first run
        if (p0 < R && (cm & 1u)) s_base = ex >= 0 ? s_tbase[(uint64_t)ex - (uint64_t)tile * T] : s_open;
        GAgg g{0, -1};
        bool walker = false;
        uint32_t sb = 0;  // bit j: position p0 + j starts a group
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) break;
            const bool c = cm >> j & 1u;
            const uint64_t xb = its[j].base;
            if (!c) s_base = xb;
            bool start;
            if (xc[j] == 1) {
                start = !c;
            } else if (xs[j] <= 0) {
                start = true;  // a non-positive stride never fits: one run per group
            } else {
                const uint64_t E = xb - s_base + xl[j];  // end of the run in its stretch
                if (E > (uint64_t)xs[j]) {  // the stretch outgrows its stride: the cut phase walks it
                    walker = true;
                    continue;
                }
                start = !c;
            }
            a.gflag[p] = start ? 1 : 0;
            if (start) {
                sb |= 1u << j;
                g.n++;
                g.last = (int64_t)p;
            }
        }
        GAgg gex, gtot;
        block_scan(g, GOp(), GAgg{0, -1}, sm.g, &gex, &gtot);
        s_first[threadIdx.x] = (uint8_t)(sb & 1u);
        const bool tile_walked = __syncthreads_or(walker) != 0;
        if (threadIdx.x == 0) {
            a.gagg[tile] = gtot;
            if (tile_walked) atomicOr(&a.ctl->walked, 1u);
        }
        if constexpr (!kFuse) {
            // groups and the carve follow as their own phases, after a barrier
            __syncthreads();  // s_tbase and s_first are rewritten by the next tile
            continue;
        }
        publish(a.ready_g + tile, tile_walked ? 2u : 1u);

        // ---- group numbering: the group counts of the tiles before this one,
        // and whether the position after the tile starts a group
        uint32_t bad = tile_walked ? 1u : 0u;  // 1: abandoned (a walk), 2: a wait gave up
        GAgg vg{0, -1};
        for (uint32_t t = threadIdx.x; t < tile && !bad; t += kT) {
            const uint32_t f = wait_ready(a.ready_g + t);
            if (f != 1) bad = f ? 1u : 2u;
            else vg = GOp()(vg, ld_cg(a.gagg + t));
        }
        if (threadIdx.x == kT - 1 && !bad) {
            const uint64_t q = (uint64_t)(tile + 1) * T;
            uint32_t nx = 1;  // the end of the table ends the last group
            if (q < R) {
                const uint32_t f = wait_ready(a.ready_g + tile + 1);
                if (f != 1) bad = f ? 1u : 2u;
                else nx = __ldcg(a.gflag + q) ? 1u : 0u;
            }
            s_next = nx;
        }
        {
            GAgg ex2, all;
            block_scan(vg, GOp(), GAgg{0, -1}, sm.g, &ex2, &all);
            vg = all;
        }
        if (threadIdx.x == 0) s_bad = 0;
        __syncthreads();
        if (bad) atomicOr(&s_bad, bad);
        __syncthreads();
        bad = s_bad;
        if (bad) {
            if (threadIdx.x == 0 && (bad & 2u)) raise_plan(a, KVX_S_TIMEOUT);
            publish(a.ready_c + tile, 2u);
            continue;
        }
        const GAgg carry_g = vg;
        // bit j: p0 + j starts a group or is the end; bit IPT: the position after the thread's
        uint32_t fl = sb;
#pragma unroll
        for (int j = 0; j <= IPT; j++)
            if (p0 + j == R) fl |= 1u << j;
        if (p0 + IPT < R)
            fl |= (threadIdx.x + 1 < kT ? (uint32_t)s_first[threadIdx.x + 1] : s_next) << IPT;

        // ---- groups: run_group / run_off; the tile's slab bytes and reads
        const GAgg run0 = GOp()(carry_g, gex);  // groups before this thread's first run
        uint64_t o_base = 0, o_block = 0, o_count = 0, o_node = 0;  // the group open at the first run
        int64_t o_stride = 0;
        if (p0 < R && !(fl & 1u)) {
            const Rec q = rec_at(a, sorted, run0.last >= 0 ? (uint64_t)run0.last : 0, R);
            o_base = q.base;
            o_stride = q.stride;
            o_block = q.block;
            o_count = q.count;
            o_node = q.node;
        }
        CAgg c{0, 0};
        {
            uint64_t n = run0.n, g_base = o_base, g_count = o_count;
            int64_t g_stride = o_stride;
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                const uint64_t p = p0 + j;
                if (p >= R) break;
                if (fl >> j & 1u) {
                    n++;
                    g_base = its[j].base;
                    g_stride = xs[j];
                    g_count = xc[j];
                }
                const uint64_t off = its[j].base - g_base;
                a.run_group[its[j].r] = (uint32_t)(n - 1);
                a.run_off[its[j].r] = off;
                if (fl >> (j + 1) & 1u) {  // the group ends here
                    kvx_group G;
                    G.stride = g_stride;
                    G.chunk = off + xl[j];
                    G.count = (uint32_t)g_count;
                    G.dense = group_dense(G.count, G.stride, G.chunk) ? 1u : 0u;
                    c.bytes += (uint64_t)G.count * G.chunk;
                    c.descs += group_pieces(G);
                }
            }
        }
        CAgg cex, ctot;
        block_scan(c, COp(), CAgg{0, 0}, sm.c, &cex, &ctot);
        if (threadIdx.x == 0) a.cagg[tile] = ctot;
        publish(a.ready_c + tile, 1u);

        // ---- the carve of the tiles before this one
        CAgg vc{0, 0};
        for (uint32_t t = threadIdx.x; t < tile && !bad; t += kT) {
            const uint32_t f = wait_ready(a.ready_c + t);
            if (f != 1) bad = f ? 1u : 2u;
            else vc = COp()(vc, ld_cg(a.cagg + t));
        }
        {
            CAgg ex2, all;
            block_scan(vc, COp(), CAgg{0, 0}, sm.c, &ex2, &all);
            vc = all;
        }
        if (threadIdx.x == 0) s_bad = 0;
        __syncthreads();
        if (bad) atomicOr(&s_bad, bad);
        __syncthreads();
        if (s_bad) {  // the barrier-separated phases redo it (after a walk), or the wait gave up
            if (threadIdx.x == 0 && (s_bad & 2u)) raise_plan(a, KVX_S_TIMEOUT);
            continue;
        }

        // ---- step 4: group records with their slab offsets, and the reads
        {
            CAgg cur = COp()(vc, cex);
            const uint64_t M = KVX_MAX_READ_BYTES;
            uint64_t n = run0.n, g_base = o_base, g_block = o_block, g_count = o_count, g_node = o_node;
            int64_t g_stride = o_stride;
#pragma unroll
            for (int j = 0; j < IPT; j++) {
                const uint64_t p = p0 + j;
                if (p >= R) break;
                if (fl >> j & 1u) {
                    n++;
                    g_base = its[j].base;
                    g_stride = xs[j];
                    g_block = blocks[j];
                    g_count = xc[j];
                    g_node = its[j].node;
                }
                if (!(fl >> (j + 1) & 1u)) continue;
                kvx_group G;
                G.base = g_base;
                G.stride = g_stride;
                G.chunk = its[j].base - g_base + xl[j];
                G.local = cur.bytes;
                G.block = (uint32_t)g_block;
                G.count = (uint32_t)g_count;
                G.node = (uint32_t)g_node;
                G.dense = group_dense(G.count, G.stride, G.chunk) ? 1u : 0u;
                const uint64_t gid = n - 1;
                if (gid < a.group_cap) st_group(a, gid, G);
                uint64_t d = cur.descs;
                if (G.dense) {
                    const uint64_t total = (uint64_t)G.count * G.chunk;
                    for (uint64_t o = 0; o < total; o += M, d++)
                        if (d < a.desc_cap)
                            st_desc(a, d, G.base + o, G.local + o, total - o < M ? total - o : M, (uint32_t)gid);
                } else if (G.chunk > 0) {  // a group of empty runs has no read
                    for (uint64_t i = 0; i < G.count; i++) {
                        const uint64_t rb = G.base + i * (uint64_t)G.stride;
                        const uint64_t lb = G.local + i * G.chunk;
                        for (uint64_t o = 0; o < G.chunk; o += M, d++)
                            if (d < a.desc_cap)
                                st_desc(a, d, rb + o, lb + o, G.chunk - o < M ? G.chunk - o : M, (uint32_t)gid);
                    }
                }
                cur.bytes += (uint64_t)G.count * G.chunk;
                cur.descs += group_pieces(G);
            }
        }
        if (tile == nt - 1 && threadIdx.x == 0) {  // the counts, with the capacity checks
            const GAgg gall = GOp()(carry_g, gtot);
            const CAgg call = COp()(vc, ctot);
            if (gall.n > a.group_cap || call.descs > a.desc_cap) {
                raise_plan(a, KVX_S_CAPACITY);
                a.counts[0] = a.counts[1] = a.counts[2] = 0;
            } else {
                a.counts[0] = gall.n;
                a.counts[1] = call.descs;
                a.counts[2] = call.bytes;
            }
        }
        __syncthreads();  // s_tbase and s_first are rewritten by the next tile
    }
}

// The run at position p outgrows the first group of its compatible stretch
// (its chunk exceeds the stride): it starts a group, and the rest of the
// stretch is cut in order, a new group wherever the chunk would outgrow the
// stride again (only tables whose block chunks exceed their stride get here).
__device__ __noinline__ void walk_stretch(const PlanArgs &a, const SortItem *sorted, uint64_t R, uint64_t p,
                                          uint64_t base, uint64_t stride) {
    a.gflag[p] = 1;
    uint64_t cur = base;
    for (uint64_t q = p + 1; q < R && __ldcg(a.compat + q); q++) {
        const Rec y = rec_at(a, sorted, q, R);
        if (y.base + y.len - cur > stride) {
            a.gflag[q] = 1;
            cur = y.base;
        } else {
            a.gflag[q] = 0;
        }
    }
}

// Step 3: group starts.
template <int IPT>
__device__ void phase_cut(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb,
                          const SortItem *sorted, ScanSmem &sm) {
    for (uint32_t tile = vb; tile < nt; tile += P) {
        const int64_t carry = reduce_prefix(a.segmax, tile, MaxOp(), (int64_t)-1, sm.i64);
        const uint64_t p0 = (uint64_t)tile * (kT * IPT) + (uint64_t)threadIdx.x * IPT;
        // every load of this thread's runs first
        uint32_t cm = 0;  // bit j: position p0 + j is compatible with its predecessor
        uint64_t xb[IPT];
        int64_t xs[IPT];
        uint32_t xc[IPT], xl[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p < R) {
                const Rec q = rec_at(a, sorted, p, R);
                if (__ldcg(a.compat + p)) cm |= 1u << j;
                xb[j] = q.base;
                xs[j] = q.stride;
                xc[j] = q.count;
                xl[j] = q.len;
            }
        }
        int64_t mx = -1;
#pragma unroll
        for (int j = 0; j < IPT; j++)
            if (p0 + j < R && !(cm >> j & 1u)) mx = (int64_t)(p0 + j);
        int64_t ex, tot;
        block_scan(mx, MaxOp(), (int64_t)-1, sm.i64, &ex, &tot);
        const int64_t s0 = carry > ex ? carry : ex;  // stretch start before this thread's first run
        uint64_t s_base = 0;                          // base of the current stretch's first run
        if (p0 < R && (cm & 1u)) s_base = ld_cg(sorted + (s0 > 0 ? s0 : 0)).base;
        // the tile's group starts, for the groups phase (valid when no
        // walker ran anywhere: then every flag was set by its own position)
        GAgg g{0, -1};
        bool walker = false;
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) break;
            const bool c = cm >> j & 1u;
            if (!c) s_base = xb[j];
            bool start;
            if (xc[j] == 1) {
                start = !c;
            } else if (xs[j] <= 0) {
                start = true;  // a non-positive stride never fits: one run per group
            } else {
                const uint64_t stride = (uint64_t)xs[j];
                const uint64_t O = xb[j] - s_base;  // offset in the stretch
                const uint64_t E = O + xl[j];
                if (E <= stride) {
                    start = !c;
                } else {
                    // O <= stride: the first run that outgrows the stretch's
                    // first group walks the rest of the stretch; O > stride:
                    // a later run of such a stretch, flagged by that walker
                    walker = true;
                    if (O <= stride) walk_stretch(a, sorted, R, p, xb[j], stride);
                    continue;
                }
            }
            a.gflag[p] = start ? 1 : 0;
            if (start) {
                g.n++;
                g.last = (int64_t)p;
            }
        }
        GAgg gex, gtot;
        block_scan(g, GOp(), GAgg{0, -1}, sm.g, &gex, &gtot);
        if (threadIdx.x == 0) a.gagg[tile] = gtot;
        if (__any_sync(0xFFFFFFFFu, walker) && (threadIdx.x & 31) == 0) atomicOr(&a.ctl->walked, 1u);
    }
}

template <int IPT>
__device__ void phase_count(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb, ScanSmem &sm) {
    for (uint32_t tile = vb; tile < nt; tile += P) {
        GAgg g{0, -1};
        const uint64_t p0 = (uint64_t)tile * (kT * IPT) + (uint64_t)threadIdx.x * IPT;
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p < R && __ldcg(a.gflag + p)) {
                g.n++;
                g.last = (int64_t)p;
            }
        }
        GAgg ex, tot;
        block_scan(g, GOp(), GAgg{0, -1}, sm.g, &ex, &tot);
        if (threadIdx.x == 0) a.gagg[tile] = tot;
    }
}

// Group records, run_group / run_off; per tile the carve bytes and pieces.
// Every load a thread needs is issued up front (flags, the fields of its
// runs, and the fields of the runs that start groups), so a thread pays one
// round trip per dependency level rather than one per run.  The thread's
// group count and carve prefix inside the tile are kept for the emit phase.
template <int IPT>
__device__ void phase_groups(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb,
                             const SortItem *sorted, ScanSmem &sm) {
    for (uint32_t tile = vb; tile < nt; tile += P) {
        const GAgg carry = reduce_prefix(a.gagg, tile, GOp(), GAgg{0, -1}, sm.g);
        const uint64_t p0 = (uint64_t)tile * (kT * IPT) + (uint64_t)threadIdx.x * IPT;
        uint32_t fl = 0;  // bit j: position p0 + j starts a group (bit IPT: the next one, or R)
#pragma unroll
        for (int j = 0; j <= IPT; j++) {
            const uint64_t p = p0 + j;
            const uint32_t v = p < R ? (__ldcg(a.gflag + p) ? 1u : 0u) : (p == R ? 1u : 0u);
            fl |= v << j;
        }
        uint64_t xb[IPT];
        uint32_t xr[IPT], xl[IPT];
        int64_t gs[IPT];
        uint32_t gb[IPT], gc[IPT], gn[IPT];
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p < R) {
                SortItem it = ld_cg(sorted + p);
                it.r = item_run(it);
                if (it.r >= R) it.r = 0;  // never taken: sorted items are a permutation of the runs
                const uint64_t bl = __ldcg(a.run_bl + it.r);
                xb[j] = it.base;
                xl[j] = (uint32_t)(bl >> 32);
                xr[j] = it.r;
                if (fl >> j & 1u) {
                    gs[j] = __ldg(a.run_stride + it.r);
                    gb[j] = (uint32_t)bl;
                    gc[j] = __ldg(a.run_count + it.r);
                    gn[j] = it.node;
                }
            }
        }
        GAgg g{0, -1};
#pragma unroll
        for (int j = 0; j < IPT; j++)
            if (p0 + j < R && (fl >> j & 1u)) {
                g.n++;
                g.last = (int64_t)(p0 + j);
            }
        GAgg ex, tot;
        block_scan(g, GOp(), GAgg{0, -1}, sm.g, &ex, &tot);
        GAgg run = GOp()(carry, ex);
        if (p0 < R) a.gthr[(uint64_t)tile * kT + threadIdx.x] = run;
        // the group open at this thread's first run (position 0 always starts one)
        uint64_t g_base = 0, g_block = 0, g_count = 0, g_node = 0;
        int64_t g_stride = 0;
        if (p0 < R && !(fl & 1u)) {
            const Rec q = rec_at(a, sorted, run.last >= 0 ? (uint64_t)run.last : 0, R);
            g_base = q.base;
            g_stride = q.stride;
            g_block = q.block;
            g_count = q.count;
            g_node = q.node;
        }
        CAgg c{0, 0};
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) break;
            if (fl >> j & 1u) {
                run.n++;
                g_base = xb[j];
                g_stride = gs[j];
                g_block = gb[j];
                g_count = gc[j];
                g_node = gn[j];
            }
            const uint64_t gid = run.n - 1;
            const uint64_t off = xb[j] - g_base;
            a.run_group[xr[j]] = (uint32_t)gid;
            a.run_off[xr[j]] = off;
            if (fl >> (j + 1) & 1u) {  // the group ends here
                kvx_group G;
                G.base = g_base;
                G.stride = g_stride;
                G.chunk = off + xl[j];
                G.local = 0;
                G.block = (uint32_t)g_block;
                G.count = (uint32_t)g_count;
                G.node = (uint32_t)g_node;
                G.dense = group_dense(G.count, G.stride, G.chunk) ? 1u : 0u;
                st_group(a, gid, G);
                c.bytes += (uint64_t)G.count * G.chunk;
                c.descs += group_pieces(G);
            }
        }
        CAgg cex, ctot;
        block_scan(c, COp(), CAgg{0, 0}, sm.c, &cex, &ctot);
        if (p0 < R) a.cthr[(uint64_t)tile * kT + threadIdx.x] = cex;
        if (threadIdx.x == 0) a.cagg[tile] = ctot;
    }
}

// Step 4: carve and descriptors.  A thread takes its group count and carve
// prefix from the groups phase, so each group end costs one load of its
// record (all of them issued at once).
template <int IPT>
__device__ void phase_emit(const PlanArgs &a, uint64_t R, uint32_t nt, uint32_t P, uint32_t vb, ScanSmem &sm) {
    for (uint32_t tile = vb; tile < nt; tile += P) {
        const CAgg carry = reduce_prefix(a.cagg, tile, COp(), CAgg{0, 0}, sm.c);
        const uint64_t p0 = (uint64_t)tile * (kT * IPT) + (uint64_t)threadIdx.x * IPT;
        if (p0 >= R) continue;
        uint32_t fl = 0;
#pragma unroll
        for (int j = 0; j <= IPT; j++) {
            const uint64_t p = p0 + j;
            const uint32_t v = p < R ? (__ldcg(a.gflag + p) ? 1u : 0u) : (p == R ? 1u : 0u);
            fl |= v << j;
        }
        const GAgg run0 = ld_cg(a.gthr + (uint64_t)tile * kT + threadIdx.x);
        const CAgg cex = ld_cg(a.cthr + (uint64_t)tile * kT + threadIdx.x);
        uint32_t gids[IPT];
        kvx_group G[IPT];
        uint64_t n = run0.n;
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            if (p0 + j < R && (fl >> j & 1u)) n++;
            gids[j] = (uint32_t)(n - 1);
            if (p0 + j < R && (fl >> (j + 1) & 1u)) G[j] = ld_group(a, gids[j]);
        }
        CAgg cur = COp()(carry, cex);
        const uint64_t M = KVX_MAX_READ_BYTES;
#pragma unroll
        for (int j = 0; j < IPT; j++) {
            if (p0 + j >= R || !(fl >> (j + 1) & 1u)) continue;
            kvx_group g = G[j];
            const uint32_t gid = gids[j];
            g.local = cur.bytes;
            a.groups[gid].local = cur.bytes;
            uint64_t d = cur.descs;
            if (g.dense) {
                const uint64_t total = (uint64_t)g.count * g.chunk;
                for (uint64_t o = 0; o < total; o += M, d++)
                    st_desc(a, d, g.base + o, g.local + o, total - o < M ? total - o : M, gid);
            } else if (g.chunk > 0) {  // a group of empty runs has no read
                for (uint64_t i = 0; i < g.count; i++) {
                    const uint64_t rb = g.base + i * (uint64_t)g.stride;
                    const uint64_t lb = g.local + i * g.chunk;
                    for (uint64_t o = 0; o < g.chunk; o += M, d++)
                        st_desc(a, d, rb + o, lb + o, g.chunk - o < M ? g.chunk - o : M, gid);
                }
            }
            cur.bytes += (uint64_t)g.count * g.chunk;
            cur.descs += group_pieces(g);
        }
    }
}

__device__ void on_abort(const PlanArgs &a) {
    if (threadIdx.x == 0) {
        atomicOr(a.status, KVX_S_TIMEOUT);
        a.counts[0] = a.counts[1] = a.counts[2] = 0;
    }
}

#define PLAN_BARRIER()                           \
    do {                                         \
        if (!grid_barrier(&a.ctl->gs, P)) {      \
            on_abort(a);                         \
            return;                              \
        }                                        \
    } while (0)


// ------------------------------------------------- single-block planner
//
// Tables of up to 2048 runs (every bump-allocated holder with up to 1024
// slots) are planned by one block of 1024 threads, 2 runs each, with the
// whole run table in shared memory: the same steps as the phases above, each
// a few shared-memory passes and warp-shuffle scans instead of global round
// trips.  The cooperative kernel returns at once for these tables.
constexpr uint32_t kSmallRuns = 2048;
constexpr int kST = 1024;
constexpr int kSW = kST / 32;

__device__ __forceinline__ bool plan_is_small(const PlanArgs &a, uint64_t R) {
    return R <= kSmallRuns && R <= a.run_cap && a.table_lanes == a.template_lanes &&
           a.table_lanes + 1 <= kLaneSmem;
}

struct SmallSmem {
    uint64_t base[kSmallRuns];
    int64_t stride[kSmallRuns];
    uint32_t lf[kLaneSmem];
    uint32_t count[kSmallRuns];
    uint32_t lane[kSmallRuns];
    uint32_t block[kSmallRuns];
    uint32_t node[kSmallRuns];
    uint32_t len[kSmallRuns];
    uint16_t idx[2][kSmallRuns];
    uint16_t wcnt[kSW][kDigits];
    uint32_t dbase[kDigits];
    uint8_t flag[kSmallRuns + 1];
    uint8_t compat[kSmallRuns];
};

template <class T>
__device__ __forceinline__ T shfl_up_any(T v, int d) {
    static_assert(sizeof(T) % 4 == 0, "4-byte multiple");
    T o;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(&v);
    uint32_t *dst = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); i++) dst[i] = __shfl_up_sync(0xFFFFFFFFu, src[i], d);
    return o;
}

// Block-wide inclusive scan (1024 threads), warp shuffles + one warp over the
// warp totals.  *excl / *total as in block_scan.
template <class T, class Op>
__device__ T small_scan(T v, Op op, T identity, T *wtot, T *excl, T *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T o = shfl_up_any(x, d);
        if (lane >= d) x = op(o, x);
    }
    __syncthreads();
    if (lane == 31) wtot[w] = x;
    __syncthreads();
    if (w == 0) {
        T t = wtot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const T o = shfl_up_any(t, d);
            if (lane >= d) t = op(o, t);
        }
        wtot[lane] = t;
    }
    __syncthreads();
    const T before = w > 0 ? wtot[w - 1] : identity;
    const T incl = op(before, x);
    const T ex_in_warp = shfl_up_any(x, 1);
    *excl = lane > 0 ? op(before, ex_in_warp) : before;
    *total = wtot[kSW - 1];
    __syncthreads();
    return incl;
}

struct SumOp64 {
    __device__ uint64_t operator()(uint64_t a, uint64_t b) const { return a + b; }
};
struct MaxOp32 {
    __device__ int32_t operator()(int32_t a, int32_t b) const { return a > b ? a : b; }
};

__global__ void __launch_bounds__(kST, 1) k_plan_small(const __grid_constant__ PlanArgs a) {
    extern __shared__ __align__(16) unsigned char sraw[];
    SmallSmem &S = *reinterpret_cast<SmallSmem *>(sraw);
    __shared__ uint64_t w64[kSW];
    __shared__ Seg wseg[kSW];
    __shared__ int32_t w32[kSW];
    __shared__ CAgg wc[kSW];
    __shared__ uint32_t s_bits;
    __shared__ unsigned long long s_or, s_and;
    __shared__ uint32_t s_orn, s_andn, s_ore, s_ande;
    // This kernel always runs just before k_plan on the same stream, so it
    // clears k_plan's control block (barrier counter, flags) for it: one
    // operation fewer per plan than a separate memset.
    static_assert(sizeof(PlanCtl) % 4 == 0, "cleared in 4-byte words");
    for (uint32_t i = threadIdx.x; i < sizeof(PlanCtl) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(a.ctl)[i] = 0;
    const uint64_t R = *a.num_runs;
    if (!plan_is_small(a, R)) return;
    const uint32_t tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const uint32_t L = a.table_lanes;
    if (tid == 0) {
        s_bits = 0;
        s_or = 0;
        s_and = ~0ull;
        s_orn = 0;
        s_andn = ~0u;
        s_ore = 0;
        s_ande = 1;
        a.counts[0] = a.counts[1] = a.counts[2] = 0;
    }
    __syncthreads();

    // ---- step 1, table level: lane_first, zero-size slots, empty lanes
    uint64_t carry = 0, lensum = 0;
    uint32_t bits = 0;
    for (uint32_t b0 = 0; b0 < L; b0 += kST) {
        const uint32_t i = b0 + tid;
        uint64_t v = 0;
        if (i < L) {
            v = a.rpl[i];
            const uint32_t len = a.seg_len[i];
            if (len == 0 && (i & 1u) == 0) bits |= KVX_S_ZERO_LEN;  // zero-size K slot
            if (v == 0 && a.B > 0) bits |= KVX_S_COVERAGE;
            lensum += len;
        }
        uint64_t ex, tot;
        small_scan(v, SumOp64(), (uint64_t)0, w64, &ex, &tot);
        if (i < L) {
            S.lf[i] = (uint32_t)(carry + ex);
            a.lane_first[i] = (uint32_t)(carry + ex);
        }
        carry += tot;
    }
    {
        uint64_t ex, lentot;
        small_scan(lensum, SumOp64(), (uint64_t)0, w64, &ex, &lentot);
        if (tid == 0) {
            S.lf[L] = (uint32_t)carry;
            a.lane_first[L] = (uint32_t)carry;
        }
        bits = __reduce_or_sync(0xFFFFFFFFu, bits);
        if (lane == 0 && bits) atomicOr(&s_bits, bits);
        __syncthreads();
        uint32_t st = s_bits;
        bool stop = false;
        if (carry != R) {
            st |= KVX_S_ARRAYS;
            stop = true;
        } else if ((unsigned __int128)a.B * (unsigned __int128)lentot >= ((unsigned __int128)1 << 63)) {
            st |= KVX_S_CAPACITY;
            stop = true;
        }
        if (stop) {
            if (tid == 0) atomicOr(a.status, st);
            return;
        }
    }
    __syncthreads();

    // ---- step 1 per run + step 2 decode (runs 2*tid, 2*tid + 1)
    const uint32_t r0 = 2 * tid;
    bits = 0;
    unsigned long long o = 0, an = ~0ull;
    uint32_t on = 0, ann = ~0u, oe = 0, ae = 1;
    Seg agg{0, 0, 0};
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t r = r0 + j;
        if (r >= R) continue;
        uint32_t lo = 0, hi = L;  // lane: largest l with lf[l] <= r
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (S.lf[mid] <= r) lo = mid; else hi = mid;
        }
        const uint32_t l = lo;
        const uint64_t base = a.run_base[r];
        const int64_t stride = a.run_stride[r];
        const uint32_t cnt = a.run_count[r];
        const uint32_t len = __ldg(a.seg_len + l);
        const uint32_t node = __ldg(a.numa + l);
        S.base[r] = base;
        S.stride[r] = stride;
        S.count[r] = cnt;
        S.lane[r] = l;
        S.len[r] = len;
        S.node[r] = node;
        if (cnt == 0) bits |= KVX_S_ZERO_COUNT;
        if (cnt == 1 && stride != 0) bits |= KVX_S_STRIDE1;
        if (cnt >= 1) {
            const __int128 first = (__int128)base;
            const __int128 last = first + (__int128)(cnt - 1) * (__int128)stride;
            const __int128 hi2 = last > first ? last : first;
            if (last < 0 || hi2 + (__int128)len > (__int128)a.pool_bytes) bits |= KVX_S_SPAN;
        }
        agg = SegOp()(agg, Seg{cnt, r == S.lf[l] ? 1u : 0u, 0});
        o |= base;
        an &= base;
        on |= node;
        ann &= node;
        oe |= len == 0;
        ae &= len == 0;
    }
    {
        Seg ex, tot;
        small_scan(agg, SegOp(), Seg{0, 0, 0}, wseg, &ex, &tot);
        uint64_t blk = ex.sum;
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t r = r0 + j;
            if (r >= R) continue;
            const uint32_t l = S.lane[r];
            if (r == S.lf[l]) blk = 0;
            S.block[r] = (uint32_t)blk;
            a.run_block[r] = (uint32_t)blk;
            blk += S.count[r];
            if (r + 1 == S.lf[l + 1] && blk != a.B) bits |= KVX_S_COVERAGE;
        }
    }
    bits = __reduce_or_sync(0xFFFFFFFFu, bits);
    on = __reduce_or_sync(0xFFFFFFFFu, on);
    ann = __reduce_and_sync(0xFFFFFFFFu, ann);
    oe = __reduce_or_sync(0xFFFFFFFFu, oe);
    ae = __reduce_and_sync(0xFFFFFFFFu, ae);
    {
        const uint32_t o_lo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)o);
        const uint32_t o_hi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(o >> 32));
        const uint32_t a_lo = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)an);
        const uint32_t a_hi = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)(an >> 32));
        if (lane == 0) {
            if (bits) atomicOr(&s_bits, bits);
            atomicOr(&s_or, ((unsigned long long)o_hi << 32) | o_lo);
            atomicAnd(&s_and, ((unsigned long long)a_hi << 32) | a_lo);
            atomicOr(&s_orn, on);
            atomicAnd(&s_andn, ann);
            if (oe) atomicOr(&s_ore, 1u);
            if (!ae) atomicAnd(&s_ande, 0u);
        }
    }
    __syncthreads();
    if (s_bits) {
        if (tid == 0) atomicOr(a.status, s_bits);
        return;
    }

    // ---- step 2: stable LSD radix sort of run indices on (node, empty, base);
    // a table already in key order (a bump-allocated holder whose lanes are
    // numbered by address) needs no pass
    bool in_order = true;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t y = r0 + j;
        if (y == 0 || y >= R) continue;
        const uint32_t x = y - 1;
        const bool ex = S.len[x] == 0, ey = S.len[y] == 0;
        const bool le = S.node[x] != S.node[y] ? S.node[x] < S.node[y]
                        : ex != ey              ? !ex
                                                : S.base[x] <= S.base[y];
        in_order = in_order && le;
    }
    const bool sorted_already = __syncthreads_and(in_order) != 0;
    uint32_t act[13], nact = 0;
    if (R > 1 && !sorted_already) nact = plan_digits(s_or ^ s_and, s_ore ^ s_ande, s_orn ^ s_andn, act);
    for (uint32_t r = tid; r < R; r += kST) S.idx[0][r] = (uint16_t)r;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (uint32_t k = 0; k < nact; k++) {
        const uint16_t *in = S.idx[k & 1];
        uint16_t *out = S.idx[(k + 1) & 1];
        const uint32_t dig = act[k];
        for (uint32_t i = tid; i < kSW * kDigits; i += kST) (&S.wcnt[0][0])[i] = 0;
        __syncthreads();
        uint32_t item[2], d[2], pos[2];
#pragma unroll
        for (int j = 0; j < 2; j++) {  // warp-contiguous: position w*64 + j*32 + lane
            const uint32_t p = w * 64 + j * 32 + lane;
            d[j] = kDigits;
            item[j] = 0;
            if (p < R) {
                item[j] = in[p];
                d[j] = digit_of(S.base[item[j]], S.node[item[j]], S.len[item[j]] == 0 ? 1u : 0u, dig);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t peers = digit_peers(d[j]);
            const uint32_t rank = __popc(peers & lt_mask);
            const uint32_t before = d[j] < kDigits ? S.wcnt[w][d[j]] : 0;
            __syncwarp();
            if (d[j] < kDigits && rank == 0) S.wcnt[w][d[j]] = (uint16_t)(before + __popc(peers));
            __syncwarp();
            pos[j] = before + rank;
        }
        __syncthreads();
        uint64_t dtot = 0;
        if (tid < kDigits) {
            uint32_t acc = 0;
            for (int ww = 0; ww < kSW; ww++) {
                const uint32_t c = S.wcnt[ww][tid];
                S.wcnt[ww][tid] = (uint16_t)acc;
                acc += c;
            }
            dtot = acc;
        }
        {
            uint64_t ex, tot;
            small_scan(dtot, SumOp64(), (uint64_t)0, w64, &ex, &tot);
            if (tid < kDigits) S.dbase[tid] = (uint32_t)ex;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 2; j++) {
            if (d[j] >= kDigits) continue;
            const uint32_t dst = S.dbase[d[j]] + S.wcnt[w][d[j]] + pos[j];
            if (dst < R) out[dst] = (uint16_t)item[j];  // always: a permutation
        }
        __syncthreads();
    }
    const uint16_t *sorted = S.idx[nact & 1];

    // ---- step 3: compat, stretch starts, group starts (positions 2*tid, +1)
    int32_t mx = -1;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t p = r0 + j;
        if (p >= R) continue;
        bool c = false;
        if (p > 0) {
            const uint32_t x = sorted[p], y = sorted[p - 1];
            c = S.node[x] == S.node[y] && S.block[x] == S.block[y] && S.count[x] == S.count[y] &&
                S.stride[x] == S.stride[y] && S.base[x] == S.base[y] + S.len[y];
        }
        S.compat[p] = c ? 1 : 0;
        if (!c) mx = (int32_t)p;
    }
    {
        int32_t ex, tot;
        small_scan(mx, MaxOp32(), (int32_t)-1, w32, &ex, &tot);
        int32_t st = ex;  // stretch start before this thread's first position
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t p = r0 + j;
            if (p >= R) continue;
            const bool c = S.compat[p] != 0;
            if (!c) st = (int32_t)p;
            const uint32_t x = sorted[p];
            const uint32_t cnt = S.count[x];
            const int64_t stride = S.stride[x];
            if (cnt == 1) {
                S.flag[p] = c ? 0 : 1;
                continue;
            }
            if (stride <= 0) {
                S.flag[p] = 1;  // a non-positive stride never fits: one run per group
                continue;
            }
            const uint64_t ustride = (uint64_t)stride;
            const uint64_t O = S.base[x] - S.base[sorted[st > 0 ? st : 0]];
            const uint64_t E = O + S.len[x];
            if (E <= ustride) {
                S.flag[p] = c ? 0 : 1;
            } else if (O <= ustride) {
                // first run that outgrows the stretch's first group: walk the rest
                S.flag[p] = 1;
                uint64_t cur = S.base[x];
                for (uint32_t q = p + 1; q < R && S.compat[q]; q++) {
                    const uint32_t y = sorted[q];
                    if (S.base[y] + S.len[y] - cur > ustride) {
                        S.flag[q] = 1;
                        cur = S.base[y];
                    } else {
                        S.flag[q] = 0;
                    }
                }
            }
        }
    }
    __syncthreads();

    // ---- group numbering, records, carve and reads
    uint64_t gcount = 0;
    int32_t glast = -1;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t p = r0 + j;
        if (p < R && S.flag[p]) {
            gcount++;
            glast = (int32_t)p;
        }
    }
    uint64_t gex, gtot;
    small_scan(gcount, SumOp64(), (uint64_t)0, w64, &gex, &gtot);
    int32_t lex, ltot;
    small_scan(glast, MaxOp32(), (int32_t)-1, w32, &lex, &ltot);
    if (gtot > a.group_cap) {
        if (tid == 0) atomicOr(a.status, KVX_S_CAPACITY);
        return;
    }
    uint64_t gid_run = gex;
    int32_t gs = lex;
    kvx_group G[2];
    bool is_end[2] = {false, false};
    uint32_t gids[2] = {0, 0};
    CAgg c{0, 0};
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const uint32_t p = r0 + j;
        if (p >= R) continue;
        if (S.flag[p]) {
            gid_run++;
            gs = (int32_t)p;
        }
        const uint32_t gid = (uint32_t)(gid_run - 1);
        const uint32_t x = sorted[p];
        const uint32_t x0 = sorted[gs > 0 ? gs : 0];
        const uint64_t off = S.base[x] - S.base[x0];
        a.run_group[x] = gid;
        a.run_off[x] = off;
        gids[j] = gid;
        if (p + 1 == R || S.flag[p + 1]) {
            is_end[j] = true;
            kvx_group &g = G[j];
            g.base = S.base[x0];
            g.stride = S.stride[x0];
            g.chunk = off + S.len[x];
            g.local = 0;
            g.block = S.block[x0];
            g.count = S.count[x0];
            g.node = S.node[x0];
            g.dense = group_dense(g.count, g.stride, g.chunk) ? 1u : 0u;
            c.bytes += (uint64_t)g.count * g.chunk;
            c.descs += group_pieces(g);
        }
    }
    CAgg cex, ctot;
    small_scan(c, COp(), CAgg{0, 0}, wc, &cex, &ctot);
    if (ctot.descs > a.desc_cap) {
        if (tid == 0) atomicOr(a.status, KVX_S_CAPACITY);
        return;
    }
    CAgg cur = cex;
    const uint64_t M = KVX_MAX_READ_BYTES;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        if (!is_end[j]) continue;
        kvx_group g = G[j];
        g.local = cur.bytes;
        a.groups[gids[j]] = g;
        uint64_t dd = cur.descs;
        if (g.dense) {
            const uint64_t total = (uint64_t)g.count * g.chunk;
            for (uint64_t off = 0; off < total; off += M, dd++)
                a.descs[dd] = kvx_desc{g.base + off, g.local + off, total - off < M ? total - off : M, gids[j], 0};
        } else if (g.chunk > 0) {  // a group of empty runs has no read
            for (uint64_t i = 0; i < g.count; i++) {
                const uint64_t rb = g.base + i * (uint64_t)g.stride;
                const uint64_t lb = g.local + i * g.chunk;
                for (uint64_t off = 0; off < g.chunk; off += M, dd++)
                    a.descs[dd] = kvx_desc{rb + off, lb + off, g.chunk - off < M ? g.chunk - off : M, gids[j], 0};
            }
        }
        cur.bytes += (uint64_t)g.count * g.chunk;
        cur.descs += group_pieces(g);
    }
    if (tid == 0) {
        a.counts[0] = gtot;
        a.counts[1] = ctot.descs;
        a.counts[2] = ctot.bytes;
    }
}

// Shared memory that two stages use in turn: lane_first and the first
// histogram while the runs are decoded and keyed, then a radix pass's
// counters.  Sharing it keeps the block at about 23 KB, small enough to sit
// beside a bulk-copy block on one SM (a transfer can be planned while another
// copies).
struct KeyStage {
    uint32_t lf[kLaneSmem];
    uint32_t hist[kDigits];
};
union PlanStages {
    KeyStage keys;
    SortCounters sort;
    uint64_t tile_base[kTile];  // the adjacent-cut phase: bases of the tile's sorted runs
};

// Every phase over tiles of kT * IPT runs.  The shared memory is the
// kernel's: every tile size uses the same 23 KB.
template <int IPT>
__device__ void plan_tiles(const PlanArgs &a, uint64_t R_in, uint64_t R, ScanSmem &sm, uint32_t *s_act,
                           uint32_t &s_nact, PlanStages &st) {
    uint32_t *s_lf = st.keys.lf;
    const uint32_t nt = (uint32_t)ceil_div(R, kT * IPT);
    const uint32_t P = nt < gridDim.x ? (nt ? nt : 1) : gridDim.x;
    if (threadIdx.x == 0) {
        uint32_t vb = blockIdx.x;
        uint32_t nsmid;  // SM ids are below this
        asm volatile("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
        if (gridDim.x > a.sms && nt <= a.sms && nsmid <= 256) {
            // two blocks per SM and at most a tile per SM: the first block to
            // start on each SM works (numbered in arrival order), so no two
            // working blocks share an SM; every SM runs one, all of them resident
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            const uint32_t rank = atomicAdd(&a.ctl->sm_rank[smid < 256 ? smid : 255], 1u);
            vb = rank == 0 ? atomicAdd(&a.ctl->primaries, 1u) : ~0u;
        }
        g_vb = vb;
    }
    __syncthreads();
    const uint32_t vb = g_vb;
    if (vb >= P) return;

    if (vb == 0) phase_init(a, R_in);
    PLAN_BARRIER();
    if (__ldcg(&a.ctl->fail)) return;

    phase_decode<IPT>(a, R, nt, P, vb, sm, s_lf);
    PLAN_BARRIER();
    if (threadIdx.x == 0) s_nact = active_digits(a, R, s_act);
    __syncthreads();
    const uint32_t nact = s_nact;
    phase_keys<IPT>(a, R, nt, P, vb, nact, nact ? s_act[0] : 0, sm, s_lf, st.keys.hist);
    PLAN_BARRIER();
    if (__ldcg(&a.ctl->st) != 0) return;  // counts stay 0

    for (uint32_t k = 0; k < nact; k++) {
        const SortItem *in = (k & 1) ? a.items1 : a.items0;
        SortItem *out = (k & 1) ? a.items0 : a.items1;
        if (kLocalHist<IPT> && k > 0) {  // pass 0's histograms came with the keys
            phase_hist<IPT>(a, R, nt, P, vb, in, a.hist[k % 3], a.ghist[k % 3], s_act[k], st.keys.hist);
            PLAN_BARRIER();
        }
        const bool has_next = k + 1 < nact;
        phase_sort_pass<IPT>(a, R, nt, P, vb, in, out, a.hist[k % 3], a.hist[(k + 1) % 3],
                             a.hist[(k + 2) % 3], a.ghist[k % 3], a.ghist[(k + 1) % 3],
                             a.ghist[(k + 2) % 3], s_act[k], has_next, has_next ? s_act[k + 1] : 0,
                             k + 2 < nact, st.sort);
        PLAN_BARRIER();
    }
    const SortItem *sorted = (nact & 1) ? a.items1 : a.items0;

    // The 2048-run tile body carries each tile through groups and the carve
    // in the same phase; the smaller bodies (tables of a few dozen tiles,
    // one short tile per block) measured faster with those steps as their
    // own phases, after barriers.
    constexpr bool kFuse = IPT == kIPT;
    phase_post_sort<IPT, kFuse>(a, R, nt, P, vb, sorted, sm, st.tile_base);
    PLAN_BARRIER();
    if (__ldcg(&a.ctl->walked)) {
        // Some stretch outgrows its stride: the cut again, phase by phase,
        // with the walks along such stretches in order, then the counts.
        phase_cut<IPT>(a, R, nt, P, vb, sorted, sm);
        PLAN_BARRIER();
        phase_count<IPT>(a, R, nt, P, vb, sm);
        PLAN_BARRIER();
    } else if (kFuse) {
        return;  // every tile was grouped and carved in that phase
    }
    const GAgg gall = reduce_prefix(a.gagg, nt, GOp(), GAgg{0, -1}, sm.g);
    if (gall.n > a.group_cap) {
        if (vb == 0 && threadIdx.x == 0) {
            raise_plan(a, KVX_S_CAPACITY);
            a.counts[0] = a.counts[1] = a.counts[2] = 0;
        }
        return;
    }
    phase_groups<IPT>(a, R, nt, P, vb, sorted, sm);
    PLAN_BARRIER();
    const CAgg call = reduce_prefix(a.cagg, nt, COp(), CAgg{0, 0}, sm.c);
    if (call.descs > a.desc_cap) {
        if (vb == 0 && threadIdx.x == 0) {
            raise_plan(a, KVX_S_CAPACITY);
            a.counts[0] = a.counts[1] = a.counts[2] = 0;
        }
        return;
    }
    if (vb == 0 && threadIdx.x == 0) {
        a.counts[0] = gall.n;
        a.counts[1] = call.descs;
        a.counts[2] = call.bytes;
    }
    phase_emit<IPT>(a, R, nt, P, vb, sm);
}

// The tile size follows the run count, which only the device knows: the
// smallest of 512, 1024 and 2048 runs whose tiles all get a block.
__host__ __device__ __forceinline__ bool tiles_fit(uint64_t R, int ipt, uint64_t blocks) {
    const uint64_t n = ceil_div(R, (uint64_t)kT * ipt);
    return n <= kSmallTiles && n <= blocks;
}

// The block's shared memory, at namespace scope so that the out-of-line
// bodies below address it as shared memory; one copy per block.
__shared__ ScanSmem g_sm;
__shared__ uint32_t g_act[13];
__shared__ uint32_t g_nact;
__shared__ PlanStages g_st;
__shared__ PlanArgs g_args;  // the launch's arguments, for the out-of-line bodies

// The 512- and 1024-run tile bodies are called, not inlined: inlined next to
// the 2048-run body they made the kernel plan 2048-run tables 5 % slower.
template <int IPT>
__device__ __noinline__ void plan_tiles_call(uint64_t R_in, uint64_t R) {
    plan_tiles<IPT>(g_args, R_in, R, g_sm, g_act, g_nact, g_st);
}

__global__ void __launch_bounds__(kT, 2) k_plan(const __grid_constant__ PlanArgs a) {
    const uint64_t R_in = *a.num_runs;
    if (plan_is_small(a, R_in)) return;  // planned by k_plan_small
    const uint64_t R = R_in <= a.run_cap ? R_in : 0;
    const int ipt = tiles_fit(R, 2, gridDim.x) ? 2 : tiles_fit(R, 4, gridDim.x) ? 4 : kIPT;
    if (ipt == kIPT) {
        plan_tiles<kIPT>(a, R_in, R, g_sm, g_act, g_nact, g_st);
        return;
    }
    if (threadIdx.x == 0) g_args = a;
    __syncthreads();
    if (ipt == 2)
        plan_tiles_call<2>(R_in, R);
    else
        plan_tiles_call<4>(R_in, R);
}

struct Ws {
    PlanCtl *ctl;
    uint32_t *run_lane;
    Seg *seg;
    SortItem *items[2];
    uint32_t *hist[3];
    uint32_t *ghist[3];
    uint64_t *run_bl;
    uint8_t *compat;
    uint8_t *gflag;
    int64_t *segmax;
    GAgg *gagg;
    CAgg *cagg;
    GAgg *gthr;
    CAgg *cthr;
    uint32_t *ready_g;
    uint32_t *ready_c;
};

// Tiles a table of up to run_cap runs can be cut into (any tile size).
uint64_t tile_cap(uint64_t run_cap) {
    const uint64_t big = ceil_div(run_cap ? run_cap : 1, kTile);
    const uint64_t small = ceil_div(run_cap ? run_cap : 1, (uint64_t)kT * 2);
    return big > kSmallTiles ? big : (small < kSmallTiles ? small : kSmallTiles);
}

Ws carve(void *base, uint64_t run_cap, size_t *bytes) {
    const uint64_t ntc = tile_cap(run_cap);
    Carver c(base);
    Ws w;
    w.ctl = c.take<PlanCtl>(1);
    w.run_lane = c.take<uint32_t>(run_cap);
    w.seg = c.take<Seg>(ntc);
    w.items[0] = c.take<SortItem>(run_cap);
    w.items[1] = c.take<SortItem>(run_cap);
    for (int i = 0; i < 3; i++) w.hist[i] = c.take<uint32_t>(kDigits * ntc);
    for (int i = 0; i < 3; i++) w.ghist[i] = c.take<uint32_t>(kDigits * ceil_div(ntc, (uint64_t)kHistGroup));
    w.run_bl = c.take<uint64_t>(run_cap);
    w.compat = c.take<uint8_t>(run_cap);
    w.gflag = c.take<uint8_t>(run_cap + 1);
    w.segmax = c.take<int64_t>(ntc);
    w.gagg = c.take<GAgg>(ntc);
    w.cagg = c.take<CAgg>(ntc);
    w.gthr = c.take<GAgg>(ntc * kT);
    w.cthr = c.take<CAgg>(ntc * kT);
    w.ready_g = c.take<uint32_t>(ntc);
    w.ready_c = c.take<uint32_t>(ntc);
    *bytes = c.off;
    return w;
}

// Blocks per SM the planner's grid may take, per device (0: the default, 1).
std::atomic<uint32_t> g_plan_share[64];
uint32_t plan_share() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    const uint32_t s = g_plan_share[dev].load(std::memory_order_relaxed);
    return s ? s : 1;
}

// Blocks of k_plan's grid: the share (blocks per SM) times the SMs.  One per
// SM, the default, lets the whole grid be resident beside a bulk copy (one
// planner block fits next to a copy block), so a transfer is planned while
// another copies; tables of more than one 2048-run tile per SM then give a
// block several tiles (many_small: 284 tiles, 2 per block).  Two per SM (the
// kernel's register budget allows two) serve an otherwise idle device.
int plan_max_blocks() { return (int)plan_share() * sm_count(); }

}  // namespace
}  // namespace kvx

namespace kvx {
// Launches the flag-wait diagnostic for kvx_selftest_timeouts.
kvx_status launch_selftest_flag_wait(uint32_t *status, cudaStream_t s) {
    k_selftest_flag<<<1, 32, 0, s>>>(status);
    KVX_LAUNCHED();
    return KVX_OK;
}
}  // namespace kvx

using namespace kvx;

extern "C" uint64_t kvx_desc_capacity(uint32_t B, uint32_t L, uint64_t seg_bytes_sum) {
    const unsigned __int128 slab = (unsigned __int128)B * seg_bytes_sum;
    return (uint64_t)B * L + (uint64_t)((slab + KVX_MAX_READ_BYTES - 1) / KVX_MAX_READ_BYTES);
}

extern "C" kvx_status kvx_plan_bounds(uint32_t B, uint32_t L, uint64_t num_runs,
                                      uint64_t max_seg_bytes_total, uint64_t *group_cap,
                                      uint64_t *desc_cap) {
    if (!group_cap || !desc_cap) return KVX_EINVAL;
    const uint64_t runs_max = kvx_run_capacity(B, L);
    if (num_runs > runs_max) return KVX_EINVAL;  // no greedy encoding of B blocks has that many
    // every group holds at least one run
    *group_cap = num_runs ? num_runs : runs_max;
    *desc_cap = kvx_desc_capacity(B, L, max_seg_bytes_total);
    return KVX_OK;
}

extern "C" kvx_status kvx_plan_set_sm_share(uint32_t blocks_per_sm) {
    if (blocks_per_sm != 1 && blocks_per_sm != 2) return KVX_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return KVX_ECUDA;
    }
    kvx::g_plan_share[dev].store(blocks_per_sm, std::memory_order_relaxed);
    return KVX_OK;
}

extern "C" size_t kvx_plan_workspace_size(uint32_t L, uint64_t run_capacity, uint64_t pool_bytes) {
    (void)L;
    (void)pool_bytes;
    size_t bytes = 0;
    carve(nullptr, run_capacity, &bytes);
    return bytes;
}

extern "C" kvx_status kvx_plan_groups(const uint32_t *runs_per_lane, uint32_t table_lanes,
                                      const uint64_t *run_base, const int64_t *run_stride,
                                      const uint32_t *run_count, const uint64_t *num_runs,
                                      uint64_t run_capacity, uint32_t B, const uint32_t *seg_len,
                                      const uint32_t *numa, uint32_t template_lanes,
                                      uint64_t pool_bytes, kvx_group *groups,
                                      uint64_t group_capacity, kvx_desc *descs,
                                      uint64_t desc_capacity, uint32_t *lane_first,
                                      uint32_t *run_block, uint32_t *run_group, uint64_t *run_off,
                                      uint64_t *counts, uint32_t *status, void *ws,
                                      size_t ws_bytes, void *stream) {
    if (!num_runs || !counts || !status || !ws || !lane_first) return KVX_EINVAL;
    if (table_lanes && !runs_per_lane) return KVX_EINVAL;
    if (template_lanes && (!seg_len || !numa)) return KVX_EINVAL;
    if (run_capacity && (!run_base || !run_stride || !run_count || !run_block || !run_group ||
                         !run_off))
        return KVX_EINVAL;
    // run indices travel in 31 bits of the sort records
    if (run_capacity > (1ull << 31) || table_lanes == 0xFFFFFFFFu) return KVX_EINVAL;
    if ((group_capacity && !groups) || (desc_capacity && !descs)) return KVX_EINVAL;
    size_t need = 0;
    Ws w = carve(ws, run_capacity, &need);
    if (ws_bytes < need) return KVX_EINVAL;
    cudaStream_t s = as_stream(stream);
    PlanArgs a;
    a.rpl = runs_per_lane;
    a.table_lanes = table_lanes;
    a.template_lanes = template_lanes;
    a.run_base = run_base;
    a.run_stride = run_stride;
    a.run_count = run_count;
    a.num_runs = num_runs;
    a.run_cap = run_capacity;
    a.B = B;
    a.seg_len = seg_len;
    a.numa = numa;
    a.pool_bytes = pool_bytes;
    a.groups = groups;
    a.group_cap = group_capacity;
    a.descs = descs;
    a.desc_cap = desc_capacity;
    a.lane_first = lane_first;
    a.run_block = run_block;
    a.run_group = run_group;
    a.run_off = run_off;
    a.counts = counts;
    a.status = status;
    a.out16 = ((reinterpret_cast<uintptr_t>(groups) | reinterpret_cast<uintptr_t>(descs)) & 15) == 0;
    a.sms = (uint32_t)sm_count();
    a.ctl = w.ctl;
    a.run_lane = w.run_lane;
    a.seg = w.seg;
    a.items0 = w.items[0];
    a.items1 = w.items[1];
    for (int i = 0; i < 3; i++) {
        a.hist[i] = w.hist[i];
        a.ghist[i] = w.ghist[i];
    }
    a.run_bl = w.run_bl;
    a.compat = w.compat;
    a.gflag = w.gflag;
    a.segmax = w.segmax;
    a.gagg = w.gagg;
    a.cagg = w.cagg;
    a.gthr = w.gthr;
    a.cthr = w.cthr;
    a.ready_g = w.ready_g;
    a.ready_c = w.ready_c;
    static bool small_ready[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return KVX_ECUDA;
    if (!small_ready[dev]) {
        if (cudaFuncSetAttribute(k_plan_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(SmallSmem)) != cudaSuccess)
            return KVX_ECUDA;
        small_ready[dev] = true;
    }
    k_plan_small<<<1, kST, sizeof(SmallSmem), s>>>(a);  // also clears k_plan's control block
    KVX_LAUNCHED();
    const uint64_t ntc = tile_cap(run_capacity);
    const int maxb = plan_max_blocks();
    const unsigned grid = (unsigned)(ntc < (uint64_t)maxb ? ntc : (uint64_t)maxb);
    void *args[] = {&a};
    if (cudaLaunchCooperativeKernel((const void *)k_plan, dim3(grid), dim3(kT), args, 0, s) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return KVX_ECUDA;
    }
    note_launch();
    return KVX_OK;
}
