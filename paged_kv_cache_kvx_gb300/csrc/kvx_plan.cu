// Transfer planning (pegaflow PR #350, Requester plan_transfer steps 1-4 and
// the READ splitting paragraph) as a chain of data-parallel kernels:
//
//   k_plan_init    step 1, table-level checks; lane_first = prefix of
//                  runs_per_lane
//   k_plan_decode  step 1 per run (zero count, one-block stride, span);
//                  lane of each run; tile sums for the per-lane block prefix;
//                  key bits that differ (for the radix passes)
//   k_plan_keys    step 2: first block of each run (segmented prefix of
//                  counts within its lane), per-lane coverage, sort items,
//                  first radix histogram
//   k_plan_sort    step 2: stable LSD radix passes on (node, base); equal
//                  keys keep run order = (lane, first block) order
//   k_plan_adjacent step 3: sorted records; compat(p) = same node, first
//                  block, count and stride as p-1 and base-adjacent to it
//   k_plan_cut     step 3: group starts; the "grown chunk fits the stride"
//                  cut inside a compatible stretch
//   k_plan_count   group numbering
//   k_plan_groups  group records, run_group / run_off, per-group bytes and
//                  read pieces
//   k_plan_emit    step 4: slab carve (groups back to back) and descriptors
//                  (one per dense group / per block, split at 32 MiB)
//
// Cross-block results move through per-tile aggregates that the last block
// of a kernel to finish scans (atomic ticket; no block ever waits on
// another).  All per-run kernels use tiles of 2048 runs, 8 per thread.
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kT = 256;
constexpr int kIPT = 8;
constexpr uint32_t kTile = kT * kIPT;
constexpr int kMaxPasses = 12;  // 8 base bytes + 4 node bytes
constexpr uint32_t kDigits = 256;

enum Ticket { TK_DECODE = 0, TK_KEYS, TK_SORT0, TK_ADJ = TK_SORT0 + kMaxPasses, TK_COUNT,
              TK_GROUPS, TK_N };

struct PlanCtl {
    uint32_t ticket[TK_N];
    uint32_t fail;
    uint32_t st;
    uint64_t R;
    uint32_t nt;
    uint32_t nactive;
    uint32_t active[kMaxPasses];
    unsigned long long or_base, and_base;
    uint32_t or_node, and_node;
    uint64_t ngroups;
};

struct SortItem {
    uint64_t base;
    uint32_t node;
    uint32_t r;
};

struct Rec {
    uint64_t base;
    int64_t stride;
    uint32_t len, block, count, node, r, pad;
};

// Segmented sum: value since the last segment head, and whether a head was seen.
struct Seg {
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
struct GAgg {
    uint64_t n;
    int64_t last;
};
struct GOp {
    __device__ GAgg operator()(const GAgg &a, const GAgg &b) const {
        return GAgg{a.n + b.n, a.last > b.last ? a.last : b.last};
    }
};
// Carve: slab bytes and descriptor count so far.
struct CAgg {
    uint64_t bytes;
    uint64_t descs;
};
struct COp {
    __device__ CAgg operator()(const CAgg &a, const CAgg &b) const {
        return CAgg{a.bytes + b.bytes, a.descs + b.descs};
    }
};

// Hillis-Steele block scan through shared memory (blockDim.x values).
// Returns the inclusive value; *excl gets the exclusive one, *total the
// block total.
template <class T, class Op>
__device__ T block_scan(T v, Op op, T identity, T *sh, T *excl, T *total) {
    const int tid = threadIdx.x;
    __syncthreads();
    sh[tid] = v;
    __syncthreads();
    for (int d = 1; d < (int)blockDim.x; d <<= 1) {
        T o = tid >= d ? sh[tid - d] : identity;
        __syncthreads();
        if (tid >= d) v = op(o, v);
        sh[tid] = v;
        __syncthreads();
    }
    *excl = tid > 0 ? sh[tid - 1] : identity;
    *total = sh[blockDim.x - 1];
    __syncthreads();
    return v;
}

// Load that bypasses L1: last blocks read what other blocks wrote in the
// same kernel.
template <class T>
__device__ __forceinline__ T ld_cg(const T *p) {
    static_assert(sizeof(T) % 8 == 0, "8-byte multiple");
    T v;
    const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p);
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(&v);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 8); i++) dst[i] = __ldcg(src + i);
    return v;
}

// Exclusive scan of n per-tile aggregates in place, by one block.
template <class T, class Op>
__device__ T block_scan_tiles(T *a, uint64_t n, Op op, T identity, T *sh) {
    T carry = identity;
    for (uint64_t base = 0; base < n; base += blockDim.x) {
        const uint64_t i = base + threadIdx.x;
        T v = identity;
        if (i < n) v = ld_cg(a + i);
        T ex, tot;
        block_scan(v, op, identity, sh, &ex, &tot);
        if (i < n) a[i] = op(carry, ex);
        carry = op(carry, tot);
    }
    __syncthreads();
    return carry;
}

__device__ __forceinline__ uint32_t digit_of(uint64_t base, uint32_t node, uint32_t dig) {
    return dig < 8 ? (uint32_t)(base >> (8 * dig)) & 0xFFu : (node >> (8 * (dig - 8))) & 0xFFu;
}

// Largest l with lane_first[l] <= r (lane_first has L + 1 entries).
__device__ __forceinline__ uint32_t lane_of(const uint32_t *lane_first, uint32_t L, uint64_t r) {
    uint32_t lo = 0, hi = L;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if ((uint64_t)__ldg(lane_first + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

struct Ws {
    PlanCtl *ctl;
    uint32_t *run_lane;
    Seg *seg;
    SortItem *items[2];
    uint32_t *hist[2];
    Rec *rec;
    uint8_t *compat;
    uint8_t *gflag;
    int64_t *segmax;
    GAgg *gagg;
    CAgg *cagg;
};

Ws carve(void *base, uint32_t L, uint64_t run_cap, size_t *bytes) {
    (void)L;
    const uint64_t ntc = ceil_div(run_cap ? run_cap : 1, kTile);
    Carver c(base);
    Ws w;
    w.ctl = c.take<PlanCtl>(1);
    w.run_lane = c.take<uint32_t>(run_cap);
    w.seg = c.take<Seg>(ntc);
    w.items[0] = c.take<SortItem>(run_cap);
    w.items[1] = c.take<SortItem>(run_cap);
    w.hist[0] = c.take<uint32_t>(kDigits * ntc);
    w.hist[1] = c.take<uint32_t>(kDigits * ntc);
    w.rec = c.take<Rec>(run_cap);
    w.compat = c.take<uint8_t>(run_cap);
    w.gflag = c.take<uint8_t>(run_cap + 1);
    w.segmax = c.take<int64_t>(ntc);
    w.gagg = c.take<GAgg>(ntc);
    w.cagg = c.take<CAgg>(ntc);
    *bytes = c.off;
    return w;
}

__device__ __forceinline__ void flag_fail(PlanCtl *ctl, uint32_t *status, uint32_t bits) {
    atomicOr(status, bits);
    atomicOr(&ctl->st, bits);
    ctl->fail = 1;
}

// ------------------------------------------------------------ step 1: table

__global__ void __launch_bounds__(1024)
k_plan_init(const uint32_t *__restrict__ rpl, uint32_t table_lanes, const uint64_t *num_runs,
            uint64_t run_cap, uint32_t B, const uint32_t *__restrict__ seg_len,
            uint32_t template_lanes, uint32_t *__restrict__ lane_first, uint64_t *counts,
            uint32_t *status, PlanCtl *ctl) {
    __shared__ uint64_t sh[33];
    __shared__ uint32_t s_bits;
    __shared__ uint64_t s_len;
    const uint32_t tid = threadIdx.x;
    if (tid < TK_N) ctl->ticket[tid] = 0;
    if (tid == 0) {
        s_bits = 0;
        s_len = 0;
        ctl->nactive = 0;
        ctl->or_base = 0;
        ctl->and_base = ~0ull;
        ctl->or_node = 0;
        ctl->and_node = ~0u;
        ctl->ngroups = 0;
        counts[0] = counts[1] = counts[2] = 0;
    }
    __syncthreads();
    uint32_t fail = 0, bits = 0;
    uint64_t R = 0;
    if (table_lanes != template_lanes) {
        bits = KVX_S_LANES;
        fail = 1;
    } else {
        const uint32_t L = table_lanes;
        uint64_t carry = 0, lensum = 0;
        uint32_t mybits = 0;
        for (uint32_t base = 0; base < L; base += blockDim.x) {
            const uint32_t i = base + tid;
            uint64_t v = 0;
            if (i < L) {
                v = rpl[i];
                const uint32_t len = seg_len[i];
                if (len == 0) mybits |= KVX_S_ZERO_LEN;
                if (v == 0 && B > 0) mybits |= KVX_S_COVERAGE;
                lensum += len;
            }
            uint64_t tot;
            const uint64_t ex = block_excl_sum<uint64_t>(v, sh, &tot);
            if (i < L) lane_first[i] = (uint32_t)(carry + ex);
            carry += tot;
        }
        mybits = __reduce_or_sync(0xFFFFFFFFu, mybits);
        if ((tid & 31) == 0 && mybits) atomicOr(&s_bits, mybits);
        uint64_t lentot;
        block_excl_sum<uint64_t>(lensum, sh, &lentot);
        if (tid == 0) s_len = lentot;
        __syncthreads();
        if (tid == 0) lane_first[L] = (uint32_t)carry;
        R = *num_runs;
        bits = s_bits;
        if (carry != R || R > run_cap) {
            bits |= KVX_S_ARRAYS;
            fail = 1;
        } else {
            const unsigned __int128 slab = (unsigned __int128)B * (unsigned __int128)s_len;
            if (slab >= ((unsigned __int128)1 << 63)) {
                bits |= KVX_S_CAPACITY;
                fail = 1;
            }
        }
    }
    if (tid == 0) {
        if (bits) atomicOr(status, bits);
        ctl->st = bits;
        ctl->fail = fail;
        ctl->R = fail ? 0 : R;
        ctl->nt = fail ? 0 : (uint32_t)ceil_div(R, kTile);
    }
}

// ----------------------------------------------------- step 1/2: per run

__global__ void __launch_bounds__(kT)
k_plan_decode(const uint32_t *__restrict__ lane_first, uint32_t L,
              const uint64_t *__restrict__ run_base, const int64_t *__restrict__ run_stride,
              const uint32_t *__restrict__ run_count, const uint32_t *__restrict__ seg_len,
              const uint32_t *__restrict__ numa, uint64_t pool_bytes, uint32_t *status,
              PlanCtl *ctl, uint32_t *__restrict__ run_lane, Seg *seg) {
    __shared__ Seg sh[kT];
    __shared__ uint32_t s_bits;
    __shared__ unsigned long long s_or, s_and;
    __shared__ uint32_t s_orn, s_andn;
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    if (threadIdx.x == 0) {
        s_bits = 0;
        s_or = 0;
        s_and = ~0ull;
        s_orn = 0;
        s_andn = ~0u;
    }
    __syncthreads();
    Seg agg{0, 0, 0};
    uint32_t bits = 0;
    unsigned long long o = 0, a = ~0ull;
    uint32_t on = 0, an = ~0u;
    if (tile < nt) {
        const uint64_t r0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
        for (int j = 0; j < kIPT; j++) {
            const uint64_t r = r0 + j;
            if (r >= R) break;
            const uint32_t l = lane_of(lane_first, L, r);
            run_lane[r] = l;
            const uint64_t base = run_base[r];
            const int64_t stride = run_stride[r];
            const uint32_t cnt = run_count[r];
            const uint32_t len = seg_len[l];
            const uint32_t node = numa[l];
            if (cnt == 0) bits |= KVX_S_ZERO_COUNT;
            if (cnt == 1 && stride != 0) bits |= KVX_S_STRIDE1;
            if (cnt >= 1) {
                const __int128 first = (__int128)base;
                const __int128 last = first + (__int128)(cnt - 1) * (__int128)stride;
                const __int128 hi = last > first ? last : first;
                if (last < 0 || hi + (__int128)len > (__int128)pool_bytes) bits |= KVX_S_SPAN;
            }
            const bool head = r == __ldg(lane_first + l);
            agg = SegOp()(agg, Seg{cnt, head ? 1u : 0u, 0});
            o |= base;
            a &= base;
            on |= node;
            an &= node;
        }
    }
    // lanes with no valid item keep the identities; one shared atomic per warp
    bits = __reduce_or_sync(0xFFFFFFFFu, bits);
    on = __reduce_or_sync(0xFFFFFFFFu, on);
    an = __reduce_and_sync(0xFFFFFFFFu, an);
    const uint32_t o_lo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)o);
    const uint32_t o_hi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(o >> 32));
    const uint32_t a_lo = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)a);
    const uint32_t a_hi = __reduce_and_sync(0xFFFFFFFFu, (uint32_t)(a >> 32));
    if ((threadIdx.x & 31) == 0) {
        if (bits) atomicOr(&s_bits, bits);
        atomicOr(&s_or, ((unsigned long long)o_hi << 32) | o_lo);
        atomicAnd(&s_and, ((unsigned long long)a_hi << 32) | a_lo);
        atomicOr(&s_orn, on);
        atomicAnd(&s_andn, an);
    }
    Seg ex, tot;
    block_scan(agg, SegOp(), Seg{0, 0, 0}, sh, &ex, &tot);
    if (threadIdx.x == 0 && tile < nt) {
        seg[tile] = tot;
        if (s_bits) {
            atomicOr(status, s_bits);
            atomicOr(&ctl->st, s_bits);
        }
        atomicOr(&ctl->or_base, s_or);
        atomicAnd(&ctl->and_base, s_and);
        atomicOr(&ctl->or_node, s_orn);
        atomicAnd(&ctl->and_node, s_andn);
    }
    if (!last_block(&ctl->ticket[TK_DECODE])) return;
    block_scan_tiles(seg, nt, SegOp(), Seg{0, 0, 0}, sh);
    if (threadIdx.x == 0) {
        const unsigned long long db = __ldcg(&ctl->or_base) ^ __ldcg(&ctl->and_base);
        const uint32_t dn = __ldcg(&ctl->or_node) ^ __ldcg(&ctl->and_node);
        uint32_t n = 0;
        if (R > 1) {  // fewer than two runs need no sort
            for (uint32_t d = 0; d < 8; d++)
                if ((db >> (8 * d)) & 0xFFu) ctl->active[n++] = d;
            for (uint32_t d = 0; d < 4; d++)
                if ((dn >> (8 * d)) & 0xFFu) ctl->active[n++] = 8 + d;
        }
        ctl->nactive = n;
    }
}

__global__ void __launch_bounds__(kT)
k_plan_keys(const uint32_t *__restrict__ lane_first, uint32_t L, uint32_t B,
            const uint64_t *__restrict__ run_base, const uint32_t *__restrict__ run_count,
            const uint32_t *__restrict__ numa, const uint32_t *__restrict__ run_lane,
            const Seg *__restrict__ seg, uint32_t *status, PlanCtl *ctl,
            uint32_t *__restrict__ run_block, SortItem *__restrict__ items,
            uint32_t *__restrict__ hist0, uint32_t *__restrict__ hist1, uint32_t npasses,
            uint64_t *counts) {
    __shared__ Seg sh[kT];
    __shared__ uint32_t s_hist[kDigits];
    __shared__ uint32_t s_bits;
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    const uint32_t nact = ctl->nactive;
    const uint32_t dig0 = nact ? ctl->active[0] : 0;
    for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x) s_hist[d] = 0;
    if (threadIdx.x == 0) s_bits = 0;
    __syncthreads();
    const uint64_t r0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
    Seg agg{0, 0, 0};
    uint32_t cnts[kIPT];
    uint32_t heads = 0;
    if (tile < nt) {
        for (int j = 0; j < kIPT; j++) {
            const uint64_t r = r0 + j;
            cnts[j] = 0;
            if (r >= R) continue;
            const uint32_t l = run_lane[r];
            cnts[j] = run_count[r];
            const bool head = r == __ldg(lane_first + l);
            if (head) heads |= 1u << j;
            agg = SegOp()(agg, Seg{cnts[j], head ? 1u : 0u, 0});
        }
    }
    Seg ex, tot;
    block_scan(agg, SegOp(), Seg{0, 0, 0}, sh, &ex, &tot);
    uint32_t bits = 0;
    if (tile < nt) {
        const Seg carry = seg[tile];
        Seg run = SegOp()(carry, ex);  // prefix before this thread's first run
        uint64_t blk = run.sum;
        for (int j = 0; j < kIPT; j++) {
            const uint64_t r = r0 + j;
            if (r >= R) break;
            if (heads >> j & 1u) blk = 0;
            const uint32_t l = run_lane[r];
            run_block[r] = (uint32_t)blk;
            blk += cnts[j];
            if (r + 1 == (uint64_t)__ldg(lane_first + l + 1) && blk != B) bits |= KVX_S_COVERAGE;
            const uint64_t base = run_base[r];
            const uint32_t node = numa[l];
            items[r] = SortItem{base, node, (uint32_t)r};
        }
    }
    if (nact && tile < nt) {
        // histogram of the first active digit, one shared atomic per distinct
        // digit in each warp round
        for (int j = 0; j < kIPT; j++) {
            const uint64_t r = r0 + j;
            const uint32_t d = r < R ? digit_of(run_base[r], numa[run_lane[r]], dig0) : kDigits;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
            if (d < kDigits && (threadIdx.x & 31) == __ffs(peers) - 1)
                atomicAdd(&s_hist[d], __popc(peers));
        }
    }
    if (bits) atomicOr(&s_bits, bits);
    __syncthreads();
    if (tile < nt) {
        if (nact)
            for (uint32_t d = threadIdx.x; d < kDigits; d += blockDim.x)
                hist0[(uint64_t)d * nt + tile] = s_hist[d];
        if (threadIdx.x == 0 && s_bits) {
            atomicOr(status, s_bits);
            atomicOr(&ctl->st, s_bits);
        }
    }
    if (!last_block(&ctl->ticket[TK_KEYS])) return;
    __shared__ uint32_t s_fail;
    if (threadIdx.x == 0) {
        s_fail = 0;
        if (__ldcg(&ctl->st) != 0) s_fail = 1;
        if (nact > npasses) {  // cannot happen once spans are validated
            atomicOr(status, KVX_S_SPAN);
            s_fail = 1;
        }
        if (s_fail) {
            ctl->fail = 1;
            counts[0] = counts[1] = counts[2] = 0;
        }
    }
    __syncthreads();
    if (s_fail || !nact) return;
    block_scan_inplace_span_u32(hist0, (uint64_t)kDigits * nt);
    for (uint64_t i = threadIdx.x; i < (uint64_t)kDigits * nt; i += blockDim.x) hist1[i] = 0;
}

// ---------------------------------------------------- step 2: radix passes

__global__ void __launch_bounds__(kT)
k_plan_sort(const SortItem *__restrict__ in, SortItem *__restrict__ out, PlanCtl *ctl,
            uint32_t *__restrict__ offs, uint32_t *__restrict__ hist_next, uint32_t k) {
    __shared__ uint32_t wcnt[kT / 32][kDigits];
    if (ctl->fail || k >= ctl->nactive) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t nact = ctl->nactive;
    const uint32_t dig = ctl->active[k];
    const bool has_next = k + 1 < nact;
    const uint32_t ndig = has_next ? ctl->active[k + 1] : 0;
    const uint32_t tile = blockIdx.x;
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (uint32_t i = threadIdx.x; i < (kT / 32) * kDigits; i += blockDim.x)
        (&wcnt[0][0])[i] = 0;
    __syncthreads();
    if (tile < nt) {
        SortItem it[kIPT];
        uint32_t d[kIPT], pos[kIPT];
        const uint64_t t0 = (uint64_t)tile * kTile + (uint64_t)w * (32 * kIPT);
        const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
        for (int j = 0; j < kIPT; j++) {
            const uint64_t idx = t0 + (uint64_t)j * 32 + lane;
            if (idx < R) {
                it[j] = in[idx];
                d[j] = digit_of(it[j].base, it[j].node, dig);
            } else {
                d[j] = kDigits;  // out-of-range items match only each other
            }
        }
#pragma unroll
        for (int j = 0; j < kIPT; j++) {
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d[j]);
            const uint32_t rank = __popc(peers & lt_mask);
            const uint32_t before = d[j] < kDigits ? wcnt[w][d[j]] : 0;
            __syncwarp();
            if (d[j] < kDigits && rank == 0) wcnt[w][d[j]] = before + __popc(peers);
            __syncwarp();
            pos[j] = before + rank;
        }
        __syncthreads();
        if (threadIdx.x < kDigits) {
            uint32_t s = 0;
            for (int ww = 0; ww < kT / 32; ww++) {
                const uint32_t c = wcnt[ww][threadIdx.x];
                wcnt[ww][threadIdx.x] = s;
                s += c;
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kIPT; j++) {
            if (d[j] >= kDigits) continue;
            const uint64_t dst = (uint64_t)offs[(uint64_t)d[j] * nt + tile] + wcnt[w][d[j]] + pos[j];
            if (dst >= R) continue;  // never taken: the offsets are a permutation of [0, R)
            out[dst] = it[j];
            if (has_next) {
                const uint32_t nd = digit_of(it[j].base, it[j].node, ndig);
                atomicAdd(&hist_next[(uint64_t)nd * nt + dst / kTile], 1u);
            }
        }
    }
    if (!last_block(&ctl->ticket[TK_SORT0 + k])) return;
    if (!has_next) return;
    block_scan_inplace_span_u32(hist_next, (uint64_t)kDigits * nt);
    for (uint64_t i = threadIdx.x; i < (uint64_t)kDigits * nt; i += blockDim.x) offs[i] = 0;
}

// -------------------------------------------------------- step 3: grouping

__device__ __forceinline__ Rec make_rec(SortItem it, uint64_t R, const int64_t *run_stride,
                                        const uint32_t *run_count, const uint32_t *run_block,
                                        const uint32_t *run_lane, const uint32_t *seg_len) {
    if (it.r >= R) it.r = 0;  // never taken: sorted items are a permutation of the runs
    Rec x;
    x.base = it.base;
    x.node = it.node;
    x.r = it.r;
    x.stride = run_stride[it.r];
    x.count = run_count[it.r];
    x.block = run_block[it.r];
    x.len = seg_len[run_lane[it.r]];
    x.pad = 0;
    return x;
}

__device__ __forceinline__ bool compatible(const Rec &prev, const Rec &x) {
    return x.node == prev.node && x.block == prev.block && x.count == prev.count &&
           x.stride == prev.stride && x.base == prev.base + prev.len;
}

__global__ void __launch_bounds__(kT)
k_plan_adjacent(const int64_t *__restrict__ run_stride,
                const uint32_t *__restrict__ run_count, const uint32_t *__restrict__ run_block,
                const uint32_t *__restrict__ run_lane, const uint32_t *__restrict__ seg_len,
                PlanCtl *ctl, const SortItem *items0, const SortItem *items1, Rec *__restrict__ rec,
                uint8_t *__restrict__ compat, int64_t *segmax) {
    __shared__ int64_t sh[kT];
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const SortItem *sorted = (ctl->nactive & 1) ? items1 : items0;
    const uint32_t tile = blockIdx.x;
    int64_t mx = -1;
    if (tile < nt) {
        const uint64_t p0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
        Rec prev;
        bool have_prev = false;
        if (p0 > 0 && p0 < R) {
            prev = make_rec(sorted[p0 - 1], R, run_stride, run_count, run_block, run_lane, seg_len);
            have_prev = true;
        }
        for (int j = 0; j < kIPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) break;
            const Rec x = make_rec(sorted[p], R, run_stride, run_count, run_block, run_lane, seg_len);
            rec[p] = x;
            const bool c = have_prev && compatible(prev, x);
            compat[p] = c ? 1 : 0;
            if (!c) mx = (int64_t)p;
            prev = x;
            have_prev = true;
        }
    }
    int64_t ex, tot;
    block_scan(mx, MaxOp(), (int64_t)-1, sh, &ex, &tot);
    if (threadIdx.x == 0 && tile < nt) segmax[tile] = tot;
    if (!last_block(&ctl->ticket[TK_ADJ])) return;
    block_scan_tiles(segmax, nt, MaxOp(), (int64_t)-1, sh);
}

__global__ void __launch_bounds__(kT)
k_plan_cut(PlanCtl *ctl, const Rec *__restrict__ rec, const uint8_t *__restrict__ compat,
           const int64_t *__restrict__ segmax, uint8_t *__restrict__ gflag) {
    __shared__ int64_t sh[kT];
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    if (tile >= nt) return;
    const uint64_t p0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
    int64_t mx = -1;
    for (int j = 0; j < kIPT; j++) {
        const uint64_t p = p0 + j;
        if (p < R && !compat[p]) mx = (int64_t)p;
    }
    int64_t ex, tot;
    block_scan(mx, MaxOp(), (int64_t)-1, sh, &ex, &tot);
    int64_t s = segmax[tile] > ex ? segmax[tile] : ex;  // stretch start before this thread
    for (int j = 0; j < kIPT; j++) {
        const uint64_t p = p0 + j;
        if (p >= R) break;
        const bool c = compat[p] != 0;
        if (!c) s = (int64_t)p;
        const Rec x = rec[p];
        if (x.count == 1) {
            gflag[p] = c ? 0 : 1;
            continue;
        }
        if (x.stride <= 0) {
            gflag[p] = 1;  // a non-positive stride never fits: one run per group
            continue;
        }
        const uint64_t stride = (uint64_t)x.stride;
        const uint64_t O = x.base - rec[s > 0 ? s : 0].base;  // offset inside the stretch
        const uint64_t E = O + x.len;
        if (E <= stride) {
            gflag[p] = c ? 0 : 1;
        } else if (O <= stride) {
            // First run that outgrows the stretch's first group: walk the rest
            // of the stretch sequentially (only tables whose block chunks
            // exceed their stride get here).
            gflag[p] = 1;
            uint64_t cur = x.base;
            for (uint64_t q = p + 1; q < R && compat[q]; q++) {
                const Rec y = rec[q];
                if (y.base + y.len - cur > stride) {
                    gflag[q] = 1;
                    cur = y.base;
                } else {
                    gflag[q] = 0;
                }
            }
        }
        // else: written by the walker of this stretch
    }
}

__global__ void __launch_bounds__(kT)
k_plan_count(PlanCtl *ctl, const uint8_t *__restrict__ gflag, GAgg *gagg, uint64_t group_cap,
             uint32_t *status, uint64_t *counts) {
    __shared__ GAgg sh[kT];
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    GAgg a{0, -1};
    if (tile < nt) {
        const uint64_t p0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
        for (int j = 0; j < kIPT; j++) {
            const uint64_t p = p0 + j;
            if (p < R && gflag[p]) {
                a.n++;
                a.last = (int64_t)p;
            }
        }
    }
    GAgg ex, tot;
    block_scan(a, GOp(), GAgg{0, -1}, sh, &ex, &tot);
    if (threadIdx.x == 0 && tile < nt) gagg[tile] = tot;
    if (!last_block(&ctl->ticket[TK_COUNT])) return;
    const GAgg all = block_scan_tiles(gagg, nt, GOp(), GAgg{0, -1}, sh);
    if (threadIdx.x == 0) {
        ctl->ngroups = all.n;
        if (all.n > group_cap) {
            flag_fail(ctl, status, KVX_S_CAPACITY);
            counts[0] = counts[1] = counts[2] = 0;
        }
    }
}

__device__ __forceinline__ bool group_dense(uint32_t count, int64_t stride, uint64_t chunk) {
    return count == 1 || (stride > 0 && chunk == (uint64_t)stride);
}

__device__ __forceinline__ uint64_t group_pieces(const kvx_group &g) {
    if (g.dense) return ceil_div((uint64_t)g.count * g.chunk, KVX_MAX_READ_BYTES);
    return (uint64_t)g.count * ceil_div(g.chunk, KVX_MAX_READ_BYTES);
}

__global__ void __launch_bounds__(kT)
k_plan_groups(PlanCtl *ctl, const Rec *__restrict__ rec, const uint8_t *__restrict__ gflag,
              const GAgg *__restrict__ gagg, kvx_group *__restrict__ groups,
              uint32_t *__restrict__ run_group, uint64_t *__restrict__ run_off, CAgg *cagg,
              uint64_t desc_cap, uint32_t *status, uint64_t *counts) {
    __shared__ GAgg shg[kT];
    __shared__ CAgg shc[kT];
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    const uint64_t p0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
    GAgg a{0, -1};
    if (tile < nt)
        for (int j = 0; j < kIPT; j++) {
            const uint64_t p = p0 + j;
            if (p < R && gflag[p]) {
                a.n++;
                a.last = (int64_t)p;
            }
        }
    GAgg ex, tot;
    block_scan(a, GOp(), GAgg{0, -1}, shg, &ex, &tot);
    CAgg c{0, 0};
    if (tile < nt) {
        GAgg run = GOp()(gagg[tile], ex);
        for (int j = 0; j < kIPT; j++) {
            const uint64_t p = p0 + j;
            if (p >= R) break;
            if (gflag[p]) {
                run.n++;
                run.last = (int64_t)p;
            }
            const uint64_t gid = run.n - 1;
            const Rec x = rec[p];
            const Rec g0 = rec[run.last >= 0 ? run.last : 0];  // position 0 always starts a group
            const uint64_t off = x.base - g0.base;
            run_group[x.r] = (uint32_t)gid;
            run_off[x.r] = off;
            const bool end = p + 1 == R || gflag[p + 1];
            if (end) {
                kvx_group g;
                g.base = g0.base;
                g.stride = g0.stride;
                g.chunk = off + x.len;
                g.local = 0;
                g.block = g0.block;
                g.count = g0.count;
                g.node = g0.node;
                g.dense = group_dense(g0.count, g0.stride, g.chunk) ? 1u : 0u;
                groups[gid] = g;
                c.bytes += (uint64_t)g.count * g.chunk;
                c.descs += group_pieces(g);
            }
        }
    }
    CAgg cex, ctot;
    block_scan(c, COp(), CAgg{0, 0}, shc, &cex, &ctot);
    if (threadIdx.x == 0 && tile < nt) cagg[tile] = ctot;
    if (!last_block(&ctl->ticket[TK_GROUPS])) return;
    const CAgg all = block_scan_tiles(cagg, nt, COp(), CAgg{0, 0}, shc);
    if (threadIdx.x == 0) {
        if (all.descs > desc_cap) {
            flag_fail(ctl, status, KVX_S_CAPACITY);
            counts[0] = counts[1] = counts[2] = 0;
        } else {
            counts[0] = ctl->ngroups;
            counts[1] = all.descs;
            counts[2] = all.bytes;
        }
    }
}

// --------------------------------------------------- step 4: carve + reads

__global__ void __launch_bounds__(kT)
k_plan_emit(PlanCtl *ctl, const Rec *__restrict__ rec, const uint8_t *__restrict__ gflag,
            const uint32_t *__restrict__ run_group, const CAgg *__restrict__ cagg,
            kvx_group *__restrict__ groups, kvx_desc *__restrict__ descs) {
    __shared__ CAgg shc[kT];
    if (ctl->fail) return;
    const uint64_t R = ctl->R;
    const uint32_t nt = ctl->nt;
    const uint32_t tile = blockIdx.x;
    if (tile >= nt) return;
    const uint64_t p0 = (uint64_t)tile * kTile + (uint64_t)threadIdx.x * kIPT;
    CAgg c{0, 0};
    uint32_t ends = 0;
    for (int j = 0; j < kIPT; j++) {
        const uint64_t p = p0 + j;
        if (p >= R) break;
        if (p + 1 == R || gflag[p + 1]) {
            ends |= 1u << j;
            const kvx_group g = groups[run_group[rec[p].r]];
            c.bytes += (uint64_t)g.count * g.chunk;
            c.descs += group_pieces(g);
        }
    }
    CAgg ex, tot;
    block_scan(c, COp(), CAgg{0, 0}, shc, &ex, &tot);
    CAgg cur = COp()(cagg[tile], ex);
    for (int j = 0; j < kIPT; j++) {
        if (!(ends >> j & 1u)) continue;
        const uint64_t p = p0 + j;
        const uint32_t gid = run_group[rec[p].r];
        kvx_group g = groups[gid];
        g.local = cur.bytes;
        groups[gid].local = cur.bytes;
        const uint64_t M = KVX_MAX_READ_BYTES;
        uint64_t d = cur.descs;
        if (g.dense) {
            const uint64_t total = (uint64_t)g.count * g.chunk;
            for (uint64_t o = 0; o < total; o += M, d++)
                descs[d] = kvx_desc{g.base + o, g.local + o, total - o < M ? total - o : M, gid, 0};
        } else {
            for (uint64_t i = 0; i < g.count; i++) {
                const uint64_t rb = g.base + i * (uint64_t)g.stride;
                const uint64_t lb = g.local + i * g.chunk;
                for (uint64_t o = 0; o < g.chunk; o += M, d++)
                    descs[d] = kvx_desc{rb + o, lb + o, g.chunk - o < M ? g.chunk - o : M, gid, 0};
            }
        }
        cur.bytes += (uint64_t)g.count * g.chunk;
        cur.descs += group_pieces(g);
    }
}

uint32_t base_digits(uint64_t pool_bytes) {
    uint32_t bits = 0;
    while (bits < 64 && (pool_bytes >> bits)) bits++;
    return (bits + 7) / 8;
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" uint64_t kvx_desc_capacity(uint32_t B, uint32_t L, uint64_t seg_bytes_sum) {
    const unsigned __int128 slab = (unsigned __int128)B * seg_bytes_sum;
    return (uint64_t)B * L + (uint64_t)((slab + KVX_MAX_READ_BYTES - 1) / KVX_MAX_READ_BYTES);
}

extern "C" size_t kvx_plan_workspace_size(uint32_t L, uint64_t run_capacity, uint64_t pool_bytes) {
    (void)pool_bytes;
    size_t bytes = 0;
    carve(nullptr, L, run_capacity, &bytes);
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
    if (run_capacity >= (1ull << 32) || table_lanes == 0xFFFFFFFFu) return KVX_EINVAL;
    if ((group_capacity && !groups) || (desc_capacity && !descs)) return KVX_EINVAL;
    size_t need = 0;
    Ws w = carve(ws, table_lanes, run_capacity, &need);
    if (ws_bytes < need) return KVX_EINVAL;
    cudaStream_t s = as_stream(stream);
    const uint32_t grid = (uint32_t)ceil_div(run_capacity ? run_capacity : 1, kTile);
    const uint32_t npasses = base_digits(pool_bytes) + 4;
    const uint32_t L = table_lanes;

    k_plan_init<<<1, 1024, 0, s>>>(runs_per_lane, table_lanes, num_runs, run_capacity, B, seg_len,
                                   template_lanes, lane_first, counts, status, w.ctl);
    KVX_LAUNCHED();
    k_plan_decode<<<grid, kT, 0, s>>>(lane_first, L, run_base, run_stride, run_count, seg_len,
                                      numa, pool_bytes, status, w.ctl, w.run_lane, w.seg);
    KVX_LAUNCHED();
    k_plan_keys<<<grid, kT, 0, s>>>(lane_first, L, B, run_base, run_count, numa, w.run_lane, w.seg,
                                    status, w.ctl, run_block, w.items[0], w.hist[0], w.hist[1],
                                    npasses, counts);
    KVX_LAUNCHED();
    for (uint32_t k = 0; k < npasses; k++) {
        k_plan_sort<<<grid, kT, 0, s>>>(w.items[k & 1], w.items[(k + 1) & 1], w.ctl,
                                        w.hist[k & 1], w.hist[(k + 1) & 1], k);
        KVX_LAUNCHED();
    }
    k_plan_adjacent<<<grid, kT, 0, s>>>(run_stride, run_count, run_block, w.run_lane,
                                        seg_len, w.ctl, w.items[0], w.items[1], w.rec, w.compat,
                                        w.segmax);
    KVX_LAUNCHED();
    k_plan_cut<<<grid, kT, 0, s>>>(w.ctl, w.rec, w.compat, w.segmax, w.gflag);
    KVX_LAUNCHED();
    k_plan_count<<<grid, kT, 0, s>>>(w.ctl, w.gflag, w.gagg, group_capacity, status, counts);
    KVX_LAUNCHED();
    k_plan_groups<<<grid, kT, 0, s>>>(w.ctl, w.rec, w.gflag, w.gagg, groups, run_group, run_off,
                                      w.cagg, desc_capacity, status, counts);
    KVX_LAUNCHED();
    k_plan_emit<<<grid, kT, 0, s>>>(w.ctl, w.rec, w.gflag, run_group, w.cagg, groups, descs);
    KVX_LAUNCHED();
    return KVX_OK;
}
