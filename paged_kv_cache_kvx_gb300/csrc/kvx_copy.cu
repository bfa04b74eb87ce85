// Pack and unpack: the data movement of the planned reads (pegaflow PR #350,
// Requester step 4: one coalesced read per dense group, per-block reads for a
// non-dense group; READ splitting: 32 MiB descriptors).  Pack gathers
// holder-pool bytes into the dense slab; unpack is the inverse scatter.
//
// HBM-bound copy, no contraction.  The slab side is always contiguous (the
// descriptors tile it), so the work is cut into fixed 64 KiB slab tiles.  A
// prep kernel checks the descriptors and sorts every tile into one of three
// lists:
//   - TMA jobs: tiles inside one 16-byte aligned descriptor (every tile of a
//     dense 32 MiB read, most tiles of a 1 MiB per-block read).  One lane per
//     SM streams them through a 3-stage shared-memory ring with bulk copies
//     (cp.async.bulk global->shared, completion on an mbarrier, then
//     cp.async.bulk shared->global): the SM's bulk-copy unit moves the
//     bytes, no register staging, up to 192 KiB of loads in flight per SM.
//     Rings claim their jobs dynamically, so the copy ends when the bytes
//     are done rather than when the slowest ring is.  Sweeps on GB300 (16-96
//     KiB tiles, 2-12 stages, 38-304 rings, static or claimed work, claims of
//     1-8 jobs) put one ring per SM, 3 x 64 KiB, claims of 2 first; one SM
//     is left free for kernels that run beside the copy.
//   - pieces: tiles shared by several 16-byte aligned descriptors of 2 to
//     16 KiB (the 4 KiB per-segment reads of a scattered holder), one piece
//     per descriptor, moved by the four 16 KiB-stage bulk-copy rings per SM
//     of kvx_ring.cuh.
//   - vector tiles: the other shared tiles (512 B segment reads, 32 KiB
//     block reads) and unaligned ones.  256 threads per tile; the tile's
//     descriptors are staged in shared memory, a table gives each 64-byte
//     bucket its first descriptor, and each 16-byte vector steps forward
//     from there (byte copies when anything is unaligned).
// The vector kernel walks its list round-robin over a persistent grid, so
// the grid streams one window of the slab at a time.  The copies run in one
// call (kvx_pack / kvx_unpack) or in two: the checks and lists first
// (kvx_copy_prepare), the bytes later (kvx_pack_prepared / _unpack_prepared).

#include "kvx_ring.cuh"

namespace kvx {
namespace {

constexpr int kThreads = 256;
constexpr uint64_t kTileBytes = 64 * 1024;
constexpr int kVecPerThread = (int)(kTileBytes / (kThreads * 16));  // 16
constexpr int kBucketShift = 6;                                       // 64-byte buckets of a vector tile
constexpr int kBuckets = (int)(kTileBytes >> kBucketShift);          // 1024
constexpr int kCtasPerSm = 3;
constexpr int kStages = 3;                  // TMA ring depth per CTA
constexpr int kTmaCtasPerSm = 1;

struct CopyCtl {
    unsigned long long used;  // end of the last descriptor (slab bytes in use)
    uint32_t bad;             // descriptors do not tile the slab
    uint32_t n_tma;           // TMA jobs
    uint32_t n_vec;           // vector tiles
    uint32_t next_job;        // next unclaimed TMA job
    uint32_t n_piece;         // descriptor pieces of shared tiles for the ring path
    ring::SegCtl seg;         // claim counter of the ring path
    uint32_t users;           // bulk-kernel blocks that have started on these lists
    unsigned long long key;   // the copy the lists were made for (see copy_key)
};

// A tile shared by several descriptors goes to the ring path of kvx_ring.cuh
// (four warps per SM, 3 x 16 KiB stages each), one piece per descriptor, when
// every descriptor there is aligned and at least this long (below it the
// register path is the faster one) ...
constexpr uint64_t kPieceMinDesc = 2048;
constexpr uint32_t kPiecesPerTile = (uint32_t)(kTileBytes / kPieceMinDesc) + 1;  // 33
// ... and when one of them is shorter than this: tiles of longer descriptors
// run faster on the register path (measured on GB300: 32 KiB descriptors
// 6572 GB/s there, 6307 through the rings; 4 KiB descriptors ~6000 there,
// 6427 through the rings).  A whole tile of one descriptor always takes the
// 64 KiB-stage ring of k_copy_tma (a ring of 16 KiB stages reached only ~6090
// on the default workload, against ~6870).
constexpr uint64_t kPieceMaxDesc = 16 * 1024;

struct TmaJob {
    uint64_t lo;      // slab offset of the tile
    uint64_t delta;   // pool offset - slab offset inside the tile's descriptor
    uint32_t len;     // bytes (multiple of 16)
    uint32_t pad;
};

struct Ws {
    CopyCtl *ctl;
    uint32_t *tile_desc;  // [ntiles]
    TmaJob *jobs;         // [ntiles]
    uint32_t *vec_tiles;  // [ntiles]
    TmaJob *pieces;       // [kPiecesPerTile * ntiles], when the workspace holds them
};

// The workspace: the tile lists, then (optional) the piece list.  base_bytes
// gets the size without the piece list.
Ws carve(void *base, uint64_t slab_bytes, size_t *bytes, size_t *base_bytes = nullptr) {
    const uint64_t nt = ceil_div(slab_bytes, kTileBytes);
    Carver c(base);
    Ws w;
    w.ctl = c.take<CopyCtl>(1);
    w.tile_desc = c.take<uint32_t>(nt);
    w.jobs = c.take<TmaJob>(nt);
    w.vec_tiles = c.take<uint32_t>(nt);
    if (base_bytes) *base_bytes = c.off;
    w.pieces = c.take<TmaJob>((size_t)kPiecesPerTile * nt);
    *bytes = c.off;
    return w;
}

__device__ __forceinline__ bool in_range(uint64_t off, uint64_t len, uint64_t size) {
    return off <= size && len <= size - off;
}

// The fields of a descriptor the tile lists need: two loads when the array
// starts on a 16-byte boundary (remote and local together), else three.
struct DescView {
    uint64_t remote, local, len;
};
__device__ __forceinline__ DescView load_desc(const kvx_desc *d, bool d16) {
    if (d16) {
        const ulonglong2 rl = __ldg(reinterpret_cast<const ulonglong2 *>(d));  // remote, local
        return DescView{rl.x, rl.y, __ldg(&d->len)};
    }
    return DescView{__ldg(&d->remote), __ldg(&d->local), __ldg(&d->len)};
}

// The descriptors from a on that start below hi, at most kWalkMax of them,
// in batches whose loads are issued together: f(e) for each; f returns false
// to stop.  Returns false when the walk hit kWalkMax with descriptors left
// (more than kPiecesPerTile pieces: some descriptor there is too short for
// the ring path anyway).
constexpr int kWalkBatch = 4;
constexpr uint64_t kWalkMax = kPiecesPerTile + 1;

template <class F>
__device__ __forceinline__ bool walk_tile_descs(const kvx_desc *__restrict__ descs, bool d16, uint64_t n,
                                                uint64_t a, uint64_t hi, F &&f) {
    const uint64_t end = n - a < kWalkMax ? n : a + kWalkMax;
    for (uint64_t k0 = a; k0 < end; k0 += kWalkBatch) {
        DescView e[kWalkBatch];
#pragma unroll
        for (int j = 0; j < kWalkBatch; j++)
            if (k0 + j < end) e[j] = load_desc(descs + k0 + j, d16);
#pragma unroll
        for (int j = 0; j < kWalkBatch; j++) {
            if (k0 + j >= end || e[j].local >= hi) return true;
            if (!f(e[j])) return true;
        }
    }
    return end == n;
}

// Descriptor checks (one thread per descriptor: tiling, bounds), then one
// thread per tile: the descriptor holding the tile's first byte (binary
// search) and the tile's list.
__global__ void __launch_bounds__(kThreads)
k_copy_prep(const kvx_desc *__restrict__ descs, const uint64_t *__restrict__ num_descs,
            uint64_t desc_cap, uint64_t pool_bytes, uint64_t slab_bytes, bool bases_aligned,
            uint32_t *__restrict__ tile_desc, TmaJob *__restrict__ jobs,
            uint32_t *__restrict__ vec_tiles, TmaJob *__restrict__ pieces, CopyCtl *ctl,
            uint32_t *status, unsigned long long key) {
    if (blockIdx.x == 0 && threadIdx.x == 0) ctl->key = key;
    const bool d16 = (reinterpret_cast<uintptr_t>(descs) & 15) == 0;  // descriptors need only 8-byte alignment
    const uint64_t n = *num_descs < desc_cap ? *num_descs : desc_cap;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t bits = 0;
    for (uint64_t k = tid; k < n; k += stride) {
        const kvx_desc d = descs[k];
        uint64_t expect = 0;
        bool tiled = true;
        if (k > 0) {
            const kvx_desc p = descs[k - 1];
            expect = p.local + p.len;
            tiled = expect >= p.local;  // no wrap
        }
        tiled = tiled && d.local == expect && d.len > 0 && d.local + d.len > d.local;
        if (!tiled) {
            bits |= KVX_S_DESC;
            ctl->bad = 1;
            continue;
        }
        if (!in_range(d.remote, d.len, pool_bytes) || !in_range(d.local, d.len, slab_bytes))
            bits |= KVX_S_BOUNDS;
        if (k + 1 == n) ctl->used = d.local + d.len;
    }
    if (bits) atomicOr(status, bits);
    if (n == 0) return;
    // The lists are only read when the descriptors tile the slab (else the
    // copy kernels do nothing), so the last descriptor's end is the bytes in use.
    const kvx_desc last = descs[n - 1];
    const uint64_t used = last.local + last.len < slab_bytes ? last.local + last.len : slab_bytes;
    const uint64_t ntiles = ceil_div(used, kTileBytes);
    // Every block takes a contiguous share of the tiles, so the walks over
    // shared tiles (one cache line per descriptor and lane) spread over all SMs.
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t per = ceil_div(ntiles, (uint64_t)gridDim.x);
    const uint64_t tb = (uint64_t)blockIdx.x * per;
    const uint64_t te = tb + per < ntiles ? tb + per : ntiles;
    for (uint64_t t0 = tb + (threadIdx.x - lane); t0 < te; t0 += blockDim.x) {  // warp-uniform loop
        const uint64_t t = t0 + lane;
        bool is_tma = false, is_vec = false;
        uint32_t npieces = 0;  // this tile's pieces for the ring path (0: not on it)
        uint64_t lo = 0, hi = 0, a = 0;
        TmaJob job{};
        if (t < te) {
            lo = t * kTileBytes;
            hi = lo + kTileBytes < used ? lo + kTileBytes : used;
            uint64_t z = n;  // last k with descs[k].local <= lo, in [a, z)
            while (z - a > 1) {
                const uint64_t m = (a + z) >> 1;
                if (descs[m].local <= lo) a = m; else z = m;
            }
            tile_desc[t] = (uint32_t)a;
            const kvx_desc d = descs[a];
            const bool single = d.local <= lo && hi - d.local <= d.len;
            const bool inb = in_range(d.remote, d.len, pool_bytes) && in_range(d.local, d.len, slab_bytes);
            const uint64_t delta = d.remote - d.local;
            if (single && !inb) {
                // skipped: its descriptor leaves the pool or the slab
            } else if (single && bases_aligned && ((lo | hi | delta) & 15) == 0) {
                is_tma = true;
                job = TmaJob{lo, delta, (uint32_t)(hi - lo), 0};
            } else {
                is_vec = true;
                if (pieces && bases_aligned) {
                    // a shared tile: one piece per descriptor, if each is aligned
                    // and long enough for the bulk engine
                    bool fit = true, short_desc = false;
                    uint32_t np = 0;
                    const bool whole = walk_tile_descs(descs, d16, n, a, hi, [&](const DescView &e) {
                        const uint64_t plo = e.local > lo ? e.local : lo;
                        const uint64_t phi = e.len < hi - e.local ? e.local + e.len : hi;
                        if (plo >= phi) return true;
                        if (e.len < kPieceMinDesc || ((plo | phi | (e.remote - e.local)) & 15)) {
                            fit = false;
                            return false;
                        }
                        short_desc |= e.len < kPieceMaxDesc;
                        if (in_range(e.remote, e.len, pool_bytes) && in_range(e.local, e.len, slab_bytes))
                            np++;  // a descriptor outside the pool or slab is skipped
                        return true;
                    });
                    if (whole && fit && short_desc && np <= kPiecesPerTile) {
                        is_vec = false;
                        npieces = np;
                    }
                }
            }
        }
        const uint32_t mt = __ballot_sync(0xFFFFFFFFu, is_tma);
        const uint32_t mv = __ballot_sync(0xFFFFFFFFu, is_vec);
        uint32_t bt = 0, bv = 0;
        if (lane == 0) {
            if (mt) bt = atomicAdd(&ctl->n_tma, __popc(mt));
            if (mv) bv = atomicAdd(&ctl->n_vec, __popc(mv));
        }
        bt = __shfl_sync(0xFFFFFFFFu, bt, 0);
        bv = __shfl_sync(0xFFFFFFFFu, bv, 0);
        const uint32_t below = (1u << lane) - 1u;
        if (is_tma) jobs[bt + __popc(mt & below)] = job;
        if (is_vec) vec_tiles[bv + __popc(mv & below)] = (uint32_t)t;
        if (pieces) {  // reserve this warp's pieces, then write them
            const uint32_t incl = warp_incl_sum(npieces);
            const uint32_t wtot = __shfl_sync(0xFFFFFFFFu, incl, 31);
            uint32_t bp = 0;
            if (lane == 0 && wtot) bp = atomicAdd(&ctl->n_piece, wtot);
            bp = __shfl_sync(0xFFFFFFFFu, bp, 0) + incl - npieces;
            if (npieces) {
                const uint64_t cap = (uint64_t)kPiecesPerTile * ntiles;
                walk_tile_descs(descs, d16, n, a, hi, [&](const DescView &e) {
                    const uint64_t plo = e.local > lo ? e.local : lo;
                    const uint64_t phi = e.len < hi - e.local ? e.local + e.len : hi;
                    if (plo >= phi) return true;
                    if (!(in_range(e.remote, e.len, pool_bytes) && in_range(e.local, e.len, slab_bytes)))
                        return true;
                    if (bp < cap)  // always: at most kPiecesPerTile per tile
                        pieces[bp] = TmaJob{plo, e.remote - e.local, (uint32_t)(phi - plo), 0};
                    bp++;
                    return true;
                });
            }
        }
    }
}

// ------------------------------------------------------------- TMA path

// Warp 0 of each bulk-copy CTA; lane 0 drives the ring.  Jobs are handed
// out dynamically: a ring claims kGrab consecutive jobs at a time from an
// atomic counter (the warp loads their records, one per lane) and claims its
// next batch while it works through the current one, so a ring that happens
// to sit on a busier part of the chip simply takes fewer tiles and the copy
// ends when the bytes are done, not when the slowest ring is.
constexpr uint32_t kGrab = 2;

struct Grab {
    uint32_t pos, n;  // warp-uniform
    TmaJob rec;       // lane j holds job j of the batch
};

template <bool PACK>
__device__ void tile_ring(const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r, uint8_t *slab_w,
                          const TmaJob *__restrict__ jobs, CopyCtl *ctl, uint32_t *status, uint8_t *ring,
                          uint64_t *bars) {
    const uint32_t lane = threadIdx.x & 31;
    if (ctl->bad) return;
    const uint32_t n = ctl->n_tma;
    if (n == 0) return;
    if (lane == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&bars[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    auto claim = [&](Grab &g) {
        uint32_t b = 0;
        if (lane == 0) b = atomicAdd(&ctl->next_job, kGrab);
        b = __shfl_sync(0xFFFFFFFFu, b, 0);
        g.pos = 0;
        g.n = b < n ? (n - b < kGrab ? n - b : kGrab) : 0;
        if (lane < g.n) g.rec = jobs[b + lane];
    };
    Grab cur, nxt;
    claim(cur);
    claim(nxt);
    uint8_t *dst_ring[kStages];
    uint32_t len_ring[kStages];
    bool ok = true;
    uint32_t issued = 0, stored = 0;  // loads issued, tiles stored (uniform)
    for (;;) {
        if (cur.pos == cur.n && cur.n != 0) {
            cur = nxt;
            claim(nxt);
        }
        const bool have = cur.pos < cur.n;
        if (stored < issued && (issued - stored == (uint32_t)kStages || !have)) {
            if (lane == 0) {
                const int s = stored % kStages;
                if (!mbar_wait(&bars[s], (stored / kStages) & 1u)) {
                    ok = false;
                } else {
                    bulk_s2g(dst_ring[s], ring + (uint64_t)s * kTileBytes, len_ring[s]);
                    bulk_commit();
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            stored++;
            continue;
        }
        if (!have) break;  // every job claimed and stored
        const uint64_t lo = __shfl_sync(0xFFFFFFFFu, cur.rec.lo, cur.pos);
        const uint64_t delta = __shfl_sync(0xFFFFFFFFu, cur.rec.delta, cur.pos);
        const uint32_t len = __shfl_sync(0xFFFFFFFFu, cur.rec.len, cur.pos);
        cur.pos++;
        if (lane == 0) {
            const int s = issued % kStages;
            if (issued >= (uint32_t)kStages) bulk_wait_read_all();  // store issued-kStages read its buffer
            const uint8_t *src = PACK ? pool_r + lo + delta : slab_r + lo;
            dst_ring[s] = PACK ? slab_w + lo : pool_w + lo + delta;
            len_ring[s] = len;
            mbar_arrive_expect_tx(&bars[s], len);
            bulk_g2s(ring + (uint64_t)s * kTileBytes, src, len, &bars[s]);
        }
        issued++;
    }
    if (lane == 0) {
        if (!ok) {
            atomicOr(status, KVX_S_TIMEOUT);
            // let the loads still in flight (at most kStages) land before the
            // ring is released; each barrier has one use outstanding
            for (uint32_t k = stored; k < issued; k++) mbar_wait(&bars[k % kStages], (k / kStages) & 1u);
        }
        bulk_wait_all();
    }
    __syncwarp();
}

// The ring path's segments: the pieces of shared tiles listed by the prep.
template <bool PACK>
struct PieceGen {
    const uint8_t *pool_r;
    uint8_t *pool_w;
    const uint8_t *slab_r;
    uint8_t *slab_w;
    const TmaJob *pieces;
    const CopyCtl *ctl;
    uint32_t *st;
    __device__ uint64_t units() const { return ctl->bad ? 0 : ctl->n_piece; }
    __device__ ring::Seg get(uint64_t u, uint32_t &) const {
        const TmaJob j = pieces[u];
        return PACK ? ring::Seg{pool_r + j.lo + j.delta, slab_w + j.lo, j.len, true}
                    : ring::Seg{slab_r + j.lo, pool_w + j.lo + j.delta, j.len, true};
    }
    __device__ uint32_t *status() const { return st; }
};

// The bulk-copy kernel, one CTA per SM but one: warp 0 streams the whole-tile jobs
// through a ring of 3 x 64 KiB stages; then the same shared memory becomes
// four rings of 3 x 16 KiB, one per remaining warp, for the pieces of shared
// tiles.  One launch for both lists: an SM that runs out of tiles moves on
// to pieces, and a copy without pieces pays nothing for them.
constexpr int kBulkWarps = 1 + ring::kRingWarps;
static_assert(kStages * kTileBytes == ring::kRingWarps * ring::kRing * ring::kStageBytes,
              "the piece rings reuse the tile ring's shared memory");

template <bool PACK>
__global__ void __launch_bounds__(32 * kBulkWarps, kTmaCtasPerSm)
k_copy_tma(const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r, uint8_t *slab_w,
           const TmaJob *__restrict__ jobs, const TmaJob *pieces, CopyCtl *ctl, uint32_t *status,
           unsigned long long key) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ ring::RingSmem rs[ring::kRingWarps];
    __shared__ bool s_go;
    // The lists must have been made for this copy, and serve one copy: a
    // second launch on them finds the tile claims spent, so it stops here.
    if (threadIdx.x == 0) {
        const bool mine = ctl->key == key;
        const bool first = atomicAdd(&ctl->users, 1u) < gridDim.x;
        s_go = mine && first;
        if (!s_go && blockIdx.x == 0) atomicOr(status, KVX_S_DESC);
    }
    __syncthreads();
    // The register-path kernel launched after this one may start as soon as
    // every block has claimed its place here (users counted) when it has at
    // most a tile per bulk block to move; with more, beside the bulk copy it
    // measured slower, so it starts as the bulk blocks exit (still without
    // the gap between two ordinary launches).
    if (__ldcg(&ctl->n_vec) <= gridDim.x) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!s_go) return;
    const uint32_t wid = threadIdx.x >> 5;
    if (wid == 0) tile_ring<PACK>(pool_r, pool_w, slab_r, slab_w, jobs, ctl, status, ring, bars);
    __syncthreads();  // the tile ring's copies are complete: its stages are free
    if (!pieces || wid == 0) return;
    const PieceGen<PACK> g{pool_r, pool_w, slab_r, slab_w, pieces, ctl, status};
    ring::ring_warp(g, &ctl->seg, ring + (uint64_t)(wid - 1) * ring::kRing * ring::kStageBytes, rs[wid - 1],
                    threadIdx.x & 31);
}

// ---------------------------------------------------------- vector path

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(uint8_t *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

template <bool PACK>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_copy_vec(const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r, uint8_t *slab_w,
           uint64_t pool_bytes, uint64_t slab_bytes, bool bases_aligned,
           const kvx_desc *__restrict__ descs, const uint64_t *__restrict__ num_descs,
           uint64_t desc_cap, const uint32_t *__restrict__ tile_desc,
           const uint32_t *__restrict__ vec_tiles, const CopyCtl *ctl, unsigned long long key,
           uint32_t bulk_blocks) {
    __shared__ uint64_t s_lo[kThreads + 1];
    __shared__ uint64_t s_delta[kThreads];
    __shared__ uint8_t s_ok[kThreads];
    __shared__ uint16_t s_first[kBuckets];  // per 64-byte bucket: the last span starting at or before it
    if (ctl->bad || ctl->key != key || __ldcg(&ctl->users) != bulk_blocks) return;
    const uint64_t n = *num_descs < desc_cap ? *num_descs : desc_cap;
    const uint64_t used = ctl->used < slab_bytes ? ctl->used : slab_bytes;
    const uint32_t nlist = ctl->n_vec;
    for (uint32_t li = blockIdx.x; li < nlist; li += gridDim.x) {
        const uint64_t t = vec_tiles[li];
        uint64_t lo = t * kTileBytes;
        if (lo >= used) continue;
        const uint64_t hi = lo + kTileBytes < used ? lo + kTileBytes : used;
        uint64_t k = tile_desc[t];
        if (k >= n) continue;
        // stage up to kThreads descriptors at a time
        while (lo < hi) {
            const uint64_t kk = k + threadIdx.x;
            bool in = false, ok = false, aligned = true;
            uint64_t slo = 0, delta = 0, shi = 0;
            if (kk < n) {
                const kvx_desc d = descs[kk];
                if (d.local < hi) {
                    slo = d.local > lo ? d.local : lo;
                    shi = d.len < hi - d.local ? d.local + d.len : hi;
                    in = slo < shi;
                    ok = in_range(d.remote, d.len, pool_bytes) && in_range(d.local, d.len, slab_bytes);
                    delta = d.remote - d.local;
                    aligned = ((slo | shi | delta) & 15) == 0;
                }
            }
            const int nb = __syncthreads_count(in);
            const bool all_aligned = __syncthreads_and(aligned || !in) && bases_aligned;
            if (in) {
                s_lo[threadIdx.x] = slo;
                s_delta[threadIdx.x] = delta;
                s_ok[threadIdx.x] = ok;
            }
            if (in && threadIdx.x == nb - 1) s_lo[nb] = shi;
            __syncthreads();
            if (nb == 0) break;
            const uint64_t bhi = s_lo[nb];
            if (all_aligned) {
                // One search per bucket instead of one per vector: a vector
                // starts from its bucket's span and steps forward (aligned
                // spans are at least 16 bytes, so at most three steps).
                for (uint32_t b = threadIdx.x; b < (uint32_t)kBuckets; b += kThreads) {
                    const uint64_t xs = lo + ((uint64_t)b << kBucketShift);
                    int a = 0, z = nb;  // last span with s_lo <= xs
                    while (z - a > 1) {
                        const int m = (a + z) >> 1;
                        if (s_lo[m] <= xs) a = m; else z = m;
                    }
                    s_first[b] = (uint16_t)a;
                }
                __syncthreads();
                constexpr int U = kVecPerThread / 2;
                for (uint64_t x = lo + (uint64_t)threadIdx.x * 16; x < bhi;
                     x += (uint64_t)kThreads * 16 * U) {
                    uint4 v[U];
                    uint64_t dst[U];
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        const uint64_t xx = x + (uint64_t)u * kThreads * 16;
                        dst[u] = ~0ull;
                        if (xx >= bhi) continue;
                        int a = s_first[(xx - lo) >> kBucketShift];  // last span with s_lo <= xx
                        while (a + 1 < nb && s_lo[a + 1] <= xx) a++;
                        if (xx < bhi && s_ok[a]) {
                            const uint64_t px = xx + s_delta[a];
                            v[u] = PACK ? ld_stream(pool_r + px) : ld_stream(slab_r + xx);
                            dst[u] = PACK ? xx : px;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        if (dst[u] != ~0ull) {
                            if (PACK) st_stream(slab_w + dst[u], v[u]);
                            else st_stream(pool_w + dst[u], v[u]);
                        }
                    }
                }
            } else {
                for (uint64_t x = lo + threadIdx.x; x < bhi; x += kThreads) {
                    int a = 0, z = nb;
                    while (z - a > 1) {
                        const int m = (a + z) >> 1;
                        if (s_lo[m] <= x) a = m; else z = m;
                    }
                    if (!s_ok[a]) continue;
                    if (PACK) slab_w[x] = pool_r[x + s_delta[a]];
                    else pool_w[x + s_delta[a]] = slab_r[x];
                }
            }
            __syncthreads();
            lo = bhi;
            k += nb;
        }
    }
}

template <bool PACK>
cudaError_t set_tma_smem() {
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_copy_tma<PACK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kStages * kTileBytes));
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

// Identifies the copy a workspace's lists were made for: the descriptor
// arrays, the sizes, whether the bases are 16-byte aligned, whether the piece
// list is in use, and the workspace itself.  The pool and slab addresses enter
// only through their alignment (the lists hold offsets), so one preparation
// serves a pack or an unpack alike; it serves one copy.
unsigned long long copy_key(const kvx_desc *descs, const uint64_t *num_descs, uint64_t desc_cap,
                            uint64_t pool_bytes, uint64_t slab_bytes, bool aligned, bool pieces,
                            const void *ws) {
    const uint64_t parts[] = {reinterpret_cast<uintptr_t>(descs), reinterpret_cast<uintptr_t>(num_descs),
                              desc_cap, pool_bytes, slab_bytes, (aligned ? 1u : 0u) | (pieces ? 2u : 0u),
                              reinterpret_cast<uintptr_t>(ws)};
    uint64_t h = 0x243F6A8885A308D3ull;
    for (uint64_t x : parts) {  // splitmix64 finaliser over the running state
        h ^= x + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= h >> 30;
        h *= 0xBF58476D1CE4E5B9ull;
        h ^= h >> 27;
        h *= 0x94D049BB133111EBull;
        h ^= h >> 31;
    }
    return h | 1;  // a cleared workspace (key 0) matches no copy
}

// The host-side checks and the workspace layout shared by every copy call.
struct CopySetup {
    Ws w;
    bool aligned;
    unsigned long long key;
};

kvx_status setup(const void *pool, uint64_t pool_bytes, const void *slab, uint64_t slab_bytes,
                 const kvx_desc *descs, const uint64_t *num_descs, uint64_t desc_cap, uint32_t *status,
                 void *ws, size_t ws_bytes, CopySetup *cs) {
    if (!descs || !num_descs || !status || !ws) return KVX_EINVAL;
    if ((pool_bytes && !pool) || (slab_bytes && !slab)) return KVX_EINVAL;
    size_t need = 0, need_base = 0;
    cs->w = carve(ws, slab_bytes, &need, &need_base);
    if (ws_bytes < need_base) return KVX_EINVAL;
    if (ws_bytes < need) cs->w.pieces = nullptr;  // shared tiles stay on the register path
    cs->aligned = ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(slab)) & 15) == 0;
    cs->key = copy_key(descs, num_descs, desc_cap, pool_bytes, slab_bytes, cs->aligned, cs->w.pieces != nullptr,
                       ws);
    return KVX_OK;
}

// The descriptor checks and the tile lists (clears the control block first).
kvx_status launch_prep(const CopySetup &cs, uint64_t pool_bytes, uint64_t slab_bytes, const kvx_desc *descs,
                       const uint64_t *num_descs, uint64_t desc_cap, uint32_t *status, cudaStream_t s) {
    if (cudaMemsetAsync(cs.w.ctl, 0, sizeof(CopyCtl), s) != cudaSuccess) return KVX_ECUDA;
    k_copy_prep<<<sm_count() * 2, kThreads, 0, s>>>(descs, num_descs, desc_cap, pool_bytes, slab_bytes,
                                                     cs.aligned, cs.w.tile_desc, cs.w.jobs, cs.w.vec_tiles,
                                                     cs.w.pieces, cs.w.ctl, status, cs.key);
    KVX_LAUNCHED();
    return KVX_OK;
}

// The byte movement along prepared lists: the bulk kernel, then the vector path.
kvx_status launch_copy(bool pack, const CopySetup &cs, const uint8_t *pool_r, uint8_t *pool_w,
                       const uint8_t *slab_r, uint8_t *slab_w, uint64_t pool_bytes, uint64_t slab_bytes,
                       const kvx_desc *descs, const uint64_t *num_descs, uint64_t desc_cap, uint32_t *status,
                       cudaStream_t s) {
    if ((pack ? set_tma_smem<true>() : set_tma_smem<false>()) != cudaSuccess) return KVX_ECUDA;
    const int sms = sm_count();
    // One SM is left without a ring: the copy moves the same bytes per second
    // on the others (measured), and small kernels of a transfer planned
    // alongside (the single-block planner) run there during the copy instead
    // of waiting for it to end (overlapped default passes 1.373 -> 1.361 ms).
    const uint32_t bulk = (uint32_t)((sms > 1 ? sms - 1 : 1) * kTmaCtasPerSm);
    const size_t smem = (size_t)kStages * kTileBytes;
    const Ws &w = cs.w;
    if (pack)
        k_copy_tma<true><<<bulk, 32 * kBulkWarps, smem, s>>>(pool_r, pool_w, slab_r, slab_w, w.jobs, w.pieces,
                                                             w.ctl, status, cs.key);
    else
        k_copy_tma<false><<<bulk, 32 * kBulkWarps, smem, s>>>(pool_r, pool_w, slab_r, slab_w, w.jobs, w.pieces,
                                                              w.ctl, status, cs.key);
    KVX_LAUNCHED();
    // The register path starts as soon as every bulk block has begun (a
    // programmatic dependency), so its tiles move beside the bulk kernel's
    // instead of after them; the two write disjoint tiles.
    const uint32_t grid = (uint32_t)(sms * kCtasPerSm);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CopyCtl *cctl = w.ctl;
    const cudaError_t e =
        pack ? cudaLaunchKernelEx(&cfg, k_copy_vec<true>, pool_r, pool_w, slab_r, slab_w, pool_bytes, slab_bytes,
                                  cs.aligned, descs, num_descs, desc_cap, (const uint32_t *)w.tile_desc,
                                  (const uint32_t *)w.vec_tiles, cctl, cs.key, bulk)
             : cudaLaunchKernelEx(&cfg, k_copy_vec<false>, pool_r, pool_w, slab_r, slab_w, pool_bytes, slab_bytes,
                                  cs.aligned, descs, num_descs, desc_cap, (const uint32_t *)w.tile_desc,
                                  (const uint32_t *)w.vec_tiles, cctl, cs.key, bulk);
    if (e != cudaSuccess) return KVX_ECUDA;
    KVX_LAUNCHED();
    return KVX_OK;
}

// mode: 0 = prepare and copy, 1 = prepare only, 2 = copy along prepared lists
kvx_status launch(bool pack, int mode, const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r,
                  uint8_t *slab_w, uint64_t pool_bytes, uint64_t slab_bytes, const kvx_desc *descs,
                  const uint64_t *num_descs, uint64_t desc_cap, uint32_t *status, void *ws,
                  size_t ws_bytes, void *stream) {
    const void *pool = pool_r ? (const void *)pool_r : (const void *)pool_w;
    const void *slab = slab_r ? (const void *)slab_r : (const void *)slab_w;
    CopySetup cs;
    kvx_status st = setup(pool, pool_bytes, slab, slab_bytes, descs, num_descs, desc_cap, status, ws, ws_bytes,
                          &cs);
    if (st != KVX_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (mode != 2) {
        st = launch_prep(cs, pool_bytes, slab_bytes, descs, num_descs, desc_cap, status, s);
        if (st != KVX_OK || mode == 1) return st;
    }
    return launch_copy(pack, cs, pool_r, pool_w, slab_r, slab_w, pool_bytes, slab_bytes, descs, num_descs,
                       desc_cap, status, s);
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" size_t kvx_copy_workspace_size(uint64_t slab_bytes) {
    size_t bytes = 0;
    carve(nullptr, slab_bytes, &bytes);
    return bytes;
}

extern "C" kvx_status kvx_pack(const uint8_t *pool, uint64_t pool_bytes, const kvx_desc *descs,
                               const uint64_t *num_descs, uint64_t desc_capacity, uint8_t *slab,
                               uint64_t slab_bytes, uint32_t *status, void *ws, size_t ws_bytes,
                               void *stream) {
    return launch(true, 0, pool, nullptr, nullptr, slab, pool_bytes, slab_bytes, descs, num_descs,
                  desc_capacity, status, ws, ws_bytes, stream);
}

extern "C" kvx_status kvx_unpack(const uint8_t *slab, uint64_t slab_bytes, const kvx_desc *descs,
                                 const uint64_t *num_descs, uint64_t desc_capacity,
                                 uint8_t *dst_pool, uint64_t pool_bytes, uint32_t *status,
                                 void *ws, size_t ws_bytes, void *stream) {
    return launch(false, 0, nullptr, dst_pool, slab, nullptr, pool_bytes, slab_bytes, descs,
                  num_descs, desc_capacity, status, ws, ws_bytes, stream);
}

extern "C" kvx_status kvx_copy_prepare(const void *pool, uint64_t pool_bytes, const kvx_desc *descs,
                                       const uint64_t *num_descs, uint64_t desc_capacity, const void *slab,
                                       uint64_t slab_bytes, uint32_t *status, void *ws, size_t ws_bytes,
                                       void *stream) {
    return launch(true, 1, static_cast<const uint8_t *>(pool), nullptr, static_cast<const uint8_t *>(slab),
                  nullptr, pool_bytes, slab_bytes, descs, num_descs, desc_capacity, status, ws, ws_bytes,
                  stream);
}

extern "C" kvx_status kvx_pack_prepared(const uint8_t *pool, uint64_t pool_bytes, const kvx_desc *descs,
                                        const uint64_t *num_descs, uint64_t desc_capacity, uint8_t *slab,
                                        uint64_t slab_bytes, uint32_t *status, void *ws, size_t ws_bytes,
                                        void *stream) {
    return launch(true, 2, pool, nullptr, nullptr, slab, pool_bytes, slab_bytes, descs, num_descs,
                  desc_capacity, status, ws, ws_bytes, stream);
}

extern "C" kvx_status kvx_unpack_prepared(const uint8_t *slab, uint64_t slab_bytes, const kvx_desc *descs,
                                          const uint64_t *num_descs, uint64_t desc_capacity,
                                          uint8_t *dst_pool, uint64_t pool_bytes, uint32_t *status,
                                          void *ws, size_t ws_bytes, void *stream) {
    return launch(false, 2, nullptr, dst_pool, slab, nullptr, pool_bytes, slab_bytes, descs, num_descs,
                  desc_capacity, status, ws, ws_bytes, stream);
}

// ------------------------------------------------------------ no-allocation pack
//
// kvx_pack_noalloc: kvx_pack for callers that cannot allocate device memory
// (for instance code running where cudaMalloc is forbidden or would stall:
// an allocation-free serving loop, a host thread without its own allocator,
// a binding to a language runtime that cannot hand out device buffers).  Its
// scratch is this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds the array until the process exits.
// All calls share it, so calls that overlap on the GPU (two streams, or two
// host threads) race on it and must be serialised by the caller; each call
// clears the part that has to start at zero before using it.
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)4 << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_pack_scratch[kNoallocScratchBytes];

// Device address of g_pack_scratch in the current context.  The name is only
// a host-side stand-in, so the address is looked up on every call, with the
// caller's device and context current: an address remembered from an earlier
// call could belong to a context that has since been reset or to another
// context on the same device.  Once this file's module is loaded in a
// context (its first call there, or any earlier launch of a kernel of this
// file), the lookup is a host-side table search that touches no device
// memory.
void *pack_scratch_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pack_scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return p;
}

}  // namespace

extern "C" kvx_status kvx_pack_noalloc(const uint8_t *pool, uint64_t pool_bytes,
                                       const kvx_desc *descs, const uint64_t *num_descs,
                                       uint64_t desc_capacity, uint8_t *slab, uint64_t slab_bytes,
                                       uint32_t *status, void *stream) {
    // the scratch always holds the tile lists, and the piece list too while it
    // fits (slabs up to about 5000 tiles); beyond that, shared tiles take the
    // register path
    size_t full = 0, base = 0;
    carve(nullptr, slab_bytes, &full, &base);
    if (base > kNoallocScratchBytes) return KVX_ECAPACITY;
    void *scratch = pack_scratch_address();
    if (!scratch) return KVX_ECUDA;
    return launch(true, 0, pool, nullptr, nullptr, slab, pool_bytes, slab_bytes, descs, num_descs,
                  desc_capacity, status, scratch, kNoallocScratchBytes, stream);
}
