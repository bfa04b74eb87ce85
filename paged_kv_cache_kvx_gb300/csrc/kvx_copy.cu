// Pack and unpack: the data movement of the planned reads (pegaflow PR #350,
// Requester step 4: one coalesced read per dense group, per-block reads for a
// non-dense group; READ splitting: 32 MiB descriptors).  Pack gathers
// holder-pool bytes into the dense slab; unpack is the inverse scatter.
//
// HBM-bound copy, no contraction.  The slab side is always contiguous (the
// descriptors tile it), so the work is cut into fixed 32 KiB slab tiles:
// a persistent grid walks the tiles round-robin, so at any moment the grid
// streams one contiguous window of the slab and, per descriptor, of the pool.
// A prep kernel checks the descriptors and records, for every tile, the
// descriptor holding the tile's first byte.  Inside a tile:
//   - one descriptor covers it (every tile of a dense 32 MiB read): each
//     thread moves 8 x 16-byte vectors, all loads issued before the stores;
//   - several descriptors, all 16-byte aligned (4 KiB / 512 B segment
//     reads): the tile's descriptors are staged in shared memory and every
//     16-byte vector finds its descriptor by binary search;
//   - anything unaligned: byte copies (correct for any layout, slow).
#include "kvx_common.cuh"

namespace kvx {
namespace {

constexpr int kThreads = 256;
constexpr uint64_t kTileBytes = 32 * 1024;
constexpr int kVecPerThread = (int)(kTileBytes / (kThreads * 16));  // 8
constexpr int kCtasPerSm = 3;

struct CopyCtl {
    unsigned long long used;  // end of the last descriptor (slab bytes in use)
    uint32_t bad;             // descriptors do not tile the slab
    uint32_t pad;
};

struct Ws {
    CopyCtl *ctl;
    uint32_t *tile_desc;  // [ceil(slab_bytes / kTileBytes)]
};

Ws carve(void *base, uint64_t slab_bytes, size_t *bytes) {
    Carver c(base);
    Ws w;
    w.ctl = c.take<CopyCtl>(1);
    w.tile_desc = c.take<uint32_t>(ceil_div(slab_bytes, kTileBytes));
    *bytes = c.off;
    return w;
}

__device__ __forceinline__ bool in_range(uint64_t off, uint64_t len, uint64_t size) {
    return off <= size && len <= size - off;
}

// One thread per descriptor: tiling check, bounds check, tile -> descriptor map.
__global__ void __launch_bounds__(kThreads)
k_copy_prep(const kvx_desc *__restrict__ descs, const uint64_t *__restrict__ num_descs,
            uint64_t desc_cap, uint64_t pool_bytes, uint64_t slab_bytes,
            uint32_t *__restrict__ tile_desc, CopyCtl *ctl, uint32_t *status) {
    const uint64_t n = *num_descs < desc_cap ? *num_descs : desc_cap;
    const uint64_t ntiles = ceil_div(slab_bytes, kTileBytes);
    uint32_t bits = 0;
    for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
         k += (uint64_t)gridDim.x * blockDim.x) {
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
        // tiles whose first byte lies in [local, local + len)
        uint64_t t = ceil_div(d.local, kTileBytes);
        const uint64_t t_end = (d.local + d.len - 1) / kTileBytes;
        for (; t <= t_end && t < ntiles; t++) tile_desc[t] = (uint32_t)k;
    }
    if (bits) atomicOr(status, bits);
}

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(uint8_t *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

// Copy slab range [x0, x1) of one span; slab offset x maps to pool offset
// x + delta.  PACK: pool -> slab; else slab -> pool.
template <bool PACK>
__device__ __forceinline__ void copy_span_vec(const uint8_t *pool_r, uint8_t *pool_w,
                                              const uint8_t *slab_r, uint8_t *slab_w, uint64_t x0,
                                              uint64_t x1, uint64_t delta) {
    for (uint64_t x = x0 + (uint64_t)threadIdx.x * 16; x < x1;
         x += (uint64_t)kThreads * 16 * kVecPerThread) {
        uint4 v[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; u++) {
            const uint64_t xx = x + (uint64_t)u * kThreads * 16;
            if (xx < x1) v[u] = PACK ? ld_stream(pool_r + xx + delta) : ld_stream(slab_r + xx);
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; u++) {
            const uint64_t xx = x + (uint64_t)u * kThreads * 16;
            if (xx < x1) {
                if (PACK) st_stream(slab_w + xx, v[u]);
                else st_stream(pool_w + xx + delta, v[u]);
            }
        }
    }
}

template <bool PACK>
__device__ __forceinline__ void copy_span_bytes(const uint8_t *pool_r, uint8_t *pool_w,
                                                const uint8_t *slab_r, uint8_t *slab_w, uint64_t x0,
                                                uint64_t x1, uint64_t delta) {
    for (uint64_t x = x0 + threadIdx.x; x < x1; x += kThreads) {
        if (PACK) slab_w[x] = pool_r[x + delta];
        else pool_w[x + delta] = slab_r[x];
    }
}

template <bool PACK>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_copy(const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r, uint8_t *slab_w,
       uint64_t pool_bytes, uint64_t slab_bytes, bool bases_aligned,
       const kvx_desc *__restrict__ descs, const uint64_t *__restrict__ num_descs,
       uint64_t desc_cap, const uint32_t *__restrict__ tile_desc, const CopyCtl *ctl) {
    __shared__ uint64_t s_lo[kThreads + 1];
    __shared__ uint64_t s_delta[kThreads];
    __shared__ uint8_t s_ok[kThreads];
    if (ctl->bad) return;
    const uint64_t n = *num_descs < desc_cap ? *num_descs : desc_cap;
    const uint64_t used = ctl->used < slab_bytes ? ctl->used : slab_bytes;
    const uint64_t ntiles = ceil_div(used, kTileBytes);
    for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        uint64_t lo = t * kTileBytes;
        const uint64_t hi = lo + kTileBytes < used ? lo + kTileBytes : used;
        uint64_t k = tile_desc[t];
        if (k >= n) continue;
        const kvx_desc d0 = descs[k];
        if (d0.local <= lo && hi - d0.local <= d0.len) {
            // one descriptor covers the whole tile
            if (!in_range(d0.remote, d0.len, pool_bytes) || !in_range(d0.local, d0.len, slab_bytes))
                continue;
            const uint64_t delta = d0.remote - d0.local;
            const bool al = bases_aligned && ((lo | hi | delta) & 15) == 0;
            if (al) copy_span_vec<PACK>(pool_r, pool_w, slab_r, slab_w, lo, hi, delta);
            else copy_span_bytes<PACK>(pool_r, pool_w, slab_r, slab_w, lo, hi, delta);
            continue;
        }
        // several descriptors: stage up to kThreads of them at a time
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
                constexpr int U = kVecPerThread / 2;
                for (uint64_t x = lo + (uint64_t)threadIdx.x * 16; x < bhi;
                     x += (uint64_t)kThreads * 16 * U) {
                    uint4 v[U];
                    uint64_t dst[U];
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        const uint64_t xx = x + (uint64_t)u * kThreads * 16;
                        int a = 0, z = nb;  // last span with s_lo <= xx
                        while (z - a > 1) {
                            const int m = (a + z) >> 1;
                            if (s_lo[m] <= xx) a = m; else z = m;
                        }
                        dst[u] = ~0ull;
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

kvx_status launch(bool pack, const uint8_t *pool_r, uint8_t *pool_w, const uint8_t *slab_r,
                  uint8_t *slab_w, uint64_t pool_bytes, uint64_t slab_bytes, const kvx_desc *descs,
                  const uint64_t *num_descs, uint64_t desc_cap, uint32_t *status, void *ws,
                  size_t ws_bytes, void *stream) {
    if (!descs || !num_descs || !status || !ws) return KVX_EINVAL;
    if ((pool_bytes && !(pool_r || pool_w)) || (slab_bytes && !(slab_r || slab_w))) return KVX_EINVAL;
    size_t need = 0;
    Ws w = carve(ws, slab_bytes, &need);
    if (ws_bytes < need) return KVX_EINVAL;
    cudaStream_t s = as_stream(stream);
    if (cudaMemsetAsync(w.ctl, 0, sizeof(CopyCtl), s) != cudaSuccess) return KVX_ECUDA;
    const uint64_t prep_grid = ceil_div(desc_cap ? desc_cap : 1, kThreads);
    const uint64_t prep_max = (uint64_t)sm_count() * kCtasPerSm;
    const uint32_t pg = (uint32_t)(prep_grid < prep_max ? prep_grid : prep_max);
    k_copy_prep<<<pg, kThreads, 0, s>>>(descs, num_descs, desc_cap, pool_bytes, slab_bytes,
                                        w.tile_desc, w.ctl, status);
    KVX_LAUNCHED();
    const uintptr_t pa = reinterpret_cast<uintptr_t>(pool_r ? (const void *)pool_r : pool_w);
    const uintptr_t sa = reinterpret_cast<uintptr_t>(slab_r ? (const void *)slab_r : slab_w);
    const bool aligned = ((pa | sa) & 15) == 0;
    const uint32_t grid = (uint32_t)(sm_count() * kCtasPerSm);
    if (pack)
        k_copy<true><<<grid, kThreads, 0, s>>>(pool_r, pool_w, slab_r, slab_w, pool_bytes, slab_bytes,
                                               aligned, descs, num_descs, desc_cap, w.tile_desc, w.ctl);
    else
        k_copy<false><<<grid, kThreads, 0, s>>>(pool_r, pool_w, slab_r, slab_w, pool_bytes,
                                                slab_bytes, aligned, descs, num_descs, desc_cap,
                                                w.tile_desc, w.ctl);
    KVX_LAUNCHED();
    return KVX_OK;
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
    return launch(true, pool, nullptr, nullptr, slab, pool_bytes, slab_bytes, descs, num_descs,
                  desc_capacity, status, ws, ws_bytes, stream);
}

extern "C" kvx_status kvx_unpack(const uint8_t *slab, uint64_t slab_bytes, const kvx_desc *descs,
                                 const uint64_t *num_descs, uint64_t desc_capacity,
                                 uint8_t *dst_pool, uint64_t pool_bytes, uint32_t *status,
                                 void *ws, size_t ws_bytes, void *stream) {
    return launch(false, nullptr, dst_pool, slab, nullptr, pool_bytes, slab_bytes, descs,
                  num_descs, desc_capacity, status, ws, ws_bytes, stream);
}
