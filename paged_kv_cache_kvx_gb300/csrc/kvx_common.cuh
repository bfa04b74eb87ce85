// Internal helpers shared by the libkvx kernels (sm_103a).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvx.h"

namespace kvx {

constexpr uint32_t kNone = 0xFFFFFFFFu;

// ------------------------------------------------------------------ host side

// Counts every kernel this library launches (reported by kvx_launch_count).
void note_launch(uint32_t n = 1);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

// Carves consecutive 256-byte aligned sub-buffers out of a workspace.  With a
// null base it only measures.
struct Carver {
    char *base;
    size_t off = 0;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    template <class T>
    T *take(size_t n) {
        off = align_up(off, 256);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += sizeof(T) * (n ? n : 1);
        return p;
    }
};

#define KVX_LAUNCHED()                                  \
    do {                                                \
        ::kvx::note_launch();                           \
        if (cudaPeekAtLastError() != cudaSuccess) {     \
            (void)cudaGetLastError();                   \
            return KVX_ECUDA;                           \
        }                                               \
    } while (0)

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void raise(uint32_t *st, uint32_t bits) {
    if (bits) atomicOr(st, bits);
}

// Grid barrier for cooperative launches (every participating block is
// resident).  One monotonic arrival counter, zeroed before the launch: the
// arrivals of the k-th barrier are exactly k*nblocks .. (k+1)*nblocks - 1 (no
// block passes a barrier before all have reached it), so a block's own
// arrival number tells it the count that releases it, and the last arrival
// releases everyone with no second atomic.  Waiters spin on the counter, hot
// at first and then with short sleeps.  The wait is bounded: after about a
// second a block gives up, raises the shared abort flag and returns false,
// and so do the blocks still waiting.  With a single participating block it
// is a plain __syncthreads().
struct GridSync {
    uint32_t count;
    uint32_t abort;
};

// Waits are bounded in time (%globaltimer nanoseconds) with a poll-count
// backstop.
constexpr uint64_t kWaitNs = 1000000000ull;  // one second
constexpr uint32_t kBarrierPolls = 1u << 26;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool grid_barrier(GridSync *gs, uint32_t nblocks) {
    __shared__ int s_ok;
    if (nblocks <= 1) {
        __syncthreads();
        return true;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        const uint32_t arrived = atomicAdd(&gs->count, 1u);
        const uint32_t target = (arrived / nblocks + 1) * nblocks;
        if (arrived + 1 != target) {
            const volatile uint32_t *vabort = &gs->abort;
            uint64_t t0 = 0;
            for (uint32_t polls = 0; ld_acquire_gpu(&gs->count) < target; polls++) {
                if (polls >= 256) {
                    if (polls == 256) t0 = global_ns();
                    if (*vabort || polls >= kBarrierPolls || global_ns() - t0 > kWaitNs) {
                        atomicExch(&gs->abort, 1u);
                        ok = 0;
                        break;
                    }
                    __nanosleep(32);
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Loads that bypass L1: data other blocks wrote earlier in the same kernel.
// Types aligned to 16 bytes move in 16-byte pieces, others in 8-byte ones.
template <class T>
__device__ __forceinline__ T ld_cg(const T *p) {
    static_assert(sizeof(T) % 8 == 0, "8-byte multiple");
    T v;
    if constexpr (alignof(T) >= 16 && sizeof(T) % 16 == 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p);
        uint4 *dst = reinterpret_cast<uint4 *>(&v);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(T) / 16); i++) dst[i] = __ldcg(src + i);
    } else {
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p);
        unsigned long long *dst = reinterpret_cast<unsigned long long *>(&v);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(T) / 8); i++) dst[i] = __ldcg(src + i);
    }
    return v;
}

// Warp-level inclusive scans.
template <class T>
__device__ __forceinline__ T warp_incl_sum(T v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        T o = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

template <class T>
__device__ __forceinline__ T warp_incl_max(T v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        T o = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v = o > v ? o : v;
    }
    return v;
}

// Block-wide exclusive sum over one value per thread; returns the exclusive
// prefix and writes the block total.  `sh` holds >= 32 elements.
template <class T>
__device__ __forceinline__ T block_excl_sum(T v, T *sh, T *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    T incl = warp_incl_sum(v);
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        T w = lane < nwarps ? sh[lane] : T(0);
        T wi = warp_incl_sum(w);
        sh[lane] = wi - w;
        if (lane == 31) sh[32] = wi;
    }
    __syncthreads();
    T res = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Block-wide inclusive max (values are signed; identity = INT64_MIN).
__device__ __forceinline__ int64_t block_incl_max(int64_t v, int64_t *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int64_t incl = warp_incl_max(v);
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < nwarps ? sh[lane] : INT64_MIN;
        int64_t wi = warp_incl_max(w);
        sh[lane] = wi;
    }
    __syncthreads();
    int64_t prev = warp > 0 ? sh[warp - 1] : INT64_MIN;
    __syncthreads();
    return incl > prev ? incl : prev;
}

// Exclusive prefix sum, in place, of n uint64 values by one whole block
// (used by last blocks on per-tile aggregates).  Returns the total.
__device__ inline uint64_t block_scan_inplace_u64(uint64_t *a, uint64_t n) {
    __shared__ uint64_t sh[33];
    __shared__ uint64_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (uint64_t base = 0; base < n; base += blockDim.x) {
        const uint64_t i = base + threadIdx.x;
        uint64_t v = i < n ? __ldcg(a + i) : 0;
        uint64_t tot;
        uint64_t ex = block_excl_sum<uint64_t>(v, sh, &tot);
        if (i < n) a[i] = carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
    return carry;
}

// Exclusive prefix sum, in place, of n uint32 values where every thread owns
// a contiguous span (large n, e.g. a digit histogram matrix).
__device__ inline uint32_t block_scan_inplace_span_u32(uint32_t *a, uint64_t n) {
    __shared__ uint64_t sh[33];
    const uint64_t per = (n + blockDim.x - 1) / blockDim.x;
    const uint64_t lo = per * threadIdx.x;
    const uint64_t hi = lo + per < n ? lo + per : n;
    uint64_t s = 0;
    for (uint64_t i = lo; i < hi; i++) s += __ldcg(a + i);
    uint64_t tot;
    uint64_t ex = block_excl_sum<uint64_t>(s, sh, &tot);
    for (uint64_t i = lo; i < hi; i++) {
        uint32_t v = __ldcg(a + i);
        a[i] = (uint32_t)ex;
        ex += v;
    }
    __syncthreads();
    return (uint32_t)tot;
}

// ------------------------------------------------- mbarrier and bulk copies

constexpr uint32_t kSpinLimit = 1u << 28;  // backstop; the time bound ends waits first

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false after about a second (try_wait itself may suspend the
// thread for a while, so the bound is time, not a poll count).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kSpinLimit; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_g2s(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace kvx
