// Diagnostic: the bounded waits of libkvx give up and report instead of
// hanging.  Three tiny kernels wait on conditions that nothing will satisfy --
// a grid barrier that expects one block more than is launched, an mbarrier
// that expects bytes no copy will deliver, and the planner's cross-block flag
// wait on a flag that nothing sets -- and each raises KVX_S_TIMEOUT in its own
// status word when its limit runs out.  Nothing faults: no copy is ever in
// flight, and each wait ends by itself after about a second.
#include "kvx_common.cuh"

namespace kvx {
namespace {

__device__ GridSync g_selftest_sync;

__global__ void k_selftest_barrier(uint32_t *status) {
    // two blocks wait for a third that is never launched
    if (!grid_barrier(&g_selftest_sync, gridDim.x + 1) && threadIdx.x == 0)
        atomicOr(status, KVX_S_TIMEOUT);
}

__global__ void k_selftest_mbarrier(uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_arrive_expect_tx(&bar, 16);  // 16 bytes that no copy will bring
    if (!mbar_wait(&bar, 0)) atomicOr(status, KVX_S_TIMEOUT);
}

}  // namespace
}  // namespace kvx

namespace kvx {
kvx_status launch_selftest_flag_wait(uint32_t *status, cudaStream_t s);  // kvx_plan.cu
}

using namespace kvx;

extern "C" kvx_status kvx_selftest_timeouts(uint32_t *status, void *stream) {
    if (!status) return KVX_EINVAL;
    cudaStream_t s = as_stream(stream);
    void *gs = nullptr;
    if (cudaGetSymbolAddress(&gs, g_selftest_sync) != cudaSuccess) return KVX_ECUDA;
    if (cudaMemsetAsync(gs, 0, sizeof(GridSync), s) != cudaSuccess) return KVX_ECUDA;
    void *args[] = {&status};
    if (cudaLaunchCooperativeKernel((const void *)k_selftest_barrier, dim3(2), dim3(32), args, 0, s) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return KVX_ECUDA;
    }
    note_launch();
    k_selftest_mbarrier<<<1, 32, 0, s>>>(status + 1);
    KVX_LAUNCHED();
    return launch_selftest_flag_wait(status + 2, s);
}
