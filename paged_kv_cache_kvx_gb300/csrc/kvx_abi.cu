// Library-wide bookkeeping of libkvx: launch accounting and device queries.
#include <atomic>

#include "kvx_common.cuh"

namespace kvx {

namespace {
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
}  // namespace

void note_launch(uint32_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < kMaxDevices) {
        const int cached = g_sms[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev < kMaxDevices) g_sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace kvx

extern "C" uint64_t kvx_launch_count(void) {
    return kvx::g_launches.load(std::memory_order_relaxed);
}

extern "C" uint32_t kvx_version(void) { return 100; }
