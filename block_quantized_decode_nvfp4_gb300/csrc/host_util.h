// host_util.h -- host-side launch helpers shared by the kernels' launchers:
// per-device attributes and per-kernel occupancy, both cached.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <mutex>

namespace bqd {

// Process-wide launch options (bqd_set_launch_flags).
constexpr unsigned kLaunchPdl = 1u;
inline std::atomic<unsigned>& launch_flags_ref()
{
    static std::atomic<unsigned> flags{0};
    return flags;
}
inline unsigned launch_flags() { return launch_flags_ref().load(std::memory_order_relaxed); }

struct DevInfo {
    int sms = 0;
    int max_smem_optin = 0;
};

inline DevInfo dev_info(int dev)
{
    static std::mutex mu;
    static DevInfo cache[64];
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return DevInfo{};
    if (cache[dev].sms == 0) {
        cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&cache[dev].max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return cache[dev];
}

// Occupancy of one kernel (one cache object per kernel instantiation) at a
// dynamic shared-memory size, cached per device for a few sizes.
struct OccCache {
    std::mutex mu;
    bool attr_set[64] = {};
    size_t smem[64][4] = {};
    int val[64][4] = {};
};

inline int blocks_per_sm(OccCache& c, const void* kern, int dev, int threads, size_t smem)
{
    std::lock_guard<std::mutex> g(c.mu);
    if (dev < 0 || dev >= 64) return 1;
    if (!c.attr_set[dev]) {
        // Allow dynamic shared memory up to the opt-in limit minus the
        // kernel's static shared memory. Errors of these calls are consumed
        // here so that they cannot surface as a launch error later.
        cudaFuncAttributes fa{};
        size_t static_smem = 0;
        if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess) static_smem = fa.sharedSizeBytes;
        const int optin = dev_info(dev).max_smem_optin;
        if (optin > static_cast<int>(static_smem))
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(static_smem));
        cudaGetLastError();
        c.attr_set[dev] = true;
    }
    for (int i = 0; i < 4; ++i)
        if (c.val[dev][i] && c.smem[dev][i] == smem) return c.val[dev][i];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) cudaGetLastError();
    if (n < 1) n = 1;
    for (int i = 0; i < 4; ++i)
        if (!c.val[dev][i]) {
            c.smem[dev][i] = smem;
            c.val[dev][i] = n;
            break;
        }
    return n;
}

}  // namespace bqd
