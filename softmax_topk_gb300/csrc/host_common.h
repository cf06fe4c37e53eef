// host_common.h -- host-side helpers shared by the library's translation units:
// cached device attributes, cluster launches and occupancy queries.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/os_softmax.h"

namespace os {

struct DeviceInfo {
    int device = -1;
    int sms = 0;
};

// Attributes of the current device, queried once per device ordinal.
inline const DeviceInfo* device_info() {
    constexpr int kMaxDevices = 64;
    static DeviceInfo cache[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = cache[dev];
    if (d.device < 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        d.sms = sms;
        d.device = dev;
    }
    return &d;
}

// Launch `kernel` with `cluster` CTAs per thread-block cluster (1 = none).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int64_t grid, int threads, int cluster,
                          int smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (cluster > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Opt `kernel` into `smem` bytes of dynamic shared memory and, for cluster
// sizes above 8, into non-portable cluster sizes.  Returns false on failure.
// Done once per (device, kernel): later calls are a table lookup, so launches
// (and stream captures) do not repeat the attribute calls.
template <typename... KArgs>
bool prepare_kernel(void (*kernel)(KArgs...), int cluster, int smem) {
    const void* k = reinterpret_cast<const void*>(kernel);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, std::pair<int, int>> done;  // smem, cluster
    std::lock_guard<std::mutex> lock(mu);
    auto& d = done[{dev, k}];
    // static plus dynamic shared memory above 48 KB needs the opt-in, so the
    // limit is raised for any dynamic size (a no-op below it)
    if (smem > d.first) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        d.first = smem;
    }
    if (cluster > 8 && d.second <= 8) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        d.second = cluster;
    }
    return true;
}

// How many clusters of `cluster` CTAs of `kernel` can be resident at once on
// the current device (0 if the size cannot be launched).
template <typename... KArgs>
int max_active_clusters(void (*kernel)(KArgs...), int threads, int cluster, int smem = 0) {
    if (!prepare_kernel(kernel, cluster, smem)) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kernel), &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Resident CTAs per SM of `kernel` (cached per device, kernel, block and smem size).
template <typename... KArgs>
int blocks_per_sm(void (*kernel)(KArgs...), int threads, int smem = 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static std::map<std::pair<std::pair<int, const void*>, std::pair<int, int>>, int> cache;
    const auto key = std::make_pair(std::make_pair(dev, reinterpret_cast<const void*>(kernel)),
                                    std::make_pair(threads, smem));
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (!prepare_kernel(kernel, 1, smem)) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void*>(kernel),
                                                      threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int pow2_at_least(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Upper bound on clusters launched per call; the kernels loop over the rest.
constexpr int64_t kMaxClustersPerLaunch = int64_t(1) << 22;

}  // namespace os
