// Fused softmax + TopK: kernel choice and launch.
//
// A row is split over a cluster of CLUSTER CTAs of 512 threads, each thread
// holding 8 vectors (32 fp32) of a tile in registers; CLUSTER is the smallest
// power of two (up to 8) whose CTAs cover the row in one tile of 16384
// elements each, and longer rows loop over several tiles per CTA.
#include "host_common.h"
#include "internal.h"
#include "kernels/topk_kernel.cuh"

namespace os {

constexpr int kTopkThreads = 512;
constexpr int kTopkVpt = 8;
constexpr int kTopkKmax = 64;
constexpr int kTopkCap = 512;
constexpr int kTopkMaxCluster = 8;
constexpr int64_t kTopkTileElems = int64_t(kTopkThreads) * kTopkVpt * 4;

using TopkKernel = void (*)(const float*, float*, int*, int64_t, int, int, KernelCtl);

template <int C>
constexpr TopkKernel topk_instance() {
    return topk_rows_kernel<kTopkThreads, kTopkVpt, C, kTopkKmax, kTopkCap>;
}

static TopkKernel topk_kernel_for(int cluster) {
    switch (cluster) {
        case 1: return topk_instance<1>();
        case 2: return topk_instance<2>();
        case 4: return topk_instance<4>();
        default: return topk_instance<8>();
    }
}

os_status plan_topk(int64_t rows, int64_t cols, int K, os_plan* p) {
    (void)K;
    if (!device_info()) return OS_ERR_CUDA;
    os_plan q = {};
    q.path = OS_PATH_ONCHIP;
    q.threads = kTopkThreads;
    q.vectors_per_thread = kTopkVpt;
    q.cluster = pow2_at_least(ceil_div(cols + 3, kTopkTileElems));
    if (q.cluster > kTopkMaxCluster) q.cluster = kTopkMaxCluster;
    q.grid = min64(rows, kMaxClustersPerLaunch) * q.cluster;
    *p = q;
    return OS_OK;
}

cudaError_t launch_topk(const os_plan& p, const float* x, float* vals, int32_t* idx,
                        int64_t rows, int cols, int K, const KernelCtl& ctl,
                        cudaStream_t stream) {
    TopkKernel k = topk_kernel_for(p.cluster);
    if (!prepare_kernel(k, p.cluster, 0)) return cudaErrorInvalidValue;
    return launch_kernel(k, p.grid, p.threads, p.cluster, 0, stream, x, vals,
                         reinterpret_cast<int*>(idx), rows, cols, K, ctl);
}

}  // namespace os
