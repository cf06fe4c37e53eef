// Fused softmax + TopK: kernel choice and launch.
//
// A row is split over a cluster of CLUSTER CTAs of 256 threads, each thread
// holding 8 vectors (32 fp32) of a tile; CLUSTER is the smallest power of two
// (up to 8) whose one-tile capacity covers the row, and longer rows loop over
// several tiles per CTA.
#include "host_common.h"
#include "internal.h"
#include "kernels/topk_kernel.cuh"

namespace os {

constexpr int kTopkThreads = 256;
constexpr int kTopkVpt = 8;
constexpr int kTopkKmax = 64;
constexpr int kTopkCap = 1024;
constexpr int kTopkMaxCluster = 8;

using TopkKernel = void (*)(const float*, float*, int*, int64_t, int, int);

static TopkKernel topk_kernel_for(int cluster) {
    switch (cluster) {
        case 1: return topk_rows_kernel<kTopkThreads, kTopkVpt, 1, kTopkKmax, kTopkCap>;
        case 2: return topk_rows_kernel<kTopkThreads, kTopkVpt, 2, kTopkKmax, kTopkCap>;
        case 4: return topk_rows_kernel<kTopkThreads, kTopkVpt, 4, kTopkKmax, kTopkCap>;
        default: return topk_rows_kernel<kTopkThreads, kTopkVpt, 8, kTopkKmax, kTopkCap>;
    }
}

os_status plan_topk(int64_t rows, int64_t cols, int K, os_plan* p) {
    (void)K;
    if (!device_info()) return OS_ERR_CUDA;
    const int64_t frame_vectors = ceil_div(cols + 3, 4);
    const int64_t tile = int64_t(kTopkThreads) * kTopkVpt;
    os_plan q = {};
    q.path = OS_PATH_ONCHIP;
    q.threads = kTopkThreads;
    q.vectors_per_thread = kTopkVpt;
    q.cluster = pow2_at_least(ceil_div(frame_vectors, tile));
    if (q.cluster > kTopkMaxCluster) q.cluster = kTopkMaxCluster;
    q.grid = min64(rows, kMaxClustersPerLaunch) * q.cluster;
    *p = q;
    return OS_OK;
}

cudaError_t launch_topk(const os_plan& p, const float* x, float* vals, int32_t* idx,
                        int64_t rows, int cols, int K, cudaStream_t stream) {
    return launch_kernel(topk_kernel_for(p.cluster), p.grid, p.threads, p.cluster, stream, x,
                         vals, reinterpret_cast<int*>(idx), rows, cols, K);
}

}  // namespace os
