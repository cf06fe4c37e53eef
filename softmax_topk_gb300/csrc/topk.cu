// Fused softmax + TopK: kernel choice and launch.
//
// A row is split over a cluster of CLUSTER CTAs of 512 threads; CLUSTER is
// the smallest power of two (up to 8) whose segments are at most 26000
// elements (two CTAs of about 100 KB of shared memory fit one SM), and rows
// longer than 8 tiles of 32768 elements loop over several tiles per CTA.  The
// tile frame is dynamic shared memory sized to the segment (at most one
// tile), staged by four bulk copies.
#include "host_common.h"
#include "internal.h"
#include "kernels/topk_kernel.cuh"

namespace os {

constexpr int kTopkThreads = 512;
constexpr int kTopkTile = 32768;
constexpr int kTopkKmax = 64;
constexpr int kTopkCap = 512;
constexpr int kTopkChunks = 4;
constexpr int kTopkMaxCluster = 8;
constexpr int kTopkSegmentTarget = 26000;  // longest segment per CTA before adding CTAs

using TopkKernel = void (*)(const float*, float*, int*, int64_t, int, int, KernelCtl);

template <int C>
constexpr TopkKernel topk_instance() {
    return topk_rows_kernel<kTopkThreads, C, kTopkTile, kTopkKmax, kTopkCap, kTopkChunks>;
}

static TopkKernel topk_kernel_for(int cluster) {
    switch (cluster) {
        case 1: return topk_instance<1>();
        case 2: return topk_instance<2>();
        case 4: return topk_instance<4>();
        default: return topk_instance<8>();
    }
}

static int frame_bytes(int64_t cols, int cluster) {
    const int64_t seg = ceil_div(cols, cluster);
    const int64_t tile = seg < kTopkTile ? seg : kTopkTile;
    return static_cast<int>(((tile + 8) * 4 + 15) / 16 * 16);
}

os_status plan_topk(int64_t rows, int64_t cols, int K, os_plan* p) {
    (void)K;
    if (!device_info()) return OS_ERR_CUDA;
    os_plan q = {};
    q.path = OS_PATH_ONCHIP;
    q.threads = kTopkThreads;
    q.cluster = pow2_at_least(ceil_div(cols, kTopkSegmentTarget));
    if (q.cluster > kTopkMaxCluster) q.cluster = kTopkMaxCluster;
    const int64_t seg = ceil_div(cols, q.cluster);
    q.vectors_per_thread = static_cast<int32_t>(ceil_div(seg < kTopkTile ? seg : kTopkTile,
                                                         4 * kTopkThreads));
    q.stages = kTopkChunks;
    q.grid = min64(rows, kMaxClustersPerLaunch) * q.cluster;
    *p = q;
    return OS_OK;
}

cudaError_t launch_topk(const os_plan& p, const float* x, float* vals, int32_t* idx,
                        int64_t rows, int cols, int K, const KernelCtl& ctl,
                        cudaStream_t stream) {
    TopkKernel k = topk_kernel_for(p.cluster);
    const int smem = frame_bytes(cols, p.cluster);
    if (!prepare_kernel(k, p.cluster, frame_bytes(kTopkTile, 1))) return cudaErrorInvalidValue;
    return launch_kernel(k, p.grid, p.threads, p.cluster, smem, stream, x, vals,
                         reinterpret_cast<int*>(idx), rows, cols, K, ctl);
}

}  // namespace os
