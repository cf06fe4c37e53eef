// Fused softmax + TopK: kernel choice and launch.
//
// Persistent CTAs of 512 threads, two per SM, each taking whole rows in
// chunks of 4 16-byte blocks per thread (8192 fp32); with fewer rows than
// resident CTAs a row is split over a cluster of S CTAs (S <= 8 for K <= 64,
// S <= 2 for K up to 256, and no more CTAs than the row has chunks) that merge
// through distributed shared memory.  Batches of many rows of up to 65536
// columns with K <= 64 take CTAs of 256 threads, four per SM.
#include "host_common.h"
#include "internal.h"
#include "kernels/topk_kernel.cuh"

namespace os {

constexpr int kTopkThreads = 512;
constexpr int kTopkVpt = 4;      // 16-byte blocks per thread per chunk
constexpr int kTopkCap = 2048;   // candidates
constexpr int kTopkGroups = 4;   // block keys kept per thread slot (groups of chunks)
constexpr int kTopkFcap = 4096;  // blocks read again in pass 2 (256 per warp)
constexpr int kTopkDynBytes =
    int(sizeof(TopkDynSmem<kTopkThreads, kTopkVpt, kTopkGroups, kTopkFcap>));
// Two builds: K <= 64 with clusters of up to 8 CTAs per row, and
// 64 < K <= 256 with up to 2 (its exchange lists are 4x longer).
constexpr int kTopkKmaxSmall = 64, kTopkClusterSmall = 8;
constexpr int kTopkKmaxLarge = 256, kTopkClusterLarge = 2;

// Many rows (at least as many as resident CTAs of 256 threads, K <= 64, one
// CTA per row, rows of up to kTopkManyMaxCols): CTAs of 256 threads, four
// per SM, so that while some CTAs run a row's threshold, rereads and ranking
// (when they read nothing) more CTAs of the SM stream; their keys cover
// groups of chunks twice as fine.  Measured on GB300 (K = 8 / 64, us per
// launch against the 512-thread CTAs): 4096x32000 109 / 127 against 137 /
// 162, 4096x50257 177 / 202 against 193 / 220; 2048x128256 slower (193 / 215
// against 186 / 205), so longer rows keep the 512-thread CTAs.
constexpr int kTopkThreadsMany = 256;
constexpr int64_t kTopkManyMaxCols = 65536;
constexpr int kTopkGroupsMany = 8;
constexpr int kTopkDynBytesMany =
    int(sizeof(TopkDynSmem<kTopkThreadsMany, kTopkVpt, kTopkGroupsMany, kTopkFcap>));

template <int KMAX, int MAXC, bool PLAIN>
static auto topk_kernel() {
    return topk_rows_kernel<kTopkThreads, kTopkVpt, KMAX, MAXC, kTopkCap, kTopkGroups, kTopkFcap,
                            PLAIN>;
}
template <bool PLAIN>
static auto topk_kernel_many() {
    return topk_rows_kernel<kTopkThreadsMany, kTopkVpt, kTopkKmaxSmall, 1, kTopkCap,
                            kTopkGroupsMany, kTopkFcap, PLAIN>;
}

os_status plan_topk(int64_t rows, int64_t cols, int K, os_plan* p) {
    const DeviceInfo* dev = device_info();
    if (!dev) return OS_ERR_CUDA;
    const bool large = K > kTopkKmaxSmall;
    if (!large) {
        const int many_sm = blocks_per_sm(topk_kernel_many<false>(), kTopkThreadsMany, kTopkDynBytesMany);
        const int64_t many_resident = int64_t(dev->sms) * many_sm;
        if (many_sm > 0 && rows >= many_resident && cols <= kTopkManyMaxCols) {
            os_plan q = {};
            q.path = OS_PATH_STREAM;
            q.threads = kTopkThreadsMany;
            q.vectors_per_thread = kTopkVpt;
            q.cluster = 1;
            q.grid = min64(many_resident, kMaxClustersPerLaunch);
            *p = q;
            return OS_OK;
        }
    }
    const int per_sm = large
        ? blocks_per_sm(topk_kernel<kTopkKmaxLarge, kTopkClusterLarge, false>(), kTopkThreads, kTopkDynBytes)
        : blocks_per_sm(topk_kernel<kTopkKmaxSmall, kTopkClusterSmall, false>(), kTopkThreads, kTopkDynBytes);
    if (per_sm <= 0) return OS_ERR_CUDA;
    const int64_t resident = int64_t(dev->sms) * per_sm;
    const int64_t blocks = (cols + 3) / 4 + 1;  // upper bound over the 4 possible row offsets
    const int64_t chunks = ceil_div(blocks, int64_t(kTopkThreads) * kTopkVpt);
    const int64_t max_cluster = large ? kTopkClusterLarge : kTopkClusterSmall;
    int64_t S = rows >= resident ? 1 : resident / rows;
    if (S > max_cluster) S = max_cluster;
    if (S > chunks) S = chunks;
    if (S < 1) S = 1;
    int64_t clusters = resident / S;
    if (clusters > rows) clusters = rows;
    if (clusters > kMaxClustersPerLaunch) clusters = kMaxClustersPerLaunch;
    os_plan q = {};
    q.path = OS_PATH_STREAM;
    q.threads = kTopkThreads;
    q.vectors_per_thread = kTopkVpt;
    q.cluster = static_cast<int32_t>(S);
    q.lanes_per_row = 0;
    q.stages = 0;
    q.grid = clusters * S;
    *p = q;
    return OS_OK;
}

cudaError_t launch_topk(const os_plan& p, const float* x, float* vals, int32_t* idx,
                        int64_t rows, int cols, int K, bool plain, const KernelCtl& ctl,
                        cudaStream_t stream) {
    const bool large = K > kTopkKmaxSmall;
    if (p.threads == kTopkThreadsMany) {
        auto k = plain ? topk_kernel_many<true>() : topk_kernel_many<false>();
        if (!prepare_kernel(k, 1, kTopkDynBytesMany)) return cudaErrorInvalidValue;
        return launch_kernel(k, p.grid, p.threads, 1, kTopkDynBytesMany, stream, x, vals,
                             reinterpret_cast<int*>(idx), rows, cols, K, 1, ctl);
    }
    auto k = large ? (plain ? topk_kernel<kTopkKmaxLarge, kTopkClusterLarge, true>()
                            : topk_kernel<kTopkKmaxLarge, kTopkClusterLarge, false>())
                   : (plain ? topk_kernel<kTopkKmaxSmall, kTopkClusterSmall, true>()
                            : topk_kernel<kTopkKmaxSmall, kTopkClusterSmall, false>());
    if (!prepare_kernel(k, p.cluster, kTopkDynBytes)) return cudaErrorInvalidValue;
    return launch_kernel(k, p.grid, p.threads, p.cluster, kTopkDynBytes, stream, x, vals,
                         reinterpret_cast<int*>(idx), rows, cols, K, p.cluster, ctl);
}

}  // namespace os
