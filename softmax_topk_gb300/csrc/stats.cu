// Row statistics (m, d, log-sum-exp): kernel choice and launch.
//
// Rows of up to 32 x U 16-byte vectors (1024 fp32 / bf16 elements with U = 8
// fp32 or 4 bf16 vectors per thread) take one warp per row, eight rows per
// 256-thread CTA; longer rows one 512-thread CTA per row.  Both grids are
// persistent (resident CTAs at most).
#include "host_common.h"
#include "internal.h"
#include "kernels/softmax_kernels.cuh"

namespace os {

namespace {

template <typename TI>
cudaError_t launch_stats_t(const TI* x, float* m, float* d, float* lse, int64_t rows, int cols,
                           bool aligned, cudaStream_t stream) {
    constexpr int EPV = VecTraits<TI>::EPV;
    constexpr int U = sizeof(TI) == 4 ? 8 : 4;
    const DeviceInfo* dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const int64_t nv = ceil_div(cols, EPV);
    if (nv <= 32 * U) {
        constexpr int T = 256;
        auto k = aligned ? stats_rows_kernel<TI, T, 32, U, true> : stats_rows_kernel<TI, T, 32, U, false>;
        const int occ = blocks_per_sm(k, T);
        const int64_t grid = min64(ceil_div(rows, T / 32), int64_t(dev->sms) * (occ > 0 ? occ : 1));
        return launch_kernel(k, grid, T, 1, 0, stream, x, m, d, lse, rows, cols);
    }
    constexpr int T = 512;
    auto k = aligned ? stats_rows_kernel<TI, T, T, U, true> : stats_rows_kernel<TI, T, T, U, false>;
    const int occ = blocks_per_sm(k, T);
    const int64_t grid = min64(rows, int64_t(dev->sms) * (occ > 0 ? occ : 1));
    return launch_kernel(k, grid, T, 1, 0, stream, x, m, d, lse, rows, cols);
}

}  // namespace

cudaError_t launch_stats(const void* x, os_dtype in, float* m, float* d, float* lse, int64_t rows,
                         int cols, bool aligned, cudaStream_t stream) {
    if (in == OS_F32)
        return launch_stats_t(static_cast<const float*>(x), m, d, lse, rows, cols, aligned, stream);
    return launch_stats_t(static_cast<const __nv_bfloat16*>(x), m, d, lse, rows, cols, aligned,
                          stream);
}

}  // namespace os
