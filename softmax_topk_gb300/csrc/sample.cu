// Top-K sampling after the fused pass: one column per row drawn from the K
// selected entries with probability proportional to their values.
//
// The draw is the smallest k with p_0 + ... + p_k > u (p_0 + ... + p_{K-1}),
// the partial sums rounded to fp32 after every addition in index order (one
// thread per row, explicit round-to-nearest operations that the compiler may
// not contract), so the result depends only on the values and u, not on how a
// parallel reduction happens to associate them.
#include "host_common.h"
#include "internal.h"

namespace os {

namespace {

__global__ void topk_sample_kernel(const float* __restrict__ vals, const int* __restrict__ idx,
                                   const float* __restrict__ u, int* __restrict__ out,
                                   int64_t rows, int K) {
    for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
         r += int64_t(gridDim.x) * blockDim.x) {
        const float* p = vals + r * K;
        float total = 0.f;
        for (int k = 0; k < K; ++k) total = __fadd_rn(total, p[k]);
        const float target = __fmul_rn(u[r], total);
        int pick = K - 1;  // u >= 1 falls back to the last entry
        float run = 0.f;
        for (int k = 0; k < K; ++k) {
            run = __fadd_rn(run, p[k]);
            if (run > target) {
                pick = k;
                break;
            }
        }
        out[r] = idx[r * K + pick];
    }
}

}  // namespace

cudaError_t launch_topk_sample(const float* vals, const int32_t* idx, const float* u, int32_t* out,
                               int64_t rows, int K, cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    constexpr int T = 256;
    const int64_t grid = min64(ceil_div(rows, T), int64_t(dev->sms) * 8);
    return launch_kernel(topk_sample_kernel, grid, T, 1, 0, stream, vals,
                         reinterpret_cast<const int*>(idx), u, reinterpret_cast<int*>(out), rows,
                         K);
}

}  // namespace os
