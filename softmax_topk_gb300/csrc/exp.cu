// Elementwise e^z with the library's own fp32 exponentials (os_exp_f32,
// os_exp_pairs_f32).
#include "host_common.h"
#include "internal.h"
#include "kernels/ops.cuh"

namespace os {

__global__ void exp_kernel(const float* z, float* out, int64_t n) {  // z and out may alias
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = exp1(z[i]);
}

cudaError_t launch_exp(const float* z, float* out, int64_t n, cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return cudaErrorNoDevice;
    const int64_t grid = min64(ceil_div(n, 256), int64_t(dev->sms) * 8);
    return launch_kernel(exp_kernel, grid, 256, 1, 0, stream, z, out, n);
}

// The streaming kernel's per-element exponential (DEG 5: fp32 results; 3:
// bf16 results, before rounding), two values per thread step (an odd tail
// pairs its last value with 0).
template <int DEG>
__global__ void exp_pairs_kernel(const float* z, float* out, int64_t n) {  // z and out may alias
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; 2 * p < n; p += stride) {
        const int64_t i = 2 * p;
        const bool two = i + 1 < n;
        const float2 r = mul2(exp_biased_pair<DEG>(make_float2(z[i], two ? z[i + 1] : 0.0f)),
                              splat2(expc::kUnbias));
        out[i] = r.x;
        if (two) out[i + 1] = r.y;
    }
}

cudaError_t launch_exp_pairs(const float* z, float* out, int64_t n, int degree,
                             cudaStream_t stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return cudaErrorNoDevice;
    const int64_t grid = min64(ceil_div(ceil_div(n, 2), 256), int64_t(dev->sms) * 8);
    return degree == 3 ? launch_kernel(exp_pairs_kernel<3>, grid, 256, 1, 0, stream, z, out, n)
                       : launch_kernel(exp_pairs_kernel<5>, grid, 256, 1, 0, stream, z, out, n);
}

}  // namespace os
