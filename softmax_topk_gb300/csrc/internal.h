// internal.h -- declarations shared between the C-ABI layer (api.cu) and the
// per-dtype translation units that hold the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/os_softmax.h"
#include "ctl.h"

namespace os {

#define OS_DECLARE_SOFTMAX_PAIR(NAME)                                                          \
    os_status plan_softmax_##NAME(int64_t rows, int64_t cols, os_path path, bool aligned,      \
                                  os_plan* p);                                                 \
    cudaError_t launch_softmax_##NAME(const os_plan& p, const void* x, void* y, int64_t rows,  \
                                      int cols, bool aligned, int64_t period, int64_t offset,  \
                                      const KernelCtl& ctl, cudaStream_t stream);

OS_DECLARE_SOFTMAX_PAIR(f32_f32)
OS_DECLARE_SOFTMAX_PAIR(bf16_bf16)
OS_DECLARE_SOFTMAX_PAIR(f32_bf16)
OS_DECLARE_SOFTMAX_PAIR(bf16_f32)

os_status plan_topk(int64_t rows, int64_t cols, int K, os_plan* p);
// plain: TopK of x itself (vals = the selected x) instead of softmax + TopK
cudaError_t launch_topk(const os_plan& p, const float* x, float* vals, int32_t* idx,
                        int64_t rows, int cols, int K, bool plain, const KernelCtl& ctl,
                        cudaStream_t stream);

cudaError_t launch_exp(const float* z, float* out, int64_t n, cudaStream_t stream);
// degree 5: the fp32 results' exponential; 3: the bf16 results'
cudaError_t launch_exp_pairs(const float* z, float* out, int64_t n, int degree,
                             cudaStream_t stream);

// one column per row drawn from its K (value, index) pairs, u[r] in [0, 1)
cudaError_t launch_topk_sample(const float* vals, const int32_t* idx, const float* u, int32_t* out,
                               int64_t rows, int K, cudaStream_t stream);

// attention forward over bh slices of [n][d] bf16 (d = 64 or 128): o bf16,
// lse fp32 (may be NULL); scale > 0
cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t bh, int n, int d, float scale, bool causal,
                             const KernelCtl& ctl, cudaStream_t stream);

// (m, d, lse) of every row; any output may be NULL
cudaError_t launch_stats(const void* x, os_dtype in, float* m, float* d, float* lse, int64_t rows,
                         int cols, bool aligned, cudaStream_t stream);

}  // namespace os
