// Attention forward: tensor maps for Q, K, V and the launch.
//
// Persistent CTAs, one per SM, walk the 128-row query tiles of every (batch,
// head) slice.  Q, K and V are
// [bh][n][D] bf16, read through 3-D tensor maps (D, n, bh) with 128-byte
// swizzle and boxes of 64 x 128 x 1, so rows past n inside a slice are
// zero-filled by the copy engine and never read from the next slice.
#include <cuda.h>

#include <mutex>

#include "host_common.h"
#include "internal.h"
#include "kernels/attention_kernel.cuh"

namespace os {

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up through the runtime once.
EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool make_map(CUtensorMap* map, const void* base, int64_t bh, int n, int d) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(n), cuuint64_t(bh)};
    const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(n) * cuuint64_t(d) * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(attn::kBN), 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* o,
                     float* lse, int64_t bh, int n, float scale_log2, bool causal,
                     const KernelCtl& ctl, cudaStream_t stream) {
    auto k = attn::attention_fwd_kernel<D>;
    constexpr int smem = attn::Layout<D, attn::Stages<D>::value>::kDynBytes;
    if (!prepare_kernel(k, 1, smem)) return cudaErrorInvalidConfiguration;
    const DeviceInfo* dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    const int nq = (n + attn::kBM - 1) / attn::kBM;
    // work units: query tiles, or with the mask pairs of them (see work_unit);
    // one persistent CTA per SM (shared memory admits one) walks them
    const int64_t units = causal ? bh * ((nq + 1) / 2) : bh * nq;
    const int64_t grid = units < dev->sms ? units : dev->sms;
    return launch_kernel(k, grid, attn::kThreads, 1, smem, stream, mq, mk, mv,
                         static_cast<__nv_bfloat16*>(o), lse, n, nq, static_cast<int>(units),
                         scale_log2, causal ? 1 : 0, ctl);
}

}  // namespace

cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t bh, int n, int d, float scale, bool causal,
                             const KernelCtl& ctl, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, bh, n, d) || !make_map(&mk, k, bh, n, d) || !make_map(&mv, v, bh, n, d))
        return cudaErrorInvalidValue;
    const float scale_log2 = scale * 1.442695041f;
    if (d == 64) return launch_d<64>(mq, mk, mv, o, lse, bh, n, scale_log2, causal, ctl, stream);
    return launch_d<128>(mq, mk, mv, o, lse, bh, n, scale_log2, causal, ctl, stream);
}

}  // namespace os
