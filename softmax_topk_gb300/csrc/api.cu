// api.cu -- the C ABI declared in include/os_softmax.h: argument checks, kernel
// choice per dtype pair, launch on the caller's stream.  No allocation, no
// synchronisation, no host fallback.
#include <cstdint>

#include "host_common.h"
#include "internal.h"

namespace {

using PlanFn = os_status (*)(int64_t, int64_t, os_path, os_plan*);
using LaunchFn = cudaError_t (*)(const os_plan&, const void*, void*, int64_t, int, bool,
                                 cudaStream_t);

struct Pair {
    PlanFn plan;
    LaunchFn launch;
};

// [in_dtype][out_dtype]
const Pair kPairs[2][2] = {
    {{os::plan_softmax_f32_f32, os::launch_softmax_f32_f32},
     {os::plan_softmax_f32_bf16, os::launch_softmax_f32_bf16}},
    {{os::plan_softmax_bf16_f32, os::launch_softmax_bf16_f32},
     {os::plan_softmax_bf16_bf16, os::launch_softmax_bf16_bf16}},
};

bool valid_dtype(int t) { return t == OS_F32 || t == OS_BF16; }
int64_t elem_bytes(os_dtype t) { return t == OS_F32 ? 4 : 2; }
int elems_per_vector(os_dtype t) { return t == OS_F32 ? 4 : 8; }

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + uintptr_t(nb) && pb < pa + uintptr_t(na);
}

// rows >= 0, 1 <= cols <= 2^31-1, and rows*cols*8 representable.
bool shape_ok(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 1 || cols > INT32_MAX) return false;
    return rows <= INT64_MAX / 8 / cols;
}

os_status softmax_checks(int64_t rows, int64_t cols, os_dtype in, os_dtype out, os_path path) {
    if (!valid_dtype(in) || !valid_dtype(out)) return OS_ERR_DTYPE;
    if (!shape_ok(rows, cols)) return OS_ERR_SHAPE;
    if (path < OS_PATH_AUTO || path > OS_PATH_STREAM) return OS_ERR_PATH;
    return OS_OK;
}

os_status topk_checks(int64_t rows, int64_t cols, int32_t K) {
    if (!shape_ok(rows, cols)) return OS_ERR_SHAPE;
    if (K < 1 || K > 64 || int64_t(K) > cols) return OS_ERR_K;
    return OS_OK;
}

}  // namespace

extern "C" {

const char* os_status_string(os_status s) {
    switch (s) {
        case OS_OK: return "OS_OK";
        case OS_ERR_NULL: return "OS_ERR_NULL: a required pointer is NULL";
        case OS_ERR_SHAPE: return "OS_ERR_SHAPE: rows < 0 or cols outside [1, 2^31-1]";
        case OS_ERR_DTYPE: return "OS_ERR_DTYPE: unknown dtype";
        case OS_ERR_K: return "OS_ERR_K: K outside [1, min(cols, 64)]";
        case OS_ERR_ALIAS: return "OS_ERR_ALIAS: an output overlaps an input or another output";
        case OS_ERR_CUDA: return "OS_ERR_CUDA: the CUDA runtime reported an error";
        case OS_ERR_TIMEOUT: return "OS_ERR_TIMEOUT: a device-side bounded wait gave up";
        case OS_ERR_PATH: return "OS_ERR_PATH: the kernel family cannot run this shape";
        case OS_ERR_ALIGN: return "OS_ERR_ALIGN: pointer not aligned to its element size";
    }
    return "unknown os_status";
}

os_status os_softmax_plan(int64_t rows, int64_t cols, os_dtype in, os_dtype out, os_path path,
                          os_plan* plan) {
    const os_status st = softmax_checks(rows, cols, in, out, path);
    if (st != OS_OK) return st;
    if (!plan) return OS_ERR_NULL;
    return kPairs[in][out].plan(rows, cols, path, plan);
}

os_status os_softmax_fwd_path(const void* x, void* y, int64_t rows, int64_t cols, os_dtype in,
                              os_dtype out, os_path path, os_stream_t stream) {
    os_status st = softmax_checks(rows, cols, in, out, path);
    if (st != OS_OK) return st;
    if (rows == 0) return OS_OK;
    if (!x || !y) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) % elem_bytes(in) ||
        reinterpret_cast<uintptr_t>(y) % elem_bytes(out))
        return OS_ERR_ALIGN;
    if (overlaps(x, rows * cols * elem_bytes(in), y, rows * cols * elem_bytes(out)))
        return OS_ERR_ALIAS;
    os_plan plan;
    st = kPairs[in][out].plan(rows, cols, path, &plan);
    if (st != OS_OK) return st;
    const bool aligned = cols % elems_per_vector(in) == 0 &&
                         reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(y) % 16 == 0;
    const cudaError_t e = kPairs[in][out].launch(plan, x, y, rows, static_cast<int>(cols), aligned,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

os_status os_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, os_dtype in,
                         os_dtype out, os_stream_t stream) {
    return os_softmax_fwd_path(x, y, rows, cols, in, out, OS_PATH_AUTO, stream);
}

os_status os_topk_plan(int64_t rows, int64_t cols, int32_t K, os_plan* plan) {
    const os_status st = topk_checks(rows, cols, K);
    if (st != OS_OK) return st;
    if (!plan) return OS_ERR_NULL;
    return os::plan_topk(rows, cols, K, plan);
}

os_status os_softmax_topk(const float* x, float* vals, int32_t* idx, int64_t rows, int64_t cols,
                          int32_t K, os_stream_t stream) {
    os_status st = topk_checks(rows, cols, K);
    if (st != OS_OK) return st;
    if (rows == 0) return OS_OK;
    if (!x || !vals || !idx) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(vals) % 4 ||
        reinterpret_cast<uintptr_t>(idx) % 4)
        return OS_ERR_ALIGN;
    const int64_t xb = rows * cols * 4, ob = rows * int64_t(K) * 4;
    if (overlaps(x, xb, vals, ob) || overlaps(x, xb, idx, ob) || overlaps(vals, ob, idx, ob))
        return OS_ERR_ALIAS;
    os_plan plan;
    st = os::plan_topk(rows, cols, K, &plan);
    if (st != OS_OK) return st;
    const cudaError_t e = os::launch_topk(plan, x, vals, idx, rows, static_cast<int>(cols), K,
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

os_status os_exp_f32(const float* z, float* out, int64_t n, os_stream_t stream) {
    if (n < 0) return OS_ERR_SHAPE;
    if (n == 0) return OS_OK;
    if (!z || !out) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(z) % 4 || reinterpret_cast<uintptr_t>(out) % 4)
        return OS_ERR_ALIGN;
    const cudaError_t e = os::launch_exp(z, out, n, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

}  // extern "C"
