// api.cu -- the C ABI declared in include/os_softmax.h: argument checks, kernel
// choice per dtype pair, launch on the caller's stream.  No allocation, no
// synchronisation, no host fallback.
#include <atomic>
#include <cstdint>

#include "host_common.h"
#include "internal.h"

// Device status word (one per device the library runs on): kernels OR in
// os::kErrWaitTimeout when a bounded wait gives up.  Read and cleared in one
// atomic exchange by os_device_status, whose result lands in the second word.
__device__ unsigned int os_device_status_word;
__device__ unsigned int os_device_status_taken;

// The status word's value at the moment it is cleared: a timeout recorded by a
// kernel on another stream lands either before the exchange (and is reported
// now) or after it (and is reported by the next call), never lost between a
// read and a separate clear.
__global__ void status_exchange_kernel() {
    os_device_status_taken = atomicExch(&os_device_status_word, 0u);
}

namespace {

std::atomic<unsigned long long> g_timeout_ns{1000000000ull};  // 1 s per wait
std::atomic<int> g_fault{0};

// Address of this device's status word (host code cannot use the symbol
// itself as a device pointer), looked up once per device.
unsigned int* status_word() {
    constexpr int kMaxDevices = 64;
    static unsigned int* cache[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, os_device_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = static_cast<unsigned int*>(p);
    }
    return cache[dev];
}

bool make_ctl(os::KernelCtl* ctl) {
    ctl->err = status_word();
    ctl->timeout_ns = g_timeout_ns.load();
    ctl->fault = g_fault.load();
    return ctl->err != nullptr;
}

using PlanFn = os_status (*)(int64_t, int64_t, os_path, bool, os_plan*);
using LaunchFn = cudaError_t (*)(const os_plan&, const void*, void*, int64_t, int, bool, int64_t,
                                 int64_t, const os::KernelCtl&, cudaStream_t);

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
    if (path < OS_PATH_AUTO || path > OS_PATH_STREAM_POLY) return OS_ERR_PATH;
    return OS_OK;
}

os_status topk_checks(int64_t rows, int64_t cols, int32_t K) {
    if (!shape_ok(rows, cols)) return OS_ERR_SHAPE;
    if (K < 1 || K > 256 || int64_t(K) > cols) return OS_ERR_K;
    return OS_OK;
}

// period > 0: causal mask; only the WARP and STREAM families take one, and AUTO
// picks between those two.
os_status softmax_entry(const void* x, void* y, int64_t rows, int64_t cols, os_dtype in,
                        os_dtype out, os_path path, int64_t period, int64_t offset,
                        os_stream_t stream) {
    os_status st = softmax_checks(rows, cols, in, out, path);
    if (st != OS_OK) return st;
    if (rows == 0) return OS_OK;
    if (!x || !y) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) % elem_bytes(in) ||
        reinterpret_cast<uintptr_t>(y) % elem_bytes(out))
        return OS_ERR_ALIGN;
    // exactly in place (y == x, one dtype) is allowed: every kernel family
    // reads each element of a row before the same thread or CTA writes it;
    // any other overlap is not
    const bool in_place = x == y && in == out;
    if (!in_place && overlaps(x, rows * cols * elem_bytes(in), y, rows * cols * elem_bytes(out)))
        return OS_ERR_ALIAS;
    const bool ptrs_aligned = reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                              reinterpret_cast<uintptr_t>(y) % 16 == 0;
    if (period > 0) {
        // the vector slots a row needs (one more when rows are not 16-byte
        // aligned whole vectors), as the plan counts them
        const int epv = elems_per_vector(in);
        const int64_t nv = (ptrs_aligned && cols % epv == 0) ? (cols + epv - 1) / epv
                                                             : (cols + 2 * epv - 2) / epv;
        if (path == OS_PATH_AUTO) path = nv <= 256 ? OS_PATH_WARP : OS_PATH_STREAM;
        if (path != OS_PATH_WARP && path != OS_PATH_STREAM && path != OS_PATH_STREAM_POLY)
            return OS_ERR_PATH;
    }
    os_plan plan;
    st = kPairs[in][out].plan(rows, cols, path, ptrs_aligned, &plan);
    if (st != OS_OK) return st;
    os::KernelCtl ctl;
    if (!make_ctl(&ctl)) return OS_ERR_CUDA;
    const bool aligned = ptrs_aligned && cols % elems_per_vector(in) == 0;
    const cudaError_t e = kPairs[in][out].launch(plan, x, y, rows, static_cast<int>(cols), aligned,
                                                 period, offset, ctl,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* os_status_string(os_status s) {
    switch (s) {
        case OS_OK: return "OS_OK";
        case OS_ERR_NULL: return "OS_ERR_NULL: a required pointer is NULL";
        case OS_ERR_SHAPE: return "OS_ERR_SHAPE: a size or head dimension outside its range";
        case OS_ERR_DTYPE: return "OS_ERR_DTYPE: unknown dtype";
        case OS_ERR_K: return "OS_ERR_K: K outside [1, min(cols, 256)]";
        case OS_ERR_ALIAS: return "OS_ERR_ALIAS: an output overlaps an input or another output";
        case OS_ERR_CUDA: return "OS_ERR_CUDA: the CUDA runtime reported an error";
        case OS_ERR_TIMEOUT: return "OS_ERR_TIMEOUT: a device-side bounded wait gave up";
        case OS_ERR_PATH: return "OS_ERR_PATH: the kernel family cannot run this shape";
        case OS_ERR_ALIGN: return "OS_ERR_ALIGN: pointer not aligned to its element size";
        case OS_ERR_VALUE: return "OS_ERR_VALUE: a scalar argument outside its range";
    }
    return "unknown os_status";
}

os_status os_softmax_plan(int64_t rows, int64_t cols, os_dtype in, os_dtype out, os_path path,
                          os_plan* plan) {
    const os_status st = softmax_checks(rows, cols, in, out, path);
    if (st != OS_OK) return st;
    if (!plan) return OS_ERR_NULL;
    return kPairs[in][out].plan(rows, cols, path, true, plan);
}

os_status os_softmax_fwd_path(const void* x, void* y, int64_t rows, int64_t cols, os_dtype in,
                              os_dtype out, os_path path, os_stream_t stream) {
    return softmax_entry(x, y, rows, cols, in, out, path, 0, 0, stream);
}

os_status os_softmax_causal_fwd(const void* x, void* y, int64_t rows, int64_t cols,
                                int64_t period, int64_t offset, os_dtype in, os_dtype out,
                                os_stream_t stream) {
    if (period < 1 || offset < 0) return OS_ERR_SHAPE;
    return softmax_entry(x, y, rows, cols, in, out, OS_PATH_AUTO, period, offset, stream);
}

os_status os_softmax_stats(const void* x, float* m, float* d, float* lse, int64_t rows,
                           int64_t cols, os_dtype in, os_stream_t stream) {
    if (!valid_dtype(in)) return OS_ERR_DTYPE;
    if (!shape_ok(rows, cols)) return OS_ERR_SHAPE;
    if (rows == 0) return OS_OK;
    if (!x || (!m && !d && !lse)) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) % elem_bytes(in) || reinterpret_cast<uintptr_t>(m) % 4 ||
        reinterpret_cast<uintptr_t>(d) % 4 || reinterpret_cast<uintptr_t>(lse) % 4)
        return OS_ERR_ALIGN;
    const int64_t xb = rows * cols * elem_bytes(in), ob = rows * 4;
    const float* outs[3] = {m, d, lse};
    for (int i = 0; i < 3; ++i) {
        if (!outs[i]) continue;
        if (overlaps(x, xb, outs[i], ob)) return OS_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (outs[j] && overlaps(outs[i], ob, outs[j], ob)) return OS_ERR_ALIAS;
    }
    const bool aligned = reinterpret_cast<uintptr_t>(x) % 16 == 0 && cols % elems_per_vector(in) == 0;
    if (!os::device_info()) return OS_ERR_CUDA;
    const cudaError_t e = os::launch_stats(x, in, m, d, lse, rows, static_cast<int>(cols), aligned,
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

static os_status topk_entry(const float* x, float* vals, int32_t* idx, int64_t rows, int64_t cols,
                     int32_t K, bool plain, os_stream_t stream) {
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
    os::KernelCtl ctl;
    if (!make_ctl(&ctl)) return OS_ERR_CUDA;
    const cudaError_t e = os::launch_topk(plan, x, vals, idx, rows, static_cast<int>(cols), K, plain,
                                          ctl, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

os_status os_softmax_topk(const float* x, float* vals, int32_t* idx, int64_t rows, int64_t cols,
                          int32_t K, os_stream_t stream) {
    return topk_entry(x, vals, idx, rows, cols, K, false, stream);
}

os_status os_topk(const float* x, float* vals, int32_t* idx, int64_t rows, int64_t cols, int32_t K,
                  os_stream_t stream) {
    return topk_entry(x, vals, idx, rows, cols, K, true, stream);
}

os_status os_topk_sample(const float* vals, const int32_t* idx, const float* u, int32_t* out,
                         int64_t rows, int32_t K, os_stream_t stream) {
    if (rows < 0) return OS_ERR_SHAPE;
    if (K < 1 || K > 256) return OS_ERR_K;
    if (rows > INT64_MAX / 8 / K) return OS_ERR_SHAPE;
    if (rows == 0) return OS_OK;
    if (!vals || !idx || !u || !out) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(vals) % 4 || reinterpret_cast<uintptr_t>(idx) % 4 ||
        reinterpret_cast<uintptr_t>(u) % 4 || reinterpret_cast<uintptr_t>(out) % 4)
        return OS_ERR_ALIGN;
    const int64_t kb = rows * int64_t(K) * 4, rb = rows * 4;
    if (overlaps(out, rb, vals, kb) || overlaps(out, rb, idx, kb) || overlaps(out, rb, u, rb))
        return OS_ERR_ALIAS;
    const cudaError_t e = os::launch_topk_sample(vals, idx, u, out, rows, K,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

os_status os_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t bh, int64_t n, int32_t head_dim, float scale, int32_t causal,
                           os_stream_t stream) {
    if (bh < 0 || n < 0 || n > INT32_MAX || (head_dim != 64 && head_dim != 128))
        return OS_ERR_SHAPE;
    if (!(scale > 0.f) || !(scale < INFINITY) || (causal != 0 && causal != 1)) return OS_ERR_VALUE;
    if (bh == 0 || n == 0) return OS_OK;
    const int64_t nq = (n + 127) / 128;
    if (bh > INT32_MAX / nq || bh > INT64_MAX / 2 / head_dim / n) return OS_ERR_SHAPE;
    if (!q || !k || !v || !o) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(k) % 16 ||
        reinterpret_cast<uintptr_t>(v) % 16 || reinterpret_cast<uintptr_t>(o) % 16 ||
        reinterpret_cast<uintptr_t>(lse) % 4)
        return OS_ERR_ALIGN;
    const int64_t tb = bh * n * head_dim * 2, lb = bh * n * 4;
    if (overlaps(o, tb, q, tb) || overlaps(o, tb, k, tb) || overlaps(o, tb, v, tb))
        return OS_ERR_ALIAS;
    if (lse && (overlaps(lse, lb, q, tb) || overlaps(lse, lb, k, tb) || overlaps(lse, lb, v, tb) ||
                overlaps(lse, lb, o, tb)))
        return OS_ERR_ALIAS;
    os::KernelCtl ctl;
    if (!make_ctl(&ctl)) return OS_ERR_CUDA;
    const cudaError_t e = os::launch_attention(q, k, v, o, lse, bh, static_cast<int>(n), head_dim,
                                               scale, causal != 0, ctl,
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

static os_status exp_pairs_entry(const float* z, float* out, int64_t n, int degree, os_stream_t stream) {
    if (n < 0) return OS_ERR_SHAPE;
    if (n == 0) return OS_OK;
    if (!z || !out) return OS_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(z) % 4 || reinterpret_cast<uintptr_t>(out) % 4)
        return OS_ERR_ALIGN;
    const cudaError_t e = os::launch_exp_pairs(z, out, n, degree,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OS_OK : OS_ERR_CUDA;
}

os_status os_exp_pairs_f32(const float* z, float* out, int64_t n, os_stream_t stream) {
    return exp_pairs_entry(z, out, n, 5, stream);
}

os_status os_exp_pairs_coarse_f32(const float* z, float* out, int64_t n, os_stream_t stream) {
    return exp_pairs_entry(z, out, n, 3, stream);
}

os_status os_device_status(os_stream_t stream) {
    if (!status_word()) return OS_ERR_CUDA;
    // one host caller at a time per process: the exchange's result word is shared
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    status_exchange_kernel<<<1, 1, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess) return OS_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, os_device_status_taken, sizeof(v), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return OS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return OS_ERR_CUDA;
    if (v == 0) return OS_OK;
    return (v & os::kErrWaitTimeout) ? OS_ERR_TIMEOUT : OS_ERR_CUDA;
}

os_status os_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 1000000ull || ns > 10000000000ull) return OS_ERR_SHAPE;
    g_timeout_ns.store(ns);
    return OS_OK;
}

os_status os_set_fault_injection(int32_t mode) {
    if (mode != 0 && mode != os::kFaultSkipFirstLoad) return OS_ERR_SHAPE;
    g_fault.store(mode);
    return OS_OK;
}

}  // extern "C"
