// topk_kernel.cuh -- fused softmax + TopK: one read of x, K probabilities out.
//
// "Online normalizer calculation for softmax" (notes), section 4, fuses the
// online normalizer with TopK: a single loop keeps (m, d) and the K best logits
// u with their indices p, and only the winners are turned into probabilities
// v_i = e^(u_i - m_V) / d_V at the end.  Selecting on logits is exact because
// softmax is monotone.  The notes keep K+1 sorted slots and insert by one
// bubble pass per element; this kernel keeps the same invariant (a sorted list
// of the K best seen so far, per CTA) but fills it a tile at a time:
//
//   1. a cluster of CLUSTER CTAs owns a row; CTA `rank` owns a contiguous
//      segment of it and loads a tile of THREADS x VPT 16-byte vectors into
//      registers (one HBM read of every element), then each thread folds its
//      elements into its running (m, d): the tile maximum of its elements, then
//      their sum of e^(x - max) (chunked update, one rescale per tile);
//   2. threshold: each warp sorts its 32 thread maxima (bitonic network over
//      shuffles).  The smallest of the warps' j*-th values (j* = ceil(K /
//      warps) - 1) has at least K elements of the tile at or above it, so no
//      element below it can be in the top K.  The running list's K-th value
//      is a second such bound; the larger one is used;
//   3. elements at or above the threshold are appended to a shared-memory
//      candidate buffer (about K + K ln(n/K) of them for random data);
//   4. the candidates and the running list are sorted together (bitonic
//      network over the CTA on 64-bit keys: order-preserving value bits, then
//      the inverted column) and the first K become the new running list.  When
//      the buffer would overflow (heavy ties), an exact fallback bisects the
//      value keys, then the column keys of the ties, to admit exactly the K
//      best elements of the tile;
//   5. every CTA pushes its (m, d) state and sorted list into CTA 0 of the
//      cluster with st.async (completing CTA 0's barrier); CTA 0 ranks the
//      lists against each other (binary search per list), folds the states
//      with (+), and writes v = e^(u - m)/d and the indices, best first.
//
// Order: larger logit first; equal logits, lower column index first.
//
// Rows only need 4-byte alignment: vectors are taken in the 16-byte-aligned
// frame of each row; the partial first and last vectors are read element-wise.
#pragma once

#include <climits>

#include "ops.cuh"
#include "softmax_kernels.cuh"

namespace os {

// Order-preserving map float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// 64-bit sort key: value first, then lower column first.  0 = empty slot
// (below every real element: order_key(-inf) is 0x007fffff).
__device__ __forceinline__ uint64_t cand_key(float v, int j) {
    return (uint64_t(order_key(v)) << 32) | uint64_t(~uint32_t(j));
}
__device__ __forceinline__ float cand_value(uint64_t k) { return key_value(uint32_t(k >> 32)); }
__device__ __forceinline__ int cand_col(uint64_t k) { return int(~uint32_t(k)); }

// Sort v descending across the 32 lanes of a warp.
__device__ __forceinline__ float warp_sort_desc(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(kFullMask, v, stride);
            const bool keep_larger = ((lane & stride) == 0) == ((lane & size) == 0);
            v = keep_larger ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return v;
}

// Number of keys of the descending list L[0..K) above key c (they form a prefix).
__device__ __forceinline__ int count_above(const uint64_t* L, int K, uint64_t c) {
    int lo = 0, hi = K;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (L[mid] > c) lo = mid + 1; else hi = mid;
    }
    return lo;
}

template <int THREADS>
__device__ __forceinline__ int block_sum(int v, int* scratch) {
    v = __reduce_add_sync(kFullMask, v);
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    int total = 0;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) total += scratch[w];
    __syncthreads();
    return total;
}

// Bitonic sort (descending) of keys[0..P), P a power of two <= 2 * THREADS.
template <int THREADS>
__device__ __forceinline__ void block_sort_desc(uint64_t* keys, int P) {
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P / 2; i += THREADS) {
                const int lo = 2 * stride * (i / stride) + (i % stride);
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t a = keys[lo], b = keys[hi];
                if ((a < b) == desc) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

template <int THREADS, int CLUSTER, int KMAX, int CAP>
struct TopkSmem {
    uint64_t xbar[2];
    float2 warp_state[THREADS / 32];
    float warp_thr[THREADS / 32];
    int scratch[THREADS / 32];
    int ncand;
    uint64_t keys[2 * THREADS];  // sort buffer: candidates, then the running list
    uint64_t run[KMAX];
    float2 xstate[2][CLUSTER];
    uint64_t xlist[2][CLUSTER][KMAX];
};

// Exact fallback when too many elements tie at or above the threshold: the
// `need` = min(K, valid) best elements of the tile (same tile geometry as the
// kernel, re-read from memory; rare, so it stays out of the hot path's
// registers) found by bisection, first on the value key, then on the
// inverted column among the ties at the K-th value.  Writes their keys to
// keys[0..need) and returns need.  Every thread of the CTA must call it.
template <int THREADS, int VPT>
__device__ __noinline__ int exact_tile_select(const float* xr, const float* frame, int s, int cols,
                                              int tb, int q_end, int K, uint64_t* keys, int* ncand,
                                              int* scratch) {
    constexpr int EPT = VPT * 4;
    const int tid = threadIdx.x;
    auto col_of = [&](int i) { return 4 * (tb + (i >> 2) * THREADS + tid) - s + (i & 3); };
    auto valid = [&](int i) {
        const int q = tb + (i >> 2) * THREADS + tid;
        const int j = 4 * q - s + (i & 3);
        return q < q_end && j >= 0 && j < cols;
    };
    auto value = [&](int i) { return valid(i) ? xr[col_of(i)] : kNegInf; };
    (void)frame;
    int nvalid = 0;
    for (int i = 0; i < EPT; ++i) nvalid += valid(i);
    const int need = min(K, block_sum<THREADS>(nvalid, scratch));
    uint32_t t = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t probe = t | (1u << bit);
        int c = 0;
        for (int i = 0; i < EPT; ++i) c += valid(i) && order_key(value(i)) >= probe;
        if (block_sum<THREADS>(c, scratch) >= need) t = probe;
    }
    int above = 0;
    for (int i = 0; i < EPT; ++i) above += valid(i) && order_key(value(i)) > t;
    above = block_sum<THREADS>(above, scratch);
    uint32_t u = 0;  // among ties at t, the (need - above) lowest columns: largest inverted column
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t probe = u | (1u << bit);
        int c = 0;
        for (int i = 0; i < EPT; ++i)
            c += valid(i) && order_key(value(i)) == t && ~uint32_t(col_of(i)) >= probe;
        if (block_sum<THREADS>(c, scratch) >= need - above) u = probe;
    }
    if (tid == 0) *ncand = 0;
    __syncthreads();
    for (int i = 0; i < EPT; ++i) {
        if (!valid(i)) continue;
        const float v = value(i);
        const uint32_t kv = order_key(v);
        if (kv > t || (kv == t && ~uint32_t(col_of(i)) >= u))
            keys[atomicAdd(ncand, 1)] = cand_key(v, col_of(i));
    }
    __syncthreads();
    if (tid == 0) *ncand = 0;
    return need;
}

template <int THREADS, int VPT, int CLUSTER, int KMAX, int CAP>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2)
topk_rows_kernel(const float* __restrict__ x, float* __restrict__ vals, int* __restrict__ idx,
                 int64_t rows, int cols, int K, KernelCtl ctl) {
    constexpr int NW = THREADS / 32, EPT = VPT * 4, TILE = THREADS * VPT;
    static_assert(CAP + KMAX <= 2 * THREADS, "sort buffer holds candidates and the list");
    __shared__ __align__(16) TopkSmem<THREADS, CLUSTER, KMAX, CAP> sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int jstar = min((K + NW - 1) / NW - 1, 31);

    if (tid == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        mbar_init_fence();
        sm.ncand = 0;
    }
    if (CLUSTER > 1) cluster_sync(); else __syncthreads();

    int parity = 0;
    int64_t local = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1, ++local) {
        // a second row of this cluster reuses CTA 0's exchange slots: keep lockstep
        if (CLUSTER > 1 && local > 0) cluster_sync();
        const float* xr = x + row * int64_t(cols);
        const int s = int((reinterpret_cast<uintptr_t>(xr) >> 2) & 3);  // row start inside its vector
        const float* frame = xr - s;                                    // 16-byte aligned
        const int nvf = (cols + s + 3) / 4;
        const int per_cta = (nvf + CLUSTER - 1) / CLUSTER;
        const int q_begin = int(rank) * per_cta;
        const int q_end = min(q_begin + per_cta, nvf);
        int nrun = 0;  // entries of the running list
        float m = kNegInf, d = 0.f;

        for (int tb = q_begin; tb < q_end; tb += TILE) {
            // ---- 1. load the tile; element l of vector q is column 4q - s + l
            float v[EPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int q = tb + k * THREADS + tid;
                const int j0 = 4 * q - s;
                if (q < q_end && j0 >= 0 && j0 + 4 <= cols) {
                    const uint4 w = ld_stream_v4(frame + 4 * q);
                    v[4 * k] = __uint_as_float(w.x);
                    v[4 * k + 1] = __uint_as_float(w.y);
                    v[4 * k + 2] = __uint_as_float(w.z);
                    v[4 * k + 3] = __uint_as_float(w.w);
                } else {
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const int j = j0 + l;
                        v[4 * k + l] = (q < q_end && j >= 0 && j < cols) ? xr[j] : kNegInf;
                    }
                }
            }
            auto col_of = [&](int i) { return 4 * (tb + (i >> 2) * THREADS + tid) - s + (i & 3); };
            auto valid = [&](int i) {  // column inside the row and the CTA's segment
                const int q = tb + (i >> 2) * THREADS + tid;
                const int j = 4 * q - s + (i & 3);
                return q < q_end && j >= 0 && j < cols;
            };
            const float tmax = max_of<EPT>(v);
            {
                const float tsum = exp_sum<EPT>(v, tmax);
                const float m_new = fmaxf(m, tmax);
                d = d * rescale(m, m_new) + tsum * rescale(tmax, m_new);
                m = m_new;
            }

            // ---- 2. threshold
            const float sorted = warp_sort_desc(tmax);
            if (lane == jstar) sm.warp_thr[warp] = sorted;
            __syncthreads();
            float T = sm.warp_thr[0];
#pragma unroll
            for (int w = 1; w < NW; ++w) T = fminf(T, sm.warp_thr[w]);
            if (nrun >= K) T = fmaxf(T, cand_value(sm.run[K - 1]));

            // ---- 3. candidates at or above T
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (max3(v[4 * k], v[4 * k + 1], fmaxf(v[4 * k + 2], v[4 * k + 3])) >= T) {
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const int i = 4 * k + l;
                        if (v[i] >= T && valid(i)) {
                            const int pos = atomicAdd(&sm.ncand, 1);
                            if (pos < CAP) sm.keys[pos] = cand_key(v[i], col_of(i));
                        }
                    }
                }
            }
            __syncthreads();
            int n = sm.ncand;
            __syncthreads();
            if (tid == 0) sm.ncand = 0;

            if (n > CAP) {
                n = exact_tile_select<THREADS, VPT>(xr, frame, s, cols, tb, q_end, K, sm.keys,
                                                    &sm.ncand, sm.scratch);
            }

            // ---- 4. running list := first K of sort(candidates U list)
            {
                const int used = n + nrun;
                int P = 32;
                while (P < used) P <<= 1;
                for (int i = tid; i < nrun; i += THREADS) sm.keys[n + i] = sm.run[i];
                for (int i = used + tid; i < P; i += THREADS) sm.keys[i] = 0;
                __syncthreads();
                block_sort_desc<THREADS>(sm.keys, P);
                nrun = min(used, K);
                for (int i = tid; i < K; i += THREADS) sm.run[i] = i < nrun ? sm.keys[i] : 0;
                __syncthreads();
            }
        }

        // ---- 5. CTA state and list pushed into CTA 0
        {
            float mm = m, dd = d;
            group_merge<32>(mm, dd);
            if (lane == 0) sm.warp_state[warp] = make_float2(mm, dd);
            __syncthreads();
            if (CLUSTER == 1) {
                if (warp == 0) {
                    float2 st = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
                    group_merge<32>(st.x, st.y);
                    if (lane == 0) sm.xstate[parity][0] = st;
                }
                for (int i = tid; i < K; i += THREADS) sm.xlist[parity][0][i] = sm.run[i];
                __syncthreads();
            } else {
                const uint32_t bar0 = map_to_rank(&sm.xbar[parity], 0);
                if (rank == 0 && tid == 0)
                    mbar_arrive_expect_tx(&sm.xbar[parity], CLUSTER * (K + 1) * 8);
                if (warp == 0) {
                    float2 st = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
                    group_merge<32>(st.x, st.y);
                    if (lane == 0)
                        st_async_b64(map_to_rank(&sm.xstate[parity][rank], 0),
                                     __float_as_uint(st.x), __float_as_uint(st.y), bar0);
                }
                for (int i = tid; i < K; i += THREADS) {
                    const uint64_t key = sm.run[i];
                    st_async_b64(map_to_rank(&sm.xlist[parity][rank][i], 0), uint32_t(key),
                                 uint32_t(key >> 32), bar0);
                }
                if (rank == 0) {
                    if (tid == 0) mbar_wait_bounded(&sm.xbar[parity], uint32_t(local >> 1) & 1u, ctl);
                    __syncthreads();
                }
            }
        }

        if (rank == 0) {
            float M = kNegInf;
#pragma unroll
            for (int c = 0; c < CLUSTER; ++c) M = fmaxf(M, sm.xstate[parity][c].x);
            float D = 0.f;
#pragma unroll
            for (int c = 0; c < CLUSTER; ++c)
                D += sm.xstate[parity][c].y * rescale(sm.xstate[parity][c].x, M);
            const float inv_d = 1.0f / D;
            for (int i = tid; i < CLUSTER * K; i += THREADS) {
                const int a = i / K, p = i - a * K;
                const uint64_t key = sm.xlist[parity][a][p];
                if (key == 0) continue;
                int r = p;
#pragma unroll
                for (int b = 0; b < CLUSTER; ++b)
                    if (b != a) r += count_above(sm.xlist[parity][b], K, key);
                if (r < K) {
                    vals[row * K + r] = exp1(cand_value(key) - M) * inv_d;
                    idx[row * K + r] = cand_col(key);
                }
            }
        }
    }
    if (CLUSTER > 1) cluster_sync();  // CTA 0's slots stay valid until every push has landed
}

}  // namespace os
