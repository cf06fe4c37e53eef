// topk_kernel.cuh -- fused softmax + TopK: one read of x, K probabilities out.
//
// "Online normalizer calculation for softmax" (notes), section 4, fuses the
// online normalizer with TopK: a single loop keeps (m, d) and the K best logits
// u with their indices p, and only the winners are turned into probabilities
// v_i = e^(u_i - m_V) / d_V at the end.  Selecting on logits is exact because
// softmax is monotone.  The notes keep K+1 sorted slots and insert by one
// bubble pass per element; this kernel keeps the same invariant (a sorted list
// of the K best seen so far, per CTA) but fills it in batches:
//
//   1. a cluster of CLUSTER CTAs owns a row; CTA `rank` stages its contiguous
//      segment (a tile of up to TILE elements at a time) in shared memory with
//      NCHUNK bulk copies, each on its own barrier.  As each chunk lands,
//      every thread folds its elements of the chunk into its running (m, d)
//      (chunk maximum, then the sum of e^(x - max): one rescale per chunk) and
//      into its maximum over the tile;
//   2. threshold: each warp sorts its 32 thread maxima (bitonic network over
//      shuffles).  The smallest of the warps' j*-th values (j* = ceil(K /
//      warps) - 1) has at least K elements of the tile at or above it, so no
//      element below it can be in the top K.  The running list's K-th value
//      is a second such bound; the larger one is used;
//   3. elements at or above the threshold are appended to a shared-memory
//      candidate buffer (about K + K ln(n/K) for random data);
//   4. the running list becomes the K best of (candidates U list), found by
//      ranking: rank(c) = number of entries that beat c, each count split over
//      the 32 lanes of a warp.  When the buffer would overflow (heavy ties at
//      the threshold), an exact fallback finds the K-th largest key of the
//      tile by bisection on the order-preserving bit pattern and admits the
//      ties at it in column order;
//   5. every CTA pushes its (m, d) state and sorted list into CTA 0 of the
//      cluster with st.async (completing CTA 0's barrier); CTA 0 ranks the
//      lists against each other (binary search per list), folds the states
//      with (+), and writes v = e^(u - m)/d and the indices, best first.
//
// Order ("beats"): larger logit first; equal logits, lower column index first.
// Index INT32_MAX marks an empty slot and never beats a real element.
//
// Rows only need 4-byte alignment: the bulk copies cover the 16-byte-aligned
// interior of a tile; its first and last few elements are read one by one.
#pragma once

#include <climits>

#include "ops.cuh"
#include "softmax_kernels.cuh"

namespace os {

struct Cand {
    float v;
    int j;
};

constexpr int kNoIndex = INT_MAX;

__device__ __forceinline__ bool beats(float v1, int j1, float v2, int j2) {
    return v1 > v2 || (v1 == v2 && j1 < j2);
}
__device__ __forceinline__ bool beats(const Cand& a, const Cand& b) { return beats(a.v, a.j, b.v, b.j); }

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

// Number of entries of the sorted list L[0..K) that beat c (they form a prefix).
__device__ __forceinline__ int count_beating(const Cand* L, int K, const Cand& c) {
    int lo = 0, hi = K;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (beats(L[mid], c)) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Order-preserving map float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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

template <int THREADS, int CLUSTER, int KMAX, int CAP, int NCHUNK>
struct TopkSmem {
    uint64_t chunk_bar[NCHUNK];
    uint64_t xbar[2];
    float2 warp_state[THREADS / 32];
    float warp_thr[THREADS / 32];
    int scratch[THREADS / 32];
    int ncand;
    int taken;
    int wait_flag[2];
    Cand cand[CAP];
    Cand run[2][KMAX];
    float2 xstate[2][CLUSTER];
    Cand xlist[2][CLUSTER][KMAX];
};

template <int THREADS, int CLUSTER, int TILE, int KMAX, int CAP, int NCHUNK>
__global__ void __launch_bounds__(THREADS)
topk_rows_kernel(const float* __restrict__ x, float* __restrict__ vals, int* __restrict__ idx,
                 int64_t rows, int cols, int K, KernelCtl ctl) {
    constexpr int NW = THREADS / 32;
    extern __shared__ __align__(128) float frame[];
    __shared__ __align__(8) TopkSmem<THREADS, CLUSTER, KMAX, CAP, NCHUNK> sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int jstar = min((K + NW - 1) / NW - 1, 31);
    const Cand pad{kNegInf, kNoIndex};
    const int seg = (cols + CLUSTER - 1) / CLUSTER;
    const int seg_begin = min(int(rank) * seg, cols);
    const int seg_end = min(seg_begin + seg, cols);

    if (tid == 0) {
        for (int c = 0; c < NCHUNK; ++c) mbar_init(&sm.chunk_bar[c], 1);
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        mbar_init_fence();
        sm.ncand = 0;
    }
    if (CLUSTER > 1) cluster_sync(); else __syncthreads();

    // Every thread keeps the phase parity of each chunk barrier (bit c of
    // `cpar`, flipped whenever chunk c of a tile is non-empty, which is the
    // same in all threads); thread 0 issues the copies.  After a wait gives up
    // a thread stops waiting and thread 0 stops issuing (outputs are garbage,
    // the status word says so); copies left in flight are waited for before exit.
    uint32_t tiles = 0, cpar = 0;
    bool failed = false;
    uint32_t pending = 0, pending_par = 0;  // thread 0: issued chunks not yet seen complete
    int parity = 0;
    int64_t local = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1, ++local) {
        // a second row of this cluster reuses CTA 0's exchange slots: keep lockstep
        if (CLUSTER > 1 && local > 0) cluster_sync();
        const float* xr = x + row * int64_t(cols);
        int cur = 0;
        if (tid < KMAX) sm.run[0][tid] = pad;
        float m = kNegInf, d = 0.f;

        for (int tb = seg_begin; tb < seg_end; tb += TILE, ++tiles) {
            const int len = min(TILE, seg_end - tb);
            // ---- 1a. stage the tile: bulk copies of the aligned interior, element loads at the ends
            const uintptr_t a = reinterpret_cast<uintptr_t>(xr + tb);
            const uintptr_t a_floor = a & ~uintptr_t(15), a_ceil = (a + 15) & ~uintptr_t(15);
            const uintptr_t a_end = a + uintptr_t(len) * 4, a_end_floor = a_end & ~uintptr_t(15);
            const int head = int(a - a_floor) / 4;  // frame index of element 0
            const bool bulk = a_end_floor > a_ceil;
            const int plain_head = bulk ? int(a_ceil - a) / 4 : len;
            const int tail_from = bulk ? int(a_end_floor - a) / 4 : len;
            const int q_bulk0 = int(a_ceil - a_floor) / 16;      // first vector of the bulk region
            const int q_bulk1 = bulk ? int(a_end_floor - a_floor) / 16 : q_bulk0;
            const int nq = (head + len + 3) / 4;
            const int qs_per_chunk = (q_bulk1 - q_bulk0 + NCHUNK - 1) / NCHUNK;
            if (tid == 0 && bulk && !failed &&
                !(ctl.fault == kFaultSkipFirstLoad && blockIdx.x == 0 && tiles == 0)) {
                for (int c = 0; c < NCHUNK; ++c) {
                    const int q0 = q_bulk0 + c * qs_per_chunk;
                    const int q1 = min(q0 + qs_per_chunk, q_bulk1);
                    if (q1 <= q0) continue;
                    const uint32_t bytes = uint32_t(q1 - q0) * 16;
                    mbar_arrive_expect_tx(&sm.chunk_bar[c], bytes);
                    bulk_g2s(frame + 4 * q0, reinterpret_cast<const void*>(a_floor + uintptr_t(q0) * 16),
                             bytes, &sm.chunk_bar[c]);
                    pending |= 1u << c;
                    pending_par = (pending_par & ~(1u << c)) | (cpar & (1u << c));
                }
            }
            if (tid < plain_head) frame[head + tid] = xr[tb + tid];
            if (tid >= 32 && tid - 32 < len - tail_from)
                frame[head + tail_from + tid - 32] = xr[tb + tail_from + tid - 32];

            // ---- 1b. per chunk: running (m, d) and the thread's maximum over the tile
            float tmax = kNegInf;
            for (int c = 0; c < NCHUNK; ++c) {
                const int q0 = q_bulk0 + c * qs_per_chunk;
                const int q1 = min(q0 + qs_per_chunk, q_bulk1);
                if (q1 <= q0) continue;
                if (!failed) {
                    failed = !cta_wait_bounded(&sm.chunk_bar[c], (cpar >> c) & 1u, ctl,
                                               sm.wait_flag, c & 1);
                    if (!failed && tid == 0) pending &= ~(1u << c);
                }
                cpar ^= 1u << c;
                float cmax = kNegInf;
                for (int q = q0 + tid; q < q1; q += THREADS) {
                    const float4 v = *reinterpret_cast<const float4*>(frame + 4 * q);
                    cmax = max3(cmax, fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                }
                float csum = 0.f;
                for (int q = q0 + tid; q < q1; q += THREADS) {
                    const float4 v = *reinterpret_cast<const float4*>(frame + 4 * q);
                    const float w[4] = {v.x, v.y, v.z, v.w};
                    csum += exp_sum<4>(w, cmax);
                }
                const float m_new = fmaxf(m, cmax);
                d = d * rescale(m, m_new) + csum * rescale(cmax, m_new);
                m = m_new;
                tmax = fmaxf(tmax, cmax);
            }
            __syncthreads();  // element-wise loads of the ends are visible
            // the partial vectors at the ends (at most two) and tiles too short for a bulk copy
            auto load4 = [&](int q, float* v) {
                const float4 w = *reinterpret_cast<const float4*>(frame + 4 * q);
                v[0] = w.x;
                v[1] = w.y;
                v[2] = w.z;
                v[3] = w.w;
                if (q < q_bulk0 || q >= q_bulk1) {
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const int e = 4 * q + l - head;
                        if (e < 0 || e >= len) v[l] = kNegInf;
                    }
                }
            };
            {
                const int nedge = q_bulk0 + (nq - q_bulk1);
                if (tid < nedge) {
                    const int q = tid < q_bulk0 ? tid : q_bulk1 + (tid - q_bulk0);
                    float v[4];
                    load4(q, v);
                    const float emax = max3(fmaxf(v[0], v[1]), v[2], v[3]);
                    const float m_new = fmaxf(m, emax);
                    d = d * rescale(m, m_new) + exp_sum<4>(v, m_new);
                    m = m_new;
                    tmax = fmaxf(tmax, emax);
                }
            }

            // ---- 2. threshold
            const float sorted = warp_sort_desc(tmax);
            if (lane == jstar) sm.warp_thr[warp] = sorted;
            __syncthreads();
            float T = sm.warp_thr[0];
#pragma unroll
            for (int w = 1; w < NW; ++w) T = fminf(T, sm.warp_thr[w]);
            T = fmaxf(T, sm.run[cur][K - 1].v);

            // ---- 3. candidates at or above T
            for (int q = tid; q < nq; q += THREADS) {
                float v[4];
                load4(q, v);
                if (fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])) >= T) {
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const int e = 4 * q + l - head;
                        if (v[l] >= T && e >= 0 && e < len) {
                            const int pos = atomicAdd(&sm.ncand, 1);
                            if (pos < CAP) sm.cand[pos] = Cand{v[l], tb + e};
                        }
                    }
                }
            }
            __syncthreads();
            int n = sm.ncand;
            __syncthreads();
            if (tid == 0) sm.ncand = 0;

            if (n > CAP) {
                // ---- 4b. exact fallback: K-th largest key of the tile by bisection
                const int need = min(K, len);
                uint32_t t = 0;
                for (int bit = 31; bit >= 0; --bit) {
                    const uint32_t probe = t | (1u << bit);
                    int c = 0;
                    for (int e = tid; e < len; e += THREADS) c += order_key(frame[head + e]) >= probe;
                    if (block_sum<THREADS>(c, sm.scratch) >= need) t = probe;
                }
                // strictly above t: fewer than `need`; then ties at t in column order
                if (tid == 0) {
                    sm.ncand = 0;
                    sm.taken = 0;
                }
                __syncthreads();
                for (int e = tid; e < len; e += THREADS) {
                    const float v = frame[head + e];
                    if (order_key(v) > t) sm.cand[atomicAdd(&sm.ncand, 1)] = Cand{v, tb + e};
                }
                __syncthreads();
                const int above = sm.ncand;
                for (int base = 0; base < len; base += THREADS) {
                    const int e = base + tid;
                    const bool tie = e < len && order_key(frame[head + e]) == t;
                    const unsigned ballot = __ballot_sync(kFullMask, tie);
                    if (lane == 0) sm.scratch[warp] = __popc(ballot);
                    __syncthreads();
                    int before = sm.taken;
                    for (int w = 0; w < warp; ++w) before += sm.scratch[w];
                    before += __popc(ballot & ((1u << lane) - 1u));
                    if (tie && above + before < need)
                        sm.cand[above + before] = Cand{frame[head + e], tb + e};
                    __syncthreads();
                    if (tid == 0) {
                        int add = 0;
                        for (int w = 0; w < NW; ++w) add += sm.scratch[w];
                        sm.taken += add;
                    }
                    __syncthreads();
                    if (above + sm.taken >= need) break;
                }
                n = need;
                __syncthreads();
                if (tid == 0) sm.ncand = 0;
            }

            // ---- 4. running list := K best of (candidates U list); one warp per item,
            // its lanes splitting the count of entries that beat it
            {
                const Cand* R = sm.run[cur];
                Cand* Rn = sm.run[cur ^ 1];
                const int real_in_R = count_beating(R, K, pad);
                const int items = n + real_in_R;
                const int total = min(items, K);
                for (int i = warp; i < items; i += NW) {
                    const Cand c = i < n ? sm.cand[i] : R[i - n];
                    int r = 0;
                    for (int q = lane; q < n; q += 32) r += beats(sm.cand[q], c);
                    r = __reduce_add_sync(kFullMask, r);
                    r += i < n ? count_beating(R, K, c) : i - n;
                    if (lane == 0 && r < K) Rn[r] = c;
                }
                if (tid >= total && tid < K) Rn[tid] = pad;
                __syncthreads();
                cur ^= 1;
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
                for (int i = tid; i < K; i += THREADS) sm.xlist[parity][0][i] = sm.run[cur][i];
                __syncthreads();
            } else {
                const uint32_t bar0 = map_to_rank(&sm.xbar[parity], 0);
                if (rank == 0 && tid == 0) mbar_arrive_expect_tx(&sm.xbar[parity], CLUSTER * (K + 1) * 8);
                if (warp == 0) {
                    float2 st = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
                    group_merge<32>(st.x, st.y);
                    if (lane == 0)
                        st_async_b64(map_to_rank(&sm.xstate[parity][rank], 0), __float_as_uint(st.x),
                                     __float_as_uint(st.y), bar0);
                }
                for (int i = tid; i < K; i += THREADS) {
                    const Cand c = sm.run[cur][i];
                    st_async_b64(map_to_rank(&sm.xlist[parity][rank][i], 0), __float_as_uint(c.v),
                                 uint32_t(c.j), bar0);
                }
                if (rank == 0 && tid == 0)
                    mbar_wait_bounded(&sm.xbar[parity], uint32_t(local >> 1) & 1u, ctl);
                if (rank == 0) __syncthreads();
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
                const Cand c = sm.xlist[parity][a][p];
                if (c.j == kNoIndex) continue;
                int r = p;
#pragma unroll
                for (int b = 0; b < CLUSTER; ++b)
                    if (b != a) r += count_beating(sm.xlist[parity][b], K, c);
                if (r < K) {
                    vals[row * K + r] = exp1(c.v - M) * inv_d;
                    idx[row * K + r] = c.j;
                }
            }
        }
    }
    if (tid == 0 && pending) {
        for (int c = 0; c < NCHUNK; ++c)
            if (pending >> c & 1u) mbar_wait_bounded(&sm.chunk_bar[c], (pending_par >> c) & 1u, ctl);
    }
    if (CLUSTER > 1) cluster_sync();  // CTA 0's slots stay valid until every push has landed
}

}  // namespace os
