// topk_kernel.cuh -- fused softmax + TopK: one read of x, K probabilities out.
//
// "Online normalizer calculation for softmax" (notes), section 4, fuses the
// online normalizer with TopK: a single loop keeps (m, d) and the K best logits
// u with their indices p, and only the winners are turned into probabilities
// v_i = e^(u_i - m_V) / d_V at the end.  Selecting on logits is exact because
// softmax is monotone.  The notes keep K+1 sorted slots per thread and insert
// by one bubble pass; on a GPU this kernel keeps the same invariant (a sorted
// list of the K best seen so far, per CTA) but fills it in batches:
//
//   1. a CTA loads a tile of its row slice into registers and folds it into
//      each thread's running (m, d) (chunked update, as in the softmax kernels);
//   2. threshold: every thread takes its best element; each warp sorts its 32
//      thread bests (bitonic network over shuffles); the worst of the warps'
//      j*-th entries (j* = ceil(K / warps) - 1) is beaten or equalled by at
//      least K elements of the tile, so nothing worse can be in the top K.  The
//      running list's K-th entry is a second such bound; the better one is used;
//   3. elements that are not worse than the threshold are appended to a
//      shared-memory candidate buffer (few for random data: ~K + K ln(...));
//   4. the new running list is the K best of (candidates U old list), found by
//      ranking: rank(c) = number of entries that beat c.  If the buffer
//      overflowed, the appended part is merged, the threshold is raised to the
//      new K-th entry and the not-yet-appended elements are scanned again;
//   5. the CTAs of the cluster send their lists and (m, d) states to CTA 0,
//      which ranks the CLUSTER sorted lists against each other (binary search
//      per list), folds the states with (+), and writes v = e^(u - m)/d and
//      the indices in order.
//
// Order ("beats"): larger logit first; equal logits, lower column index first.
// Index INT32_MAX marks an empty slot and never beats a real element.
//
// Rows need only 4-byte alignment: vectors are taken in the 16-byte-aligned
// frame of each row; the partial first and last vectors are read element-wise.
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

// Sort (v, j) descending by `beats` across the 32 lanes of a warp.
__device__ __forceinline__ void warp_bitonic_desc(float& v, int& j) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float ov = __shfl_xor_sync(kFullMask, v, stride);
            const int oj = __shfl_xor_sync(kFullMask, j, stride);
            const bool keep_better = ((lane & stride) == 0) == ((lane & size) == 0);
            const bool take = keep_better ? beats(ov, oj, v, j) : beats(v, j, ov, oj);
            if (take) {
                v = ov;
                j = oj;
            }
        }
    }
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

template <int THREADS, int CLUSTER, int KMAX, int CAP>
struct TopkSmem {
    float2 warp_state[THREADS / 32];
    Cand warp_thr[THREADS / 32];
    Cand cand[CAP];
    Cand run[2][KMAX];
    int ncand[2];
    float2 xstate[2][CLUSTER];
    Cand xlist[2][CLUSTER][KMAX];
};

template <int THREADS, int VPT, int CLUSTER, int KMAX, int CAP>
__global__ void __launch_bounds__(THREADS)
topk_rows_kernel(const float* __restrict__ x, float* __restrict__ vals, int* __restrict__ idx,
                 int64_t rows, int cols, int K) {
    constexpr int EPT = VPT * 4, NW = THREADS / 32, TILE = THREADS * VPT;
    static_assert(EPT <= 32, "processed-element mask is 32 bits");
    __shared__ TopkSmem<THREADS, CLUSTER, KMAX, CAP> sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int jstar = min((K + NW - 1) / NW - 1, 31);
    const Cand pad{kNegInf, kNoIndex};

    if (tid < 2) sm.ncand[tid] = 0;
    if (CLUSTER > 1) cluster_sync(); else __syncthreads();

    int parity = 0, pass = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1) {
        const float* xr = x + row * int64_t(cols);
        const int s = int((reinterpret_cast<uintptr_t>(xr) >> 2) & 3);  // row start inside its 16-B vector
        const float* frame = xr - s;                                    // 16-byte aligned
        const int64_t nvf = (int64_t(cols) + s + 3) / 4;
        const int64_t per_cta = (nvf + CLUSTER - 1) / CLUSTER;
        const int64_t begin = int64_t(rank) * per_cta;
        const int64_t end = begin + per_cta < nvf ? begin + per_cta : nvf;

        int cur = 0;
        if (tid < KMAX) sm.run[0][tid] = pad;
        float m = kNegInf, d = 0.f;

        for (int64_t tb = begin; tb < end; tb += TILE) {
            // 1. load the tile; element (k, q) has column 4u - s + q
            float v[EPT];
            int64_t u0[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t u = tb + int64_t(k) * THREADS + tid;
                u0[k] = u;
                const int64_t j0 = 4 * u - s;
                if (u < end && j0 >= 0 && j0 + 4 <= cols) {
                    const uint4 w = ld_stream_v4(frame + 4 * u);
                    v[4 * k] = __uint_as_float(w.x);
                    v[4 * k + 1] = __uint_as_float(w.y);
                    v[4 * k + 2] = __uint_as_float(w.z);
                    v[4 * k + 3] = __uint_as_float(w.w);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t j = j0 + q;
                        v[4 * k + q] = (u < end && j >= 0 && j < cols) ? xr[j] : kNegInf;
                    }
                }
            }
            auto col_of = [&](int k, int q) -> int {
                const int64_t j = 4 * u0[k] - s + q;
                return (u0[k] < end && j >= 0 && j < cols) ? int(j) : kNoIndex;
            };

            // running (m, d): one rescale per tile
            {
                const float m_new = fmaxf(m, max_of<EPT>(v));
                d = d * rescale(m, m_new) + exp_sum<EPT>(v, m_new);
                m = m_new;
            }

            // 2. threshold from the warps' sorted thread bests
            float bv = kNegInf;
            int bj = kNoIndex;
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = col_of(k, q);
                    if (beats(v[4 * k + q], j, bv, bj)) {
                        bv = v[4 * k + q];
                        bj = j;
                    }
                }
            warp_bitonic_desc(bv, bj);
            if (lane == jstar) sm.warp_thr[warp] = Cand{bv, bj};
            __syncthreads();
            Cand T = sm.warp_thr[0];
#pragma unroll
            for (int w = 1; w < NW; ++w)
                if (beats(T, sm.warp_thr[w])) T = sm.warp_thr[w];
            if (beats(sm.run[cur][K - 1], T)) T = sm.run[cur][K - 1];

            // 3-4. collect candidates not worse than T, merge into the running list
            uint32_t done = 0;  // bit i: element i already appended
            while (true) {
                int* counter = &sm.ncand[pass & 1];
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = 4 * k + q;
                        const int j = col_of(k, q);
                        if (j != kNoIndex && !(done >> i & 1u) && !beats(T.v, T.j, v[i], j)) {
                            const int pos = atomicAdd(counter, 1);
                            if (pos < CAP) {
                                sm.cand[pos] = Cand{v[i], j};
                                done |= 1u << i;
                            }
                        }
                    }
                __syncthreads();
                const int n_all = *counter;
                const int n = min(n_all, CAP);
                if (tid == 0) sm.ncand[(pass + 1) & 1] = 0;
                const Cand* R = sm.run[cur];
                Cand* Rn = sm.run[cur ^ 1];
                int real_in_R = count_beating(R, K, pad);  // entries of R that are not empty
                const int total = min(n + real_in_R, K);
                for (int i = tid; i < n + K; i += THREADS) {
                    const Cand c = i < n ? sm.cand[i] : R[i - n];
                    if (c.j == kNoIndex) continue;
                    int r = i < n ? count_beating(R, K, c) : i - n;
                    for (int q = 0; q < n; ++q) r += beats(sm.cand[q], c);
                    if (r < K) Rn[r] = c;
                }
                if (tid >= total && tid < K) Rn[tid] = pad;
                __syncthreads();
                cur ^= 1;
                ++pass;
                if (beats(sm.run[cur][K - 1], T)) T = sm.run[cur][K - 1];
                if (n_all <= CAP) break;
            }
        }

        // 5. CTA state and list to CTA 0 of the cluster
        {
            float mm = m, dd = d;
            group_merge<32>(mm, dd);
            if (lane == 0) sm.warp_state[warp] = make_float2(mm, dd);
            __syncthreads();
            if (warp == 0) {
                float2 st = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
                group_merge<32>(st.x, st.y);
                if (lane == 0) {
                    if (CLUSTER == 1) sm.xstate[parity][0] = st;
                    else st_cluster_f2(map_to_rank(&sm.xstate[parity][rank], 0), st);
                }
            }
            for (int i = tid; i < K; i += THREADS) {
                const Cand c = sm.run[cur][i];
                if (CLUSTER == 1) {
                    sm.xlist[parity][0][i] = c;
                } else {
                    st_cluster_b64(map_to_rank(&sm.xlist[parity][rank][i], 0),
                                   __float_as_uint(c.v), uint32_t(c.j));
                }
            }
        }
        if (CLUSTER > 1) cluster_sync(); else __syncthreads();

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
}

}  // namespace os
