// topk_kernel.cuh -- fused softmax + TopK: one read of x from HBM, K
// probabilities out.
//
// "Online normalizer calculation for softmax" (notes), section 4, fuses the
// online normalizer with TopK: one pass keeps (m, d) and the K best logits u
// with their indices p, and only the winners become probabilities
// v_i = e^(u_i - m_V) / d_V at the end (selecting on logits is exact because
// softmax is monotone).  The notes insert every element into a sorted list
// behind a rejection test against the list's last entry.  Here the rejection
// threshold comes from the data itself, and only the few survivors are ever
// compared with one another:
//
//   pass 1 (HBM): a CTA streams its segment of the row (the whole row, or one
//     of S <= 8 segments of a thread-block cluster when rows are too few to
//     fill the GPU) in chunks of U 16-byte blocks per thread.  Every thread
//     folds each chunk into its running (m, d) (chunk maximum, then the sum of
//     e^(x - max) on the SFU: one FMA and one ex2 per element, one rescale
//     per chunk) and into its running maximum, and keeps each block's maximum
//     as a rounded-up 16-bit key in shared memory;
//   threshold: each warp sorts its 32 thread maxima (bitonic network over
//     shuffles); the smallest of the warps' j*-th largest (j* = ceil(K /
//     warps) - 1) has at least K elements of the segment at or above it (that
//     many threads of every warp hold one), so nothing below it can be in the
//     top K;
//   pass 2 (L2): only the blocks whose key reaches the threshold's are read
//     again (about one in a hundred for random data): each warp lists its own
//     in its share of a shared-memory list and rereads them one per lane (no
//     CTA barrier in between), and their elements at or above the threshold
//     become the candidates, a warp reserving its slots in the shared-memory
//     buffer with one atomic;
//   selection: up to 512 candidates (K <= 64; 256 for larger K), each one's
//     rank is the number of candidates that beat it (one thread per
//     candidate, comparing against register-held slabs of all candidates by
//     broadcast shuffles) and rank r < K puts it in slot r of the list; more
//     candidates are first cut to the K best by a radix select on their
//     order keys (four 8-bit digit rounds, the lowest columns taken among
//     ties at the K-th key) when K <= 64, and sorted whole by a CTA-wide
//     bitonic sort of 64-bit keys (logit order key, then column) for larger K.  If the candidates
//     overflow the buffer (heavy
//     ties at the threshold), an exact path finds the K-th largest key of the
//     segment by bisection and admits the ties at it in column order;
//   output: the CTA's (m, d) is the (+)-fold of its threads' states.  With
//     S = 1 the CTA writes v = e^(u - m)/d and the indices, best first.  With
//     S > 1 every CTA pushes its state and list into CTA 0 of the cluster with
//     st.async (completing CTA 0's barrier), and CTA 0 ranks the lists against
//     each other (binary search per list) and writes the row.
//
// Order ("beats"): larger logit first; equal logits, lower column index first.
// Index INT32_MAX marks an empty slot and never beats a real element.
//
// Rows need only 4-byte alignment: block b of a row covers columns
// 4b - head .. 4b + 3 - head, where head (0..3) is the row start's offset in
// its 16-byte block.  Blocks lying wholly inside the row are read with one
// 128-bit load; the (at most two) partial blocks at the ends element by
// element, so nothing outside the row is touched.
#pragma once

#include <climits>

#include "ops.cuh"
#include "softmax_kernels.cuh"

namespace os {

constexpr float kLn2f = 0.693147182f;  // fp32(ln 2)

// 8-byte aligned: candidates move as one 64-bit word (cluster exchange) and
// the selection sort reuses the candidate buffer for 64-bit keys.
struct __align__(8) Cand {
    float v;
    int j;
};

constexpr int kNoIndex = INT_MAX;
// Candidate counts up to this are ranked by counting (one thread per
// candidate, so at most the CTA's width); more are cut to the K best by a
// radix select (K <= 64) or sorted (larger K, whose rows bring hundreds of
// candidates, where the sort is faster).
template <int THREADS, int KMAX>
constexpr int rank_max() { return KMAX <= 64 ? (THREADS < 512 ? THREADS : 512) : 256; }
// Candidates compared per batch of register-held slabs (8 slabs of 32).
constexpr int kSlabBatch = 8;

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

__device__ __forceinline__ float order_key_inverse(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Sort key of a candidate: ascending key = "beats" order (larger logit first,
// then lower column).  -0 is keyed as +0, as the comparison treats them equal.
__device__ __forceinline__ uint64_t cand_key(const Cand& c) {
    return (uint64_t(~order_key(c.v + 0.0f)) << 32) | uint32_t(c.j);
}

// The best min(K, n) of the n candidates cand[0..n) into list[0..), best
// first, by a bitonic sort of their keys over the CTA: partners within a warp
// exchange by shuffles, across warps through shared memory (cand[] is reused
// for the keys), and across a thread's own elements (element e * THREADS +
// tid) in registers.  n <= THREADS * EMAX.  Entries past n stay as they were.
// Zero values come back as +0 (the caller restores the sign from the row).
// Every thread of the CTA must call it.
template <int THREADS, int EMAX>
__device__ __forceinline__ void bitonic_select(Cand* cand, int n, Cand* list, int K) {
    static_assert(EMAX == 1 || EMAX == 2 || EMAX == 4, "elements per thread");
    const int tid = threadIdx.x;
    int P = 32;
    while (P < n) P <<= 1;
    const int E = P > THREADS ? P / THREADS : 1;  // elements per thread
    const bool active = tid < P;                  // whole warps (P is a multiple of 32)
    uint64_t key[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int i = e * THREADS + tid;
        key[e] = (active && e < E && i < n) ? cand_key(cand[i]) : ~0ull;
    }
    uint64_t* ks = reinterpret_cast<uint64_t*>(cand);
    __syncthreads();  // every candidate read before cand[] holds keys
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {  // uniform over the CTA
            if (j >= THREADS) {  // j / THREADS is 1 or 2: element pairs (0,1),(2,3) or (0,2),(1,3)
                auto cas = [&](uint64_t& a, uint64_t& b, int i) {
                    const uint64_t lo = min(a, b), hi = max(a, b);
                    const bool up = (i & k) == 0;
                    a = up ? lo : hi;
                    b = up ? hi : lo;
                };
                if constexpr (EMAX >= 2) {
                    if (j == THREADS) {
                        cas(key[0], key[1], tid);
                        if constexpr (EMAX >= 4) cas(key[2], key[3], 2 * THREADS + tid);
                    } else if constexpr (EMAX >= 4) {
                        cas(key[0], key[2], tid);
                        cas(key[1], key[3], THREADS + tid);
                    }
                }
            } else if (j >= 32) {
#pragma unroll
                for (int e = 0; e < EMAX; ++e)
                    if (active && e < E) ks[e * THREADS + tid] = key[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < EMAX; ++e) {
                    if (active && e < E) {
                        const int i = e * THREADS + tid;
                        const uint64_t o = ks[i ^ j];
                        const bool keep_min = ((i & k) == 0) == ((i & j) == 0);
                        key[e] = keep_min ? min(key[e], o) : max(key[e], o);
                    }
                }
                __syncthreads();
            } else if (active) {
#pragma unroll
                for (int e = 0; e < EMAX; ++e) {
                    if (e < E) {
                        const int i = e * THREADS + tid;
                        const uint64_t o = __shfl_xor_sync(kFullMask, key[e], j);
                        const bool keep_min = ((i & k) == 0) == ((i & j) == 0);
                        key[e] = keep_min ? min(key[e], o) : max(key[e], o);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int i = e * THREADS + tid;
        if (active && e < E && i < K && i < n)
            list[i] = Cand{order_key_inverse(~uint32_t(key[e] >> 32)), int(uint32_t(key[e]))};
    }
}

// The K best of the n candidates cand[0..n) (K <= n <= THREADS * EMAX, by
// "beats"), moved unordered into cand[0..K).  A radix select finds the K-th
// largest order key (four rounds of 8-bit digits, histograms in shared
// memory), then the candidates above it and the lowest-column ties at it are
// compacted into out[0..K) and copied back.  work: at least 256 + 8 ints of
// shared memory; out: room for K candidates.  Every thread of the CTA must
// call it.
template <int THREADS, int EMAX>
__device__ __forceinline__ void radix_select_compact(Cand* cand, int n, int K, int* work, Cand* out) {
    const int tid = threadIdx.x, lane = tid & 31;
    int* hist = work;             // 256 bins
    int* ctl = work + 256;        // [0] digit, [1] count above it, [2] > count, [3] tie count
    uint32_t key[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int i = e * THREADS + tid;
        key[e] = i < n ? order_key(cand[i].v + 0.0f) : 0u;  // -0 keyed as +0, as beats() compares
    }
    uint32_t prefix = 0, mask = 0;
    int kleft = K;  // how many still to take among the keys matching the prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += THREADS) hist[b] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            const int i = e * THREADS + tid;
            if (i < n && (key[e] & mask) == prefix) atomicAdd(&hist[(key[e] >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {  // the digit holding the kleft-th largest key: lane l scans bins 8 l .. 8 l + 7
            int c[8], s = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = hist[8 * lane + q];
                s += c[q];
            }
            int x = s;  // inclusive suffix sum over lanes lane .. 31
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_down_sync(kFullMask, x, o);
                if (lane + o < 32) x += v;
            }
            int run = x - s;  // keys in the bins of higher lanes
#pragma unroll
            for (int q = 7; q >= 0; --q) {
                if (run < kleft && run + c[q] >= kleft) {
                    ctl[0] = 8 * lane + q;
                    ctl[1] = run;
                }
                run += c[q];
            }
        }
        __syncthreads();
        const uint32_t d = uint32_t(ctl[0]);
        kleft -= ctl[1];
        prefix |= d << shift;
        mask |= 255u << shift;
        __syncthreads();  // ctl is rewritten by the next digit round
    }
    // prefix is the K-th largest key; K - kleft candidates lie above it and
    // kleft of its ties (the lowest columns) complete the K
    if (tid == 0) {
        ctl[2] = 0;
        ctl[3] = 0;
    }
    __syncthreads();
    const int n_gt = K - kleft;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int i = e * THREADS + tid;
        if (i < n && key[e] > prefix) out[atomicAdd(&ctl[2], 1)] = cand[i];
    }
    // ties at the K-th key: each counts the ties with a lower column
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int i = e * THREADS + tid;
        if (i < n && key[e] == prefix) {
            const int j = cand[i].j;
            int lower = 0;
            for (int q = 0; q < n; ++q)
                lower += order_key(cand[q].v + 0.0f) == prefix && cand[q].j < j;
            if (lower < kleft) out[n_gt + lower] = cand[i];
        }
    }
    __syncthreads();
    for (int i = tid; i < K; i += THREADS) cand[i] = out[i];
    __syncthreads();
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

// Exclusive prefix over the CTA of per-thread counts, in thread order; also
// returns the CTA total.  Every thread must call it.
template <int THREADS>
__device__ __forceinline__ int block_exclusive_scan(int c, int* scratch, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) {
        const int s = scratch[w];
        if (w < warp) before += s;
        total += s;
    }
    __syncthreads();
    return before + incl - c;
}

template <int THREADS, int KMAX, int CAP, int MAXC>
struct TopkSmem {
    uint64_t xbar[2];
    float warp_thr[THREADS / 32];
    float2 warp_state[THREADS / 32];
    int scratch[THREADS / 32];
    int ncand[2];  // candidate counters of alternate rows
    int nflag[2];  // listed-block counters of alternate rows
    int flag;
    Cand cand[CAP];
    Cand list[KMAX];
    float2 xstate[2][MAXC];
    Cand xlist[2][MAXC][KMAX];
};

// Dynamic shared memory: per group of chunks and thread, the maximum of each
// of the thread's U block slots (as a 16-bit key rounded up, see block_key;
// U = 4 keys in 8 bytes), and the list of the blocks that pass 2 reads again.
template <int THREADS, int U, int GROUPS, int FCAP>
struct TopkDynSmem {
    static_assert(U == 4, "four 16-bit keys per 8-byte slot");
    uint2 bkey[GROUPS][THREADS];
    int flagged[FCAP];
};

// Upper 16 bits of the order-preserving key, rounded up: block_key(x) >=
// threshold_key(t) whenever x >= t, so a block whose key is below the
// threshold's holds nothing at or above it.
__device__ __forceinline__ uint32_t block_key(float x) { return (order_key(x) + 0xffffu) >> 16; }
__device__ __forceinline__ uint32_t threshold_key(float t) { return order_key(t) >> 16; }

// A CTA's segment of one row.
struct TopkSegment {
    const float* xr;       // the row's first element
    int head;              // the row start's offset in its 16-byte block, in elements
    int full_lo, full_hi;  // blocks [full_lo, full_hi) lie wholly inside the row
    int b0, b1;            // the CTA's blocks of the row
};

// PLAIN: the K largest values themselves (TopK of x, no softmax): no (m, d)
// is formed and vals are the selected x.
// KMAX: largest K; MAXC: largest cluster (CTAs per row) the launch may use.
template <int THREADS, int U, int KMAX, int MAXC, int CAP, int GROUPS, int FCAP, bool PLAIN>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2)
topk_rows_kernel(const float* __restrict__ x, float* __restrict__ vals, int* __restrict__ idx,
                 int64_t rows, int cols, int K, int S, KernelCtl ctl) {
    constexpr int NW = THREADS / 32;
    constexpr int CHUNK = THREADS * U;  // 16-byte blocks per chunk
    constexpr int RANKMAX = rank_max<THREADS, KMAX>();
    static_assert(CAP % THREADS == 0 && CAP >= 128 && KMAX <= THREADS && KMAX <= RANKMAX &&
                  RANKMAX <= THREADS, "buffer sizes");
    __shared__ __align__(16) TopkSmem<THREADS, KMAX, CAP, MAXC> sm;
    extern __shared__ __align__(16) unsigned char dyn_raw[];
    auto& dyn = *reinterpret_cast<TopkDynSmem<THREADS, U, GROUPS, FCAP>*>(dyn_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = S > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / S, nclusters = gridDim.x / S;
    const int jstar = min((K + NW - 1) / NW - 1, 31);
    const Cand pad{kNegInf, kNoIndex};
    const uint64_t policy = l2_policy_evict_first();

    // The exchange barriers exist only for a row split over a cluster.  With
    // one CTA per row nothing here needs a CTA barrier: thread 0 clears a
    // row's counters before its pass 1, and every other thread first uses
    // them after the threshold barrier that follows.
    if (S > 1) {
        if (tid == 0) {
            mbar_init(&sm.xbar[0], 1);
            mbar_init(&sm.xbar[1], 1);
            mbar_init_fence();
        }
        cluster_sync();
    }

    bool failed = false;  // a wait gave up: outputs are garbage, the status word says so
    int parity = 0;
    int64_t local = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1, ++local) {
        // a new row of this cluster reuses CTA 0's exchange slots: keep lockstep
        if (S > 1 && local > 0) cluster_sync();
        TopkSegment g;
        g.xr = x + row * int64_t(cols);
        g.head = int((reinterpret_cast<uintptr_t>(g.xr) >> 2) & 3);
        {
            const int64_t span = int64_t(cols) + g.head;
            const int nb = int((span + 3) >> 2);
            g.full_lo = g.head > 0 ? 1 : 0;
            g.full_hi = int(span >> 2);
            const int per = (nb + S - 1) / S;
            g.b0 = min(int(rank) * per, nb);
            g.b1 = min(g.b0 + per, nb);
        }
        const float* xb = g.xr - g.head;  // 16-byte aligned; dereferenced only inside the row
        const int nchunks = (g.b1 - g.b0 + CHUNK - 1) / CHUNK;
        const int G = max(1, (nchunks + GROUPS - 1) / GROUPS);  // chunks per group
        const int ngroups = (nchunks + G - 1) / G;
        int* counter = &sm.ncand[parity];
        int* nflag = &sm.nflag[parity];
        if (tid == 0) {  // last used two rows ago
            *counter = 0;
            *nflag = 0;
        }
        if (tid < K) sm.list[tid] = pad;

        // ---- pass 1 (HBM): running (m, d) and maximum; block maxima kept as keys
        float m = kNegInf, d = 0.f, tmax = kNegInf;
        for (int c = 0; c < nchunks; ++c) {
            float v[U][4];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int b = g.b0 + c * CHUNK + k * THREADS + tid;
                if (b < g.b1 && b >= g.full_lo && b < g.full_hi) {
                    const uint4 w = ld_policy_v4(xb + 4 * int64_t(b), policy);
                    v[k][0] = __uint_as_float(w.x);
                    v[k][1] = __uint_as_float(w.y);
                    v[k][2] = __uint_as_float(w.z);
                    v[k][3] = __uint_as_float(w.w);
                } else {
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        const int64_t col = 4 * int64_t(b) + l - g.head;
                        v[k][l] = (b < g.b1 && col >= 0 && col < cols) ? g.xr[col] : kNegInf;
                    }
                }
            }
            float bm[U];
#pragma unroll
            for (int k = 0; k < U; ++k) bm[k] = fmaxf(max3(v[k][0], v[k][1], v[k][2]), v[k][3]);
            float cmax = bm[0];
#pragma unroll
            for (int k = 1; k < U; k += 2) cmax = max3(cmax, bm[k], bm[k + 1 < U ? k + 1 : k]);
            // (m, d) against the new running maximum m': e^(x - m') is taken as
            // 2^(x log2e - M_hi) (2^(-M_lo)), where M_hi + M_lo = m' log2e exactly
            // (the residual of an FMA): one FMA and one SFU ex2 per element
            // (an FMA-pipe polynomial instead measured 16-21 % slower here).
            // Dropping log2e's own rounding costs 1.3e-8 |x - m'| relative per term.
            if constexpr (!PLAIN) {
                const float m_new = fmaxf(m, cmax);
                const float ms = finite_shift(m_new);
                const float M_hi = ms * expc::kLog2e;
                const float M_lo = fmaf(ms, expc::kLog2e, -M_hi);
                const float2 L2 = splat2(expc::kLog2e), nM = splat2(-M_hi);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const float2 t0 = fma2(make_float2(v[k][0], v[k][1]), L2, nM);
                    const float2 t1 = fma2(make_float2(v[k][2], v[k][3]), L2, nM);
                    acc = add2(acc, make_float2(ex2_sfu(t0.x), ex2_sfu(t0.y)));
                    acc = add2(acc, make_float2(ex2_sfu(t1.x), ex2_sfu(t1.y)));
                }
                const float keep = m == m_new ? 1.0f : ex2_sfu((m - m_new) * expc::kLog2e);
                d = fmaf(d, keep, (acc.x + acc.y) * fmaf(-M_lo, kLn2f, 1.0f));
                m = m_new;
            }
            tmax = fmaxf(tmax, cmax);
            // block keys (thread-private slot): a group's first chunk writes, later ones raise
            const int grp = c / G;
            uint2 key = make_uint2(block_key(bm[0]) | (block_key(bm[1]) << 16),
                                   block_key(bm[2]) | (block_key(bm[3]) << 16));
            if (c != grp * G) {
                const uint2 old = dyn.bkey[grp][tid];
                key = make_uint2(__vmaxu2(key.x, old.x), __vmaxu2(key.y, old.y));
            }
            dyn.bkey[grp][tid] = key;
        }

        // ---- threshold T over the whole segment (at least K elements are >= T);
        // the same barrier publishes each warp's (m, d)
        {
            const float sorted = warp_sort_desc(tmax);
            if (lane == jstar) sm.warp_thr[warp] = sorted;
            float mm = m, dd = d;
            group_merge<32>(mm, dd);
            if (lane == 0) sm.warp_state[warp] = make_float2(mm, dd);
        }
        __syncthreads();
        float T = sm.warp_thr[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) T = fminf(T, sm.warp_thr[w]);
        const uint32_t tk = threshold_key(T);

        // ---- the blocks whose key reaches T's, listed per warp in the warp's
        // share of the list, then read again (L2) by the same warp, one block
        // per lane, their elements >= T becoming the candidates; no CTA barrier
        // in between.  The keys are read in one batch: shared-memory round
        // trips are slow while the SM's other CTA streams.
        constexpr int WCAP = FCAP / NW;  // list entries per warp
        {
            uint32_t hit = 0;  // bit q * U + k: slot k of group q reaches the threshold
#pragma unroll
            for (int q = 0; q < GROUPS; ++q) {
                if (q < ngroups) {
                    const uint2 kk = dyn.bkey[q][tid];
                    hit |= uint32_t((kk.x & 0xffffu) >= tk) << (q * U);
                    hit |= uint32_t((kk.x >> 16) >= tk) << (q * U + 1);
                    hit |= uint32_t((kk.y & 0xffffu) >= tk) << (q * U + 2);
                    hit |= uint32_t((kk.y >> 16) >= tk) << (q * U + 3);
                }
            }
            int mine = 0;
            for (uint32_t h = hit; h != 0; h &= h - 1) {
                const int s = __ffs(h) - 1, q = s / U, k = s % U;
                const int c_end = min(nchunks, (q + 1) * G);
                for (int c = q * G; c < c_end; ++c) mine += g.b0 + c * CHUNK + k * THREADS + tid < g.b1;
            }
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += t;
            }
            const int wn = __shfl_sync(kFullMask, incl, 31);  // the warp's flagged blocks
            int* wl = dyn.flagged + warp * WCAP;
            int pos = incl - mine;
            if (mine > 0) {
                for (uint32_t h = hit; h != 0; h &= h - 1) {
                    const int s = __ffs(h) - 1, q = s / U, k = s % U;
                    const int c_end = min(nchunks, (q + 1) * G);
                    for (int c = q * G; c < c_end; ++c) {
                        const int b = g.b0 + c * CHUNK + k * THREADS + tid;
                        if (b < g.b1) {
                            if (pos < WCAP) wl[pos] = b;
                            ++pos;
                        }
                    }
                }
            }
            if (wn > WCAP) {
                if (lane == 0) atomicOr(nflag, 1);  // this warp's list overflowed
            } else {
                __syncwarp();
                for (int i0 = 0; i0 < wn; i0 += 32) {  // uniform over the warp
                    const int i = i0 + lane;
                    float v[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
                    int b = 0;
                    uint32_t live = 0;
                    if (i < wn) {
                        b = wl[i];
                        if (b >= g.full_lo && b < g.full_hi) {
                            const uint4 w = ld_policy_v4(xb + 4 * int64_t(b), policy);
                            v[0] = __uint_as_float(w.x);
                            v[1] = __uint_as_float(w.y);
                            v[2] = __uint_as_float(w.z);
                            v[3] = __uint_as_float(w.w);
                            live = 0xfu;
                        } else {
#pragma unroll
                            for (int l = 0; l < 4; ++l) {
                                const int64_t col = 4 * int64_t(b) + l - g.head;
                                const bool in = col >= 0 && col < cols;
                                if (in) v[l] = g.xr[col];
                                live |= uint32_t(in) << l;
                            }
                        }
                    }
                    uint32_t hitmask = 0;  // bit l: element l is a candidate
#pragma unroll
                    for (int l = 0; l < 4; ++l) hitmask |= uint32_t(v[l] >= T) << l;
                    hitmask &= live;
                    const int cnt = __popc(hitmask);
                    int cincl = cnt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int t = __shfl_up_sync(kFullMask, cincl, o);
                        if (lane >= o) cincl += t;
                    }
                    int base = 0;
                    if (lane == 31 && cincl > 0) base = atomicAdd(counter, cincl);
                    int cpos = __shfl_sync(kFullMask, base, 31) + cincl - cnt;
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        if ((hitmask >> l) & 1u) {
                            if (cpos < CAP)
                                sm.cand[cpos] = Cand{v[l], int(4u * uint32_t(b) + uint32_t(l) -
                                                              uint32_t(g.head))};
                            ++cpos;
                        }
                    }
                }
            }
        }
        __syncthreads();
        // a warp whose list overflowed sends the row to the exact path
        int n = *nflag == 0 ? *counter : CAP + 1;

        if (n > CAP) {
            // ---- exact path (heavy ties at T; rare): the K-th largest key of the
            // segment by bisection over its columns, read again from memory;
            // then the keys above it in any order and the ties at it in column order.
            // -0 is keyed as +0 (x + 0 is +0 for both zeros), as beats() compares,
            // so a tie between the two zeros goes to the lower column.
            const int c_lo = int(max(int64_t(0), 4 * int64_t(g.b0) - g.head));
            const int c_hi = int(min(int64_t(cols), 4 * int64_t(g.b1) - g.head));
            const float* xr = g.xr;
            const int need = min(K, c_hi - c_lo);
            uint32_t t = 0;
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t probe = t | (1u << bit);
                int cnt = 0;
                // 64-bit element indices: c_hi can be 2^31 - 1, and e + THREADS must not wrap
                for (int64_t e = int64_t(c_lo) + tid; e < c_hi; e += THREADS)
                    cnt += order_key(xr[e] + 0.0f) >= probe;
                if (block_sum<THREADS>(cnt, sm.scratch) >= need) t = probe;
            }
            int admitted = 0;
            for (int64_t base = c_lo; base < c_hi; base += THREADS) {
                const int64_t e = base + tid;
                const bool above = e < c_hi && order_key(xr[e] + 0.0f) > t;
                int round_total = 0;
                const int p = admitted + block_exclusive_scan<THREADS>(above, sm.scratch, round_total);
                if (above) sm.cand[p] = Cand{xr[e], int(e)};
                admitted += round_total;
            }
            for (int64_t base = c_lo; base < c_hi && admitted < need; base += THREADS) {  // uniform
                const int64_t e = base + tid;
                const bool tie = e < c_hi && order_key(xr[e] + 0.0f) == t;
                int round_total = 0;
                const int p = admitted + block_exclusive_scan<THREADS>(tie, sm.scratch, round_total);
                if (tie && p < need) sm.cand[p] = Cand{xr[e], int(e)};
                admitted += round_total;
            }
            n = need;
            __syncthreads();
        }

        // ---- selection.  More than RANKMAX candidates are sorted (the large-K
        // build) or first cut to the K best by a radix select on their order
        // keys (K <= 64).  Up to RANKMAX, thread t ranks candidate t by
        // counting the candidates that beat it; rank r < K puts it in slot r
        // of the list.  Each warp holding candidates loads them into registers
        // in batches of kSlabBatch slabs (lane l of slab s holds candidate
        // 32 s + l) and compares against them by broadcast shuffles, so the
        // count is a few hundred shuffles with few shared-memory round trips.
        if constexpr (KMAX <= 64) {
            if (n > RANKMAX) {  // uniform
                radix_select_compact<THREADS, CAP / THREADS>(sm.cand, n, K, dyn.flagged + 1024,
                                                             reinterpret_cast<Cand*>(dyn.flagged));
                n = K;
            }
        }
        if (n <= RANKMAX) {  // uniform
            if (warp * 32 < n) {  // warp-uniform
                const Cand mine = tid < n ? sm.cand[tid] : pad;
                int r = 0;
                for (int s0 = 0; s0 * 32 < n; s0 += kSlabBatch) {  // uniform
                    Cand slab[kSlabBatch];
#pragma unroll
                    for (int s = 0; s < kSlabBatch; ++s) {
                        const int i = 32 * (s0 + s) + lane;
                        slab[s] = i < n ? sm.cand[i] : pad;
                    }
#pragma unroll
                    for (int s = 0; s < kSlabBatch; ++s) {
                        if (32 * (s0 + s) < n) {  // uniform
#pragma unroll 8
                            for (int q = 0; q < 32; ++q) {
                                const float v = __shfl_sync(kFullMask, slab[s].v, q);
                                const int jj = __shfl_sync(kFullMask, slab[s].j, q);
                                r += beats(v, jj, mine.v, mine.j);
                            }
                        }
                    }
                }
                if (tid < n && r < K) sm.list[r] = mine;
            }
        } else if constexpr (KMAX > 64) {
            // K up to 256: a bitonic sort of all candidates gives the list
            // (zeros come back as +0 and take their sign from the row)
            bitonic_select<THREADS, CAP / THREADS>(sm.cand, n, sm.list, K);
            __syncthreads();
            if (tid < K && tid < n && sm.list[tid].v == 0.f) sm.list[tid].v = g.xr[sm.list[tid].j];
        }

        __syncthreads();  // the list is complete

        // ---- the CTA's (m, d) (warp states published at the threshold barrier),
        // then the outputs
        float2 st = make_float2(kNegInf, 0.f);
        if (warp == 0 || (S == 1 && warp * 32 < K)) {  // every warp that writes outputs folds it
            st = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
            group_merge<32>(st.x, st.y);
        }
        if (S == 1) {
            if (tid < K) {
                const Cand c = sm.list[tid];
                vals[row * K + tid] = PLAIN ? c.v : exp1(c.v - st.x) * (1.0f / st.y);
                idx[row * K + tid] = c.j;
            }
            __syncthreads();  // list and warp states are rewritten by the next row
            continue;
        }
        const bool withhold = ctl.fault == kFaultSkipFirstLoad && blockIdx.x == 1 && local == 0;
        const uint32_t bar0 = map_to_rank(&sm.xbar[parity], 0);
        if (rank == 0 && tid == 0) mbar_arrive_expect_tx(&sm.xbar[parity], S * (K + 1) * 8);
        if (!withhold) {
            if (tid == 0)
                st_async_b64(map_to_rank(&sm.xstate[parity][rank], 0), __float_as_uint(st.x),
                             __float_as_uint(st.y), bar0);
            if (tid < K)
                st_async_b64(map_to_rank(&sm.xlist[parity][rank][tid], 0), __float_as_uint(sm.list[tid].v),
                             uint32_t(sm.list[tid].j), bar0);
        }
        if (rank == 0) {
            if (tid == 0 && !failed)
                sm.flag = mbar_wait_bounded(&sm.xbar[parity], uint32_t(local >> 1) & 1u, ctl) ? 1 : 0;
            __syncthreads();
            failed = failed || sm.flag == 0;
            float M = kNegInf;
            for (int c = 0; c < S; ++c) M = fmaxf(M, sm.xstate[parity][c].x);
            float D = 0.f;
            for (int c = 0; c < S; ++c) D += sm.xstate[parity][c].y * rescale(sm.xstate[parity][c].x, M);
            const float inv_d = 1.0f / D;
            for (int i = tid; i < S * K; i += THREADS) {
                const int a = i / K, p = i - a * K;
                const Cand c = sm.xlist[parity][a][p];
                if (c.j == kNoIndex) continue;
                int r = p;
                for (int b = 0; b < S; ++b)
                    if (b != a) r += count_beating(sm.xlist[parity][b], K, c);
                if (r < K) {
                    vals[row * K + r] = PLAIN ? c.v : exp1(c.v - M) * inv_d;
                    idx[row * K + r] = c.j;
                }
            }
        }
        __syncthreads();  // list and warp states are rewritten by the next row
    }
    if (S > 1) cluster_sync();  // CTA 0's slots stay valid until every push has landed
}

}  // namespace os
