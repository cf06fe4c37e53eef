// softmax_kernels.cuh -- row-wise online-normalizer softmax, three kernel families.
//
// All three compute, per row, y_i = e^(x_i - m) / d with (m, d) the row's
// online-normalizer state ("Online normalizer calculation for softmax"
// notes, section 3; "5.2 CUDA Online Softmax", sections 2-7):
//
//   * each thread reduces the elements it owns to a state (m_t, d_t) with
//     the chunked update m' = max(m, max chunk), d' = d e^(m - m') +
//     sum_chunk e^(x - m') (Lesson 7, NumPy chunked simulation);
//   * thread states are merged with the (+) operator: across lanes with
//     shuffles, across warps through shared memory, across the CTAs of a
//     thread-block cluster through distributed shared memory;
//   * the output pass writes y_i = e^(x_i - m) / d.
//
// warp_rows   Rows of at most 32 x VPT vectors.  A group of L lanes owns one
//             row, held in registers: one HBM read and one write per element
//             ("CUDA operator optimization (3)", warp per row; "5.2", V3
//             register cache).
// onchip_rows Rows up to CLUSTER x THREADS x VPT vectors.  The row is split
//             over the CTAs of a cluster and held in registers; each thread
//             keeps e^(x - m_t) for its elements, so the output pass is one
//             multiply by e^(m_t - m)/d per element (one exponential per
//             element in total) and HBM sees one read and one write.
// stream_rows Any row length.  Pass 1 streams the row and keeps a running
//             (m, d) per thread with one rescale per chunk of UNROLL vectors;
//             pass 2 re-reads the row and writes y ("5.2", V2/V4 two-pass).
//
// Layout: x and y are dense row-major [rows, cols]; a "vector" is 16 bytes of
// input (4 fp32 or 8 bf16).  When cols is a multiple of the vector width and
// both base pointers are 16-byte aligned ("aligned"), every row starts on a
// vector boundary and all traffic is 128-bit; otherwise the same register
// layout is filled and drained element by element.
#pragma once

#include "ops.cuh"

namespace os {

constexpr float kNegInf = -__builtin_huge_valf();

// Load vector slot v of a row (elements v*EPV .. v*EPV+EPV-1) into out[];
// elements at or beyond `cols` read as -inf.
// Column limit of row `row` under a causal mask: columns c > (row mod period)
// + offset are masked; period 0 means no mask (the whole row).
__device__ __forceinline__ int causal_limit(int64_t row, int cols, int64_t period, int64_t offset) {
    if (period <= 0) return cols;
    const int64_t lim = row % period + offset + 1;
    return int(lim < cols ? (lim > 0 ? lim : 0) : cols);
}

template <typename TI>
__device__ __forceinline__ void load_slot(const TI* row, int64_t v, int cols, bool aligned,
                                          float* out) {
    constexpr int EPV = VecTraits<TI>::EPV;
    if (aligned) {
        unpack(ld_coherent_v4(row + v * EPV), out, TI());
    } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int64_t j = v * EPV + e;
            out[e] = j < cols ? to_f32(row[j]) : kNegInf;
        }
    }
}

template <typename TI, typename TO>
__device__ __forceinline__ void store_slot(TO* row, int64_t v, int cols, bool aligned,
                                           const float* vals) {
    constexpr int EPV = VecTraits<TI>::EPV;
    if (aligned) {
        VecStore<TO, EPV>::run(row + v * EPV, vals);
    } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int64_t j = v * EPV + e;
            if (j < cols) row[j] = from_f32<TO>(vals[e]);
        }
    }
}

// A row's vector slots.  Slot u of a row covers its columns
// [u EPV - head, u EPV - head + EPV): head (0 .. EPV - 1) is the number of
// elements between the start of the row's first 16-byte block of memory and
// the row itself, so every slot is one aligned 16-byte block.  Rows whose
// start is aligned (head = 0) have ceil(cols / EPV) slots; otherwise the
// first and last slots hold columns of neighbouring rows, which are never
// read or written.
template <typename T>
__device__ __forceinline__ int row_head(const T* row) {
    return int((reinterpret_cast<uintptr_t>(row) & 15u) / sizeof(T));
}

// Whether the output row yr can take vector stores for input slots of a row
// with this head: the slot's first column lands on an address aligned to the
// store width (EPV outputs, at most 16 bytes).
template <typename TO, int EPV>
__device__ __forceinline__ bool out_vec_ok(const TO* yr, int head) {
    constexpr uintptr_t A = EPV * sizeof(TO) < 16 ? EPV * sizeof(TO) : 16;
    return ((reinterpret_cast<uintptr_t>(yr) - uintptr_t(head) * sizeof(TO)) & (A - 1)) == 0;
}

// Slot v of a row that does not start on a 16-byte boundary (head: the row
// start's offset in its 16-byte block, row_head()): columns v EPV - head ..
// v EPV - head + EPV - 1.  A slot wholly inside [0, lim) is one 16-byte load
// (it is an aligned block of memory); the at most two partial slots of a row
// are read element by element, columns outside [0, lim) as -inf.
template <typename TI>
__device__ __forceinline__ void load_slot_peeled(const TI* row, int head, int64_t v, int lim,
                                                 float* out) {
    constexpr int EPV = VecTraits<TI>::EPV;
    const int64_t c0 = v * EPV - head;
    if (c0 >= 0 && c0 + EPV <= lim) {
        unpack(ld_coherent_v4(row + c0), out, TI());
    } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int64_t j = c0 + e;
            out[e] = j >= 0 && j < lim ? to_f32(row[j]) : kNegInf;
        }
    }
}

// The matching store: whole slots by one vector store when the output row
// has the input's block phase (vec), otherwise and at the row ends element by
// element, columns [0, cols) only.
template <typename TI, typename TO>
__device__ __forceinline__ void store_slot_peeled(TO* row, int head, bool vec, int64_t v, int cols,
                                                  const float* vals) {
    constexpr int EPV = VecTraits<TI>::EPV;
    const int64_t c0 = v * EPV - head;
    if (vec && c0 >= 0 && c0 + EPV <= cols) {
        VecStore<TO, EPV>::run(row + c0, vals);
    } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int64_t j = c0 + e;
            if (j >= 0 && j < cols) row[j] = from_f32<TO>(vals[e]);
        }
    }
}

// The shift used for e^(x - m): m itself, or 0 where m = -inf (every x seen
// so far is -inf, so every term is e^-inf = 0, the identity state's d).
__device__ __forceinline__ float finite_shift(float m) { return m > kNegInf ? m : 0.f; }

// e[i] := e^(e[i] - m) for all N entries, returning the sum (pairs on f32x2).
template <int N, bool FAST = false>
__device__ __forceinline__ float exp_shift_sum(float* e, float m) {
    static_assert(N % 2 == 0, "pairs");
    float2 acc = make_float2(0.f, 0.f);
    const float2 neg_m = splat2(-finite_shift(m));
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        float2 z = add2(make_float2(e[i], e[i + 1]), neg_m);
        float2 p = exp_pair<FAST>(z);
        e[i] = p.x;
        e[i + 1] = p.y;
        acc = add2(acc, p);
    }
    return acc.x + acc.y;
}

template <int N>
__device__ __forceinline__ float max_of(const float* e) {
    float m = e[0];
    int i = 1;
#pragma unroll
    for (; i + 1 < N; i += 2) m = max3(m, e[i], e[i + 1]);
    if (i < N) m = fmaxf(m, e[i]);
    return m;
}

template <int N>
__device__ __forceinline__ void scale_all(float* e, float s) {
    const float2 s2 = splat2(s);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        float2 p = mul2(make_float2(e[i], e[i + 1]), s2);
        e[i] = p.x;
        e[i + 1] = p.y;
    }
}

// ---------------------------------------------------------------------------
// warp_rows: L lanes per row (L in 1..32, power of two), VPT vectors per lane.
// Lane l of a group owns vector slots l, l + L, ..., l + (VPT-1) L, so a warp
// instruction covers 32 consecutive vectors of one row (or 32/L rows).
// PEEL (rows not all 16-byte aligned whole vectors): slots follow each row's
// 16-byte blocks (load_slot_peeled); otherwise `aligned` chooses between
// 16-byte and element access for the whole launch.
// Four vectors per thread: at most 64 registers (four CTAs of 256 threads
// per SM), which bf16 rows exceeded unbounded (80-99) and then kept fewer
// rows in flight: bf16 1024 columns 3130 -> 5021 GB/s on GB300.
template <typename TI, typename TO, int L, int VPT, int THREADS, bool PEEL = false>
__global__ void __launch_bounds__(THREADS, VPT == 4 ? 2048 / THREADS / 2 : 1)
warp_rows_kernel(const TI* x, TO* y, int64_t rows, int cols,
                 int aligned, int64_t period, int64_t offset) {
    constexpr int EPV = VecTraits<TI>::EPV, EPT = VPT * EPV, RPW = 32 / L;
    const int lane_in_row = threadIdx.x % L;
    const int64_t warp = (int64_t(blockIdx.x) * THREADS + threadIdx.x) / 32;
    const int64_t nwarps = int64_t(gridDim.x) * THREADS / 32;
    const int64_t nv = (int64_t(cols) + EPV - 1) / EPV;

    for (int64_t base = warp * RPW; base < rows; base += nwarps * RPW) {
        const int64_t row = base + (threadIdx.x % 32) / L;
        const bool live = row < rows;
        const TI* xr = x + (live ? row : 0) * int64_t(cols);
        TO* yr = y + (live ? row : 0) * int64_t(cols);
        // causal mask: columns at or past `lim` are -inf and never read
        const int lim = live ? causal_limit(row, cols, period, offset) : 0;
        const int head = PEEL ? row_head(xr) : 0;

        float e[EPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = int64_t(k) * L + lane_in_row;
            if (v * EPV - head < lim) {
                if constexpr (PEEL) load_slot_peeled(xr, head, v, lim, e + k * EPV);
                else load_slot(xr, v, lim, aligned && (v + 1) * EPV <= lim, e + k * EPV);
            } else {
#pragma unroll
                for (int q = 0; q < EPV; ++q) e[k * EPV + q] = kNegInf;
            }
        }
        float m = max_of<EPT>(e);
        float d = exp_shift_sum<EPT>(e, m);
        const float m_t = m;
        group_merge<L>(m, d);
        scale_all<EPT>(e, rescale(m_t, m) * (1.0f / d));
        if (live) {
            const bool yvec = PEEL && out_vec_ok<TO, EPV>(yr, head);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t v = int64_t(k) * L + lane_in_row;
                if constexpr (PEEL) {
                    if (v * EPV - head < cols) store_slot_peeled<TI, TO>(yr, head, yvec, v, cols, e + k * EPV);
                } else {
                    if (v < nv) store_slot<TI, TO>(yr, v, cols, aligned, e + k * EPV);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Merge of per-thread states of one CTA (and of the CTAs of a cluster).
// Each CTA's state goes into slot[parity][rank] of every CTA of the cluster;
// after one cluster barrier every thread folds the CLUSTER slots itself.
// The parity double buffer keeps row r+1's writes away from row r's reads:
// a CTA writes row r+2's slots only after the barrier of row r+1, which every
// peer reaches after reading row r's slots.
template <int THREADS, int CLUSTER>
struct RowMergeSmem {
    float2 warp_state[THREADS / 32];
    float2 slot[2][CLUSTER];
};

template <int THREADS, int CLUSTER>
__device__ __forceinline__ float2 merge_row_state(RowMergeSmem<THREADS, CLUSTER>& sm, float m,
                                                  float d, int parity, uint32_t rank) {
    constexpr int NW = THREADS / 32;
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    group_merge<32>(m, d);
    if (lane == 0) sm.warp_state[warp] = make_float2(m, d);
    __syncthreads();
    if (warp == 0) {
        float2 s = lane < NW ? sm.warp_state[lane] : make_float2(kNegInf, 0.f);
        group_merge<32>(s.x, s.y);
        if (lane < CLUSTER) {
            if (CLUSTER == 1) {
                sm.slot[parity][0] = s;
            } else {
                st_cluster_f2(map_to_rank(&sm.slot[parity][rank], lane), s);
            }
        }
    }
    if (CLUSTER == 1) {
        __syncthreads();
        return sm.slot[parity][0];
    }
    cluster_sync();
    float M = kNegInf;
#pragma unroll
    for (int c = 0; c < CLUSTER; ++c) M = fmaxf(M, sm.slot[parity][c].x);
    float D = 0.f;
#pragma unroll
    for (int c = 0; c < CLUSTER; ++c) D += sm.slot[parity][c].y * rescale(sm.slot[parity][c].x, M);
    return make_float2(M, D);
}

// ---------------------------------------------------------------------------
// onchip_rows: one cluster of CLUSTER CTAs per row (persistent over rows).
// CTA `rank` owns vector slots [rank*S, rank*S + S) with S = THREADS*VPT;
// thread t owns slots rank*S + t + k*THREADS.  PEEL as for warp_rows.
// CTAs of up to 256 threads: at most 64 registers, so that eight (128
// threads) or four (256) CTAs per SM keep their rows in flight (unbounded
// they took 104-125 and four or two): bf16 4096 columns 4335 -> 6968 GB/s,
// fp32 2048 4532 -> 6820, fp32 4096 6808 -> 7106 on GB300.
template <typename TI, typename TO, int THREADS, int VPT, int CLUSTER, bool PEEL = false>
__global__ void __launch_bounds__(THREADS, THREADS <= 256 ? 65536 / (THREADS * 64) : 1)
onchip_rows_kernel(const TI* x, TO* y, int64_t rows, int cols,
                   int aligned) {
    constexpr int EPV = VecTraits<TI>::EPV, EPT = VPT * EPV;
    __shared__ RowMergeSmem<THREADS, CLUSTER> sm;
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int64_t nv = (int64_t(cols) + EPV - 1) / EPV;
    const int64_t v0 = int64_t(rank) * THREADS * VPT + threadIdx.x;
    if (CLUSTER > 1) cluster_sync();  // every CTA of the cluster is running before DSMEM use

    int parity = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1) {
        const TI* xr = x + row * int64_t(cols);
        TO* yr = y + row * int64_t(cols);
        const int head = PEEL ? row_head(xr) : 0;
        const int64_t nvr = PEEL ? (int64_t(cols) + head + EPV - 1) / EPV : nv;  // this row's slots
        float e[EPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = v0 + int64_t(k) * THREADS;
            if (v < nvr) {
                if constexpr (PEEL) load_slot_peeled(xr, head, v, cols, e + k * EPV);
                else load_slot(xr, v, cols, aligned, e + k * EPV);
            } else {
#pragma unroll
                for (int q = 0; q < EPV; ++q) e[k * EPV + q] = kNegInf;
            }
        }
        const float m_t = max_of<EPT>(e);
        const float d_t = exp_shift_sum<EPT>(e, m_t);
        const float2 md = merge_row_state<THREADS, CLUSTER>(sm, m_t, d_t, parity, rank);
        scale_all<EPT>(e, rescale(m_t, md.x) * (1.0f / md.y));
        const bool yvec = PEEL && out_vec_ok<TO, EPV>(yr, head);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = v0 + int64_t(k) * THREADS;
            if (v < nvr) {
                if constexpr (PEEL) store_slot_peeled<TI, TO>(yr, head, yvec, v, cols, e + k * EPV);
                else store_slot<TI, TO>(yr, v, cols, aligned, e + k * EPV);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Exchange of CTA states inside a cluster without a cluster-wide barrier:
// every CTA sends its (m, d) with st.async into slot[parity][rank] of each
// CTA (itself included); each CTA's barrier bar[parity] expects CLUSTER x 8
// bytes and completes when all have landed.  A CTA sends row r+2's state only
// after its own barrier for row r+1 completed, which needed every peer's row
// r+1 state, sent after that peer had read its row r slots: so the parity
// double buffer is never overwritten while being read.
template <int CLUSTER>
struct ClusterExchange {
    uint64_t bar[2];
    float2 slot[2][CLUSTER];
};

template <int CLUSTER>
__device__ __forceinline__ void exchange_init(ClusterExchange<CLUSTER>& cx) {
    mbar_init(&cx.bar[0], 1);
    mbar_init(&cx.bar[1], 1);
}

// Called by all 32 lanes of one warp holding the CTA state in every lane.
template <int CLUSTER>
__device__ __forceinline__ void exchange_send(ClusterExchange<CLUSTER>& cx, float2 s, int parity,
                                              uint32_t rank) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) mbar_arrive_expect_tx(&cx.bar[parity], CLUSTER * 8);
    __syncwarp();
    if (lane < CLUSTER)
        st_async_b64(map_to_rank(&cx.slot[parity][rank], lane), __float_as_uint(s.x),
                     __float_as_uint(s.y), map_to_rank(&cx.bar[parity], lane));
}

// Waits for all CLUSTER states of this row (bounded; thread 0 polls, the
// others sleep in the CTA barrier), then folds them: lane l of each warp takes
// slot l % CLUSTER and the lanes merge in groups of CLUSTER, so every thread
// ends with the row's (m, d) after one exponential.
template <int CLUSTER>
__device__ __forceinline__ float2 exchange_receive(ClusterExchange<CLUSTER>& cx, int parity,
                                                   uint32_t use, const KernelCtl& ctl) {
    if (threadIdx.x == 0) mbar_wait_bounded(&cx.bar[parity], use & 1u, ctl);
    __syncthreads();
    float2 s = cx.slot[parity][(threadIdx.x & 31) % CLUSTER];
    group_merge<CLUSTER>(s.x, s.y);
    return s;
}

// ---------------------------------------------------------------------------
// tma_rows: persistent clusters with a ring of STAGES row slices in shared
// memory, filled by bulk copies (cp.async.bulk) STAGES-1 rows ahead of the row
// being computed, so HBM reads stay in flight while a row is reduced, merged
// and written.  Cluster `c` of G processes rows c, c+G, c+2G, ...; CTA `rank`
// of the cluster owns the contiguous slice [rank*S, rank*S + S) of every row
// (S = ceil(cols / CLUSTER) rounded up to whole 16-byte vectors).  A thread
// copies its EPT elements out of the stage into registers as e^(x - m_t)
// (one exponential per element), the stage is refilled with the row STAGES
// ahead, the (m, d) states are merged (shuffles, shared memory, st.async
// between the CTAs of the cluster), and the thread writes
// y = e^(x - m_t) * e^(m_t - m)/d from registers.
// Requires 16-byte aligned rows: x 16-byte aligned and cols*sizeof(TI) a
// multiple of 16 (so every slice starts and ends on a vector boundary).
template <typename TI, int THREADS, int EPT, int STAGES>
struct TmaRing {
    static constexpr int EPV = VecTraits<TI>::EPV;
    static constexpr int VPT = EPT / EPV;
    static constexpr int STAGE_BYTES = THREADS * EPT * int(sizeof(TI));
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES;
};

template <typename TI, typename TO, int THREADS, int EPT, int CLUSTER, int STAGES>
__global__ void __launch_bounds__(THREADS, 65536 / (THREADS * 128))
tma_rows_kernel(const TI* x, TO* y, int64_t rows, int cols,
                KernelCtl ctl) {
    using Ring = TmaRing<TI, THREADS, EPT, STAGES>;
    constexpr int EPV = Ring::EPV, VPT = Ring::VPT, NW = THREADS / 32;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ float2 warp_state[NW];
    __shared__ float2 cta_state[2];
    __shared__ int wait_flag[2];
    __shared__ __align__(8) ClusterExchange<CLUSTER> cx;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int slice = int(((int64_t(cols) + CLUSTER - 1) / CLUSTER + EPV - 1) / EPV * EPV);
    const int begin = int(rank) * slice;
    const int len = max(0, min(cols - begin, slice));
    const uint32_t bytes = uint32_t(len) * uint32_t(sizeof(TI));
    const int nvec = len / EPV;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        if (CLUSTER > 1) exchange_init(cx);
        mbar_init_fence();
    }
    if (CLUSTER > 1) cluster_sync(); else __syncthreads();

    // Producer (thread 0): loads issued into each stage.  After a wait gives
    // up, a thread stops waiting on the ring (its data for the rest of the
    // launch is garbage and the status word says so) and thread 0 stops issuing.
    int issued[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued[s] = 0;
    bool failed = false;
    auto issue = [&](int64_t local_row, int stage) {
        const int64_t row = cluster_id + local_row * nclusters;
        if (failed || row >= rows || bytes == 0) return;
        if (ctl.fault == kFaultSkipFirstLoad && local_row == 0 && blockIdx.x == 0) return;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_g2s(ring + stage * Ring::STAGE_BYTES, x + row * int64_t(cols) + begin, bytes,
                 &full[stage]);
        ++issued[stage];
    };
    if (tid == 0)
#pragma unroll
        for (int s = 0; s < STAGES; ++s) issue(s, s);

    int parity = 0;
    int64_t i = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, ++i, parity ^= 1) {
        const int stage = int(i % STAGES);
        if (!failed && bytes != 0)
            failed = !cta_wait_bounded(&full[stage], uint32_t((i / STAGES) & 1), ctl, wait_flag,
                                       int(i & 1));

        const unsigned char* src = ring + stage * Ring::STAGE_BYTES;
        float e[EPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * THREADS;
            if (v < nvec) {
                unpack(ld_shared_v4(src + v * 16), e + k * EPV, TI());
            } else {
#pragma unroll
                for (int q = 0; q < EPV; ++q) e[k * EPV + q] = kNegInf;
            }
        }
        const float m_t = max_of<EPT>(e);
        float m = m_t, d = exp_shift_sum<EPT>(e, m_t);
        group_merge<32>(m, d);
        if (lane == 0) warp_state[warp] = make_float2(m, d);
        __syncthreads();                                   // stage consumed, warp states ready
        if (tid == 0) issue(i + STAGES, stage);
        float2 md;
        if (warp == 0) {
            float2 s = lane < NW ? warp_state[lane] : make_float2(kNegInf, 0.f);
            group_merge<32>(s.x, s.y);
            if (CLUSTER > 1) exchange_send(cx, s, parity, rank);
            else if (lane == 0) cta_state[parity] = s;
        }
        if (CLUSTER > 1) {
            md = exchange_receive(cx, parity, uint32_t(i >> 1), ctl);
        } else {
            __syncthreads();
            md = cta_state[parity];
        }
        scale_all<EPT>(e, rescale(m_t, md.x) * (1.0f / md.y));
        TO* yr = y + row * int64_t(cols) + begin;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * THREADS;
            if (v < nvec) VecStore<TO, EPV>::run(yr + v * EPV, e + k * EPV);
        }
    }
    // Loads can be left in flight only after a wait gave up: wait for each
    // stage's last issued load (under the fixed drain bound, not the
    // caller's data-wait bound) so nothing lands after the CTA exits.
    if (tid == 0 && failed) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
            if (issued[s] > 0)
                mbar_wait_bounded_ns(&full[s], uint32_t((issued[s] - 1) & 1), kDrainTimeoutNs,
                                     ctl.err);
    }
    if (CLUSTER > 1) cluster_sync();  // no CTA leaves while a peer may still address it
}

// Chunks of a row that the streaming kernel keeps in shared memory between
// its passes: as many as fit in kStreamKeptBytesPerThread per thread, 96 KB
// for a CTA of 512 threads (two per SM), 48 KB for one of 256 (four per SM).
constexpr int kStreamKeptBytesPerThread = 192;
// Bytes per thread of a CTA's next row that it asks L2 to fetch when its
// second pass over the current row begins (that pass reads nothing from
// memory).  Measured on GB300 against none: fp32 rows with 512 threads 96 KB
// (4096x32000 0.1710 against 0.1785 ms), bf16 rows 32 KB with 512 threads
// (8192x128256 0.6783 against 0.6820 ms; more evicts what the second pass
// rereads from L2: 96 KB took 0.7503 ms) and 16 KB with 256 (bf16 16384
// columns 5614 against 5153 GB/s); fp32 rows with 256 threads (four CTAs
// per SM) none (16 KB was 2 % slower at 8193 and 24000 columns).
template <typename TI, int THREADS>
constexpr int stream_prefetch_bytes_per_thread() {
    return sizeof(TI) == 2 ? 64 : THREADS == 512 ? 192 : 0;
}
constexpr int kStreamPrefetchPiece = 16 * 1024;
template <typename TI, int THREADS, int UNROLL>
constexpr int stream_kept_chunks() { return kStreamKeptBytesPerThread / (UNROLL * 16); }

// ---------------------------------------------------------------------------
// Chunk arithmetic of the streaming kernel.  A chunk is UNROLL 16-byte
// vectors per thread, kept as raw words: bf16 inputs are never unpacked by
// shifts -- their maximum is taken on packed pairs (max.bf16x2) and x - m is
// formed by mixed-precision subtraction straight from the halves.
template <typename TI, int UNROLL>
struct Chunk {
    uint4 raw[UNROLL];
    static constexpr int EPV = VecTraits<TI>::EPV;

    __device__ __forceinline__ float max() const {
        if constexpr (sizeof(TI) == 2) {
            uint32_t w = raw[0].x;
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                if (k > 0) w = max_bf16x2(w, raw[k].x);
                w = max_bf16x2(w, raw[k].y);
                w = max_bf16x2(w, raw[k].z);
                w = max_bf16x2(w, raw[k].w);
            }
            return bf16x2_max_to_f32(w);
        } else {
            float m = __uint_as_float(raw[0].x);
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                m = max3(m, __uint_as_float(raw[k].x), __uint_as_float(raw[k].y));
                m = max3(m, __uint_as_float(raw[k].z), __uint_as_float(raw[k].w));
            }
            return m;
        }
    }

    // e[i] = x_i - m for the UNROLL * EPV elements (m = -inf: x_i itself)
    __device__ __forceinline__ void shifted(float m, float* e) const {
        m = finite_shift(m);
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
            if constexpr (sizeof(TI) == 2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 z = sub_bf16x2(w[i], m);
                    e[k * 8 + 2 * i] = z.x;
                    e[k * 8 + 2 * i + 1] = z.y;
                }
            } else {
                const float2 a = add2(make_float2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                      splat2(-m));
                const float2 b = add2(make_float2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                      splat2(-m));
                e[k * 4] = a.x;
                e[k * 4 + 1] = a.y;
                e[k * 4 + 2] = b.x;
                e[k * 4 + 3] = b.y;
            }
        }
    }

    // f(pair index, q) for the chunk's pairs, q = 2^((x - m) log2 e + 66)
    // (exp_biased_pair), m finite and every x <= m + 30.  PACKED (bf16
    // inputs, |m| < kPackedClampMaxAbs): each word is first clamped from
    // below at lo2 (packed_clamp_bound(m)) with one packed max, so x - m lies
    // in [-126, 30]; otherwise x - m is clamped at -110 in fp32.  Either way
    // a clamped entry (e^-inf included) comes out as exactly +0 once scaled.
    template <int DEG, bool PACKED, typename F>
    __device__ __forceinline__ void for_each_biased(float m, uint32_t lo2, F&& f) const {
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
            if constexpr (sizeof(TI) == 2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t v = PACKED ? max_bf16x2(w[i], lo2) : w[i];
                    f(k * 4 + i, exp_biased_pair<DEG, !PACKED>(sub_bf16x2(v, m)));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 z = add2(make_float2(__uint_as_float(w[2 * i]),
                                                      __uint_as_float(w[2 * i + 1])), splat2(-m));
                    f(k * 2 + i, exp_biased_pair<DEG, true>(z));
                }
            }
        }
    }

    // bf16 inputs, the shift folded into the exponential: f(pair index, q)
    // with q = 2^(x log2 e + c_int + 66) (exp_folded_pair with the constant k
    // of folded_shift(m)), each word first clamped from below at lo2
    // (packed_clamp_bound(m), |m| < kPackedClampMaxAbs) by one packed max.
    template <int DEG, typename F>
    __device__ __forceinline__ void for_each_folded(uint32_t lo2, float2 kk, F&& f) const {
        static_assert(sizeof(TI) == 2, "bf16 inputs");
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                f(k * 4 + i, exp_folded_pair<DEG>(unpack_bf16x2(max_bf16x2(w[i], lo2)), kk));
        }
    }

    template <int DEG>
    __device__ __forceinline__ float folded_sum(uint32_t lo2, float2 kk) const {
        float2 acc = make_float2(0.f, 0.f);
        for_each_folded<DEG>(lo2, kk, [&](int, float2 q) { acc = add2(acc, q); });
        return acc.x + acc.y;
    }

    template <int DEG>
    __device__ __forceinline__ void folded_scaled(uint32_t lo2, float2 kk, float2 scale,
                                                  float* e) const {
        for_each_folded<DEG>(lo2, kk, [&](int j, float2 q) {
            const float2 y = mul2(q, scale);
            e[2 * j] = y.x;
            e[2 * j + 1] = y.y;
        });
    }

    // Pass 1: the sum of q over the chunk.
    template <int DEG, bool PACKED>
    __device__ __forceinline__ float biased_sum(float m, uint32_t lo2) const {
        float2 acc = make_float2(0.f, 0.f);
        for_each_biased<DEG, PACKED>(m, lo2, [&](int, float2 q) { acc = add2(acc, q); });
        return acc.x + acc.y;
    }

    // Pass 2: e[2j], e[2j + 1] = q * scale, scale = 2^-66 / d.
    template <int DEG, bool PACKED>
    __device__ __forceinline__ void biased_scaled(float m, uint32_t lo2, float2 scale,
                                                  float* e) const {
        for_each_biased<DEG, PACKED>(m, lo2, [&](int j, float2 q) {
            const float2 y = mul2(q, scale);
            e[2 * j] = y.x;
            e[2 * j + 1] = y.y;
        });
    }
};

// Packed lower bound of bf16 inputs for a (finite) reference m: m - 118
// rounded to bf16 in both halves.  For |m| < kPackedClampMaxAbs the rounding
// moves it by at most 8, so the bound lies at x - m in [-126, -110]: above
// -132, where 2^((x - m) log2 e + 66) would leave the exponent range, and
// below -110, where e^(x - m) / d is under 2^-150 and the scaled result is +0.
constexpr float kPackedClampMaxAbs = 2048.0f;
__device__ __forceinline__ uint32_t packed_clamp_bound(float m) {
    return pack_bf16x2(m - 118.0f, m - 118.0f);
}

// How far a value may lie above a thread's pass-1 reference before the
// reference moves (e^30: sums of 2^((x - m) log2 e + 66) stay finite).
constexpr float kRefWindow = 30.0f;

// Which slots of a CTA's range [begin, begin + len) hold columns below a
// limit `lim` (the row length, or its causal limit): [lo, full) wholly,
// [0, lo) and [full, any) in part, none from `any` on.
struct VecLimits {
    int lo, full, any;
};
template <int EPV, bool ALIGNED = false>
__device__ __forceinline__ VecLimits vec_limits(int len, int begin, int lim, int head) {
    if constexpr (ALIGNED) {  // head = 0
        const int lim_v = int((int64_t(lim) + EPV - 1) / EPV);  // lim can be 2^31 - 1
        return {0, min(len, max(0, lim / EPV - begin)), min(len, max(0, lim_v - begin))};
    } else {  // in 64 bits: lim + head can pass 2^31
        const int64_t whole = (int64_t(lim) + head) / EPV;           // slots ending by lim
        const int64_t some = (int64_t(lim) + head + EPV - 1) / EPV;  // slots starting before lim
        auto rel = [&](int64_t u) { return int(min(int64_t(len), max(int64_t(0), u - begin))); };
        return {rel(head > 0 ? 1 : 0), rel(whole), rel(some)};
    }
}

// Slots t + k*GROUP (k < UNROLL) of chunk c of a CTA's range that starts at
// slot `begin` of a row; xs points at that slot's first element (16-byte
// aligned: the row start minus head, plus begin slots).  Columns at or past `lim` read
// as -inf; slots wholly inside [0, lim) are read with one 16-byte load, the
// rest element by element, slots wholly past lim not at all.  ALIGNED: the
// row starts on a 16-byte boundary (head = 0) and cols is a whole number of
// slots, so only causal limits leave partial slots.  Vector addresses are a
// per-row base plus 32-bit slot offsets (slot offsets stay below 2^31:
// (begin + v) EPV - head < cols + EPV).
template <typename TI, int GROUP, int UNROLL, bool ALIGNED>
__device__ __forceinline__ void load_stream_chunk(const TI* xs, int c, VecLimits vl, int begin,
                                                  int lim, int head, uint64_t policy,
                                                  Chunk<TI, UNROLL>& ch, int t) {
    constexpr int EPV = VecTraits<TI>::EPV, STEP = GROUP * UNROLL;
    const int v0 = c * STEP + t;
    const uint32_t neg_inf_word = sizeof(TI) == 2 ? 0xff80ff80u : 0xff800000u;
    if constexpr (ALIGNED) {
        const bool full = c * STEP + STEP <= vl.full;
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const int v = v0 + k * GROUP;
            if (full || v < vl.full) {
                ch.raw[k] = ld_coherent_policy_v4(xs + v * EPV, policy);
            } else if (v < vl.any) {  // the slot a causal limit cuts
                TI tmp[EPV];
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const int j = (begin + v) * EPV + q;
                    tmp[q] = j < lim ? xs[v * EPV + q] : from_f32<TI>(kNegInf);
                }
                ch.raw[k] = *reinterpret_cast<const uint4*>(tmp);
            } else {
                ch.raw[k] = make_uint4(neg_inf_word, neg_inf_word, neg_inf_word, neg_inf_word);
            }
        }
    } else {
        const bool full = c * STEP >= vl.lo && c * STEP + STEP <= vl.full;
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const int v = v0 + k * GROUP;
            if (full || (v >= vl.lo && v < vl.full)) {
                ch.raw[k] = ld_coherent_policy_v4(xs + v * EPV, policy);
            } else if (v < vl.any) {
                TI tmp[EPV];
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const int64_t j = int64_t(begin + v) * EPV + q - head;  // column
                    tmp[q] = j >= 0 && j < lim ? xs[int64_t(v) * EPV + q] : from_f32<TI>(kNegInf);
                }
                ch.raw[k] = *reinterpret_cast<const uint4*>(tmp);
            } else {
                ch.raw[k] = make_uint4(neg_inf_word, neg_inf_word, neg_inf_word, neg_inf_word);
            }
        }
    }
}

// Stores the UNROLL * EPV values e of chunk c (same slots as load_stream_chunk)
// through ys (slot `begin` of the output row): columns [0, cols) only; slots wholly inside by vector
// stores when `vec` (the output row has the input's block phase: the slot's
// first column is suitably aligned in y too), element by element otherwise.
template <typename TO, int THREADS, int UNROLL, int EPV, bool ALIGNED>
__device__ __forceinline__ void store_stream_chunk(TO* ys, int c, VecLimits vl, int begin,
                                                   int cols, int head, bool vec, const float* e) {
    constexpr int STEP = THREADS * UNROLL;
    const int v0 = c * STEP + int(threadIdx.x);
    if constexpr (ALIGNED) {  // every slot is whole: vl.full slots, all stored as vectors
        const bool full = c * STEP + STEP <= vl.full;
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const int v = v0 + k * THREADS;
            if (full || v < vl.full) VecStore<TO, EPV>::run(ys + v * EPV, e + k * EPV);
        }
    } else {
        const bool full = vec && c * STEP >= vl.lo && c * STEP + STEP <= vl.full;
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const int v = v0 + k * THREADS;
            if (full || (vec && v >= vl.lo && v < vl.full)) {
                VecStore<TO, EPV>::run(ys + v * EPV, e + k * EPV);
            } else if (v < vl.any) {
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const int64_t j = int64_t(begin + v) * EPV + q - head;
                    if (j >= 0 && j < cols) ys[int64_t(v) * EPV + q] = from_f32<TO>(e[k * EPV + q]);
                }
            }
        }
    }
}

// Slots per row: every row has the same number, that of the worst head.
template <int EPV, bool ALIGNED>
__device__ __forceinline__ int row_slots(int cols) {  // cols can be 2^31 - 1
    return int((int64_t(cols) + (ALIGNED ? EPV - 1 : 2 * EPV - 2)) / EPV);
}


// sum over N entries of e^(z_i), z given, on the SFU (statistics kernel)
template <int N, bool FAST>
__device__ __forceinline__ float exp_sum_z(const float* z) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < N; i += 2) acc = add2(acc, exp_pair<FAST>(make_float2(z[i], z[i + 1])));
    return acc.x + acc.y;
}

// Degree of the FMA-pipe exponential's 2^f fit by output type: 3 where the
// results are rounded to bf16, 5 for fp32 results.
template <typename TO> constexpr int exp_degree() { return sizeof(TO) == 2 ? 3 : 5; }

// sum over N entries of 2^(z_i log2 e + 66), z given (z <= 0): the streaming
// kernels' pass-1 sum before its one scale by 2^-66 (exp_biased_pair)
template <int N, int DEG>
__device__ __forceinline__ float exp_biased_sum(const float* z) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < N; i += 2) acc = add2(acc, exp_biased_pair<DEG>(make_float2(z[i], z[i + 1])));
    return acc.x + acc.y;
}

// y = e^z / d for the N entries of e[] (z in place): q = 2^(z log2 e + 66),
// times the row's scale 2^-66 / d.
template <int N, int DEG>
__device__ __forceinline__ void exp_scale_all(float* e, float2 scale) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 p = mul2(exp_biased_pair<DEG>(make_float2(e[i], e[i + 1])), scale);
        e[i] = p.x;
        e[i + 1] = p.y;
    }
}

// ---------------------------------------------------------------------------
// stream_rows: one CTA (or a cluster) per row, persistent over rows; CTA
// `rank` owns a contiguous range of vector slots and reads it twice.
// Pass 1 keeps a running (m, d) per thread with one rescale per chunk of
// UNROLL vectors; its loads ask L2 to keep the lines (evict_last) because
// pass 2 reads them again right after the merge.  Pass 2 walks the chunks in
// reverse order (the most recently read lines are the likeliest still in
// L2), marks its loads evict_first (last use) and writes y = e^(x - m) / d
// with streaming stores.  The row's first NS chunks (the ones pass 1 read
// longest ago, so the likeliest to have left L2) are also kept raw in shared
// memory by the thread that loaded them, and pass 2 takes them from there
// (bf16 rows on 512-thread CTAs read them with evict_first, see KEPT_FIRST).
// When pass 2 begins (it reads nothing from memory) the CTA asks L2 for the
// start of its next row, so that the next pass 1 finds it there and memory
// stays busy between the rows.
// With one CTA per row there is no exchange between SMs at all: each row
// costs one __syncthreads-level merge.
// Per-element exponentials (SFU = false): the FMA-pipe form exp_biased_pair
// (no ex2.approx): pass 1 sums a chunk's biased values and scales the sum
// once, pass 2 multiplies each by the row's 2^-66 / d (one product per
// element normalises and unbiases together); bf16 -> bf16 folds the shift
// into the rounding constant (exp_folded_pair).  SFU = true (bf16 results,
// AUTO's choice): the SFU's 2^x against a running maximum.
// Every slot wholly inside the row moves with one 128-bit load and store;
// ALIGNED (rows start on 16-byte boundaries and are whole slots) drops the
// per-row head and output-phase arithmetic.  Chunks lying wholly inside the
// row skip the per-slot range checks.
template <typename TI, typename TO, int THREADS, int UNROLL, int CLUSTER, bool ALIGNED, bool SFU>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2 > 0 ? 2048 / THREADS / 2 : 1)
stream_rows_kernel(const TI* x, TO* y, int64_t rows, int cols,
                   int64_t period, int64_t offset) {
    static_assert(!SFU || sizeof(TO) == 2, "the SFU form serves bf16 results only");
    constexpr int EPV = VecTraits<TI>::EPV, EPC = UNROLL * EPV;
    constexpr int DEG = exp_degree<TO>();             // output pass
    constexpr int DEG1 = sizeof(TO) == 2 ? 2 : DEG;   // normaliser sum
    constexpr bool FOLD = sizeof(TI) == 2 && sizeof(TO) == 2;  // bf16 -> bf16
    constexpr int STEP = THREADS * UNROLL;  // vectors per chunk
    constexpr int NS = stream_kept_chunks<TI, THREADS, UNROLL>();
    // bf16 rows on 512-thread CTAs read their kept chunks with evict_first:
    // pass 2 takes those from shared memory, and L2 (full with the rest of
    // the rows, their outputs and the prefetched next rows) keeps the lines
    // it does reread.  Measured on 8192x128256: 0.6663 against 0.6777 ms; the
    // same on fp32 rows was slower (4096x32000: 0.1734 against 0.1711 ms).
    constexpr bool KEPT_FIRST = sizeof(TI) == 2 && THREADS == 512;
    __shared__ RowMergeSmem<THREADS, CLUSTER> sm;
    extern __shared__ uint4 kept[];  // [NS][UNROLL][THREADS]: the row's first chunks, raw
    const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0;
    const int64_t cluster_id = blockIdx.x / CLUSTER, nclusters = gridDim.x / CLUSTER;
    const int nv = row_slots<EPV, ALIGNED>(cols);
    const int per_cta = (nv + CLUSTER - 1) / CLUSTER;
    const int begin = int(rank) * per_cta;
    const int len = max(0, min(per_cta, nv - begin));  // vectors of this CTA
    const int nchunks = (len + STEP - 1) / STEP;
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    if (CLUSTER > 1) cluster_sync();

    int parity = 0;
    for (int64_t row = cluster_id; row < rows; row += nclusters, parity ^= 1) {
        const TI* xr = x + row * int64_t(cols);
        TO* yr = y + row * int64_t(cols);
        const int head = ALIGNED ? 0 : row_head(xr);
        const bool yvec = ALIGNED || out_vec_ok<TO, EPV>(yr, head);
        const TI* xs = xr + (int64_t(begin) * EPV - head);  // the CTA's first slot
        TO* ys = yr + (int64_t(begin) * EPV - head);
        // columns at or past `lim` are masked (-inf, never read): chunks from
        // `live` on hold none of this CTA's unmasked columns
        const int lim = causal_limit(row, cols, period, offset);
        const VecLimits vl = vec_limits<EPV, ALIGNED>(len, begin, lim, head);
        // output slots: for aligned rows every one of the CTA's len slots is whole
        const VecLimits vo = ALIGNED ? VecLimits{0, len, len} : vec_limits<EPV, ALIGNED>(len, begin, cols, head);
        const int live = (vl.any + STEP - 1) / STEP;
        auto load_chunk = [&](int c, uint64_t policy, Chunk<TI, UNROLL>& ch) {
            load_stream_chunk<TI, THREADS, UNROLL, ALIGNED>(xs, c, vl, begin, lim, head, policy, ch,
                                                            int(threadIdx.x));
        };
        // pass 1: per thread a state (m, d) with d = sum e^(x - m) over the
        // elements seen.  m is a reference that moves (d rescaled once) only
        // when a chunk's maximum exceeds it by more than kRefWindow, which
        // after the first chunks is rare; the (+) merge takes any such state.
        float m = kNegInf, d = 0.f;
        float ms = 0.f;                               // finite_shift(m)
        uint32_t lo2 = packed_clamp_bound(0.f);       // bf16 inputs' packed clamp
        bool packed = sizeof(TI) == 2;                // |ms| < kPackedClampMaxAbs
        FoldedShift fs = {splat2(expc::kBiasedRound), expc::kUnbias};  // folded_shift(ms)
        auto fold_in = [&](const Chunk<TI, UNROLL>& ch, int c) {
            if (c < NS) {  // kept on chip for pass 2 (thread-private slots)
#pragma unroll
                for (int k = 0; k < UNROLL; ++k) kept[(c * UNROLL + k) * THREADS + threadIdx.x] = ch.raw[k];
            }
            const float cm = ch.max();
            if (__any_sync(kFullMask, cm > m + kRefWindow)) {  // warp-uniform branch
                if (cm > m + kRefWindow) {
                    d *= rescale(m, cm);  // m = -inf: d is 0 and stays 0
                    m = cm;
                    ms = cm;
                    lo2 = packed_clamp_bound(cm);
                    packed = sizeof(TI) == 2 && fabsf(cm) < kPackedClampMaxAbs;
                    if (FOLD && packed) fs = folded_shift(cm);
                }
            }
            if (__all_sync(kFullMask, packed)) {  // warp-uniform
                if constexpr (FOLD) d = fmaf(ch.template folded_sum<DEG1>(lo2, fs.k), fs.frac, d);
                else d = fmaf(ch.template biased_sum<DEG1, true>(ms, lo2), expc::kUnbias, d);
            } else {
                d = fmaf(ch.template biased_sum<DEG1, false>(ms, lo2), expc::kUnbias, d);
            }
        };
        // a warp whose slots of chunk c all lie past the row's last column
        // (the ragged last chunk) skips it in both passes
        const int warp_first = int(threadIdx.x) & ~31;
        for (int c = 0; c < live; ++c) {
            if (c * STEP + warp_first >= vl.any) break;  // warp-uniform; later chunks too
            Chunk<TI, UNROLL> ch;
            load_chunk(c, KEPT_FIRST && c < NS ? drop : keep, ch);
            if constexpr (SFU) {  // running maximum, one rescale per chunk, ex2 per element
                if (c < NS) {
#pragma unroll
                    for (int k = 0; k < UNROLL; ++k) kept[(c * UNROLL + k) * THREADS + threadIdx.x] = ch.raw[k];
                }
                const float m_new = fmaxf(m, ch.max());
                float z[EPC];
                ch.shifted(m_new, z);
                d = d * rescale(m, m_new) + exp_sum_z<EPC, true>(z);
                m = m_new;
            } else {
                fold_in(ch, c);
            }
        }
        const float2 md = merge_row_state<THREADS, CLUSTER>(sm, m, d, parity, rank);
        if constexpr (CLUSTER == 1) {
            // the start of this CTA's next row, asked of L2 in pieces (the
            // 16-byte aligned part of the row only)
            constexpr int NPF = THREADS * stream_prefetch_bytes_per_thread<TI, THREADS>() / kStreamPrefetchPiece;
            const int64_t next = row + nclusters;
            if (NPF > 0 && next < rows && int(threadIdx.x) < NPF) {
                const uintptr_t r0 = reinterpret_cast<uintptr_t>(x + next * int64_t(cols));
                const uintptr_t lo = (r0 + 15) & ~uintptr_t(15);
                const uintptr_t hi = (r0 + uintptr_t(cols) * sizeof(TI)) & ~uintptr_t(15);
                const uintptr_t a = lo + uintptr_t(threadIdx.x) * kStreamPrefetchPiece;
                if (a < hi)
                    bulk_prefetch_l2(reinterpret_cast<const void*>(a),
                                     uint32_t(min(uintptr_t(kStreamPrefetchPiece), hi - a)), keep);
            }
        }
        const float inv_d = 1.0f / md.y;
        const float2 scale = splat2(expc::kUnbias * inv_d);  // 2^-66 / d, exact product
        const float ms2 = finite_shift(md.x);
        const uint32_t lo2r = packed_clamp_bound(ms2);
        const bool packed2 = sizeof(TI) == 2 && fabsf(ms2) < kPackedClampMaxAbs;  // uniform
        FoldedShift fs2 = {splat2(expc::kBiasedRound), expc::kUnbias};
        if (FOLD && packed2) fs2 = folded_shift(ms2);
        const float2 fscale = splat2(fs2.frac * inv_d);  // 2^(c_frac - 66) / d
        const float neg_log2_d = SFU ? -__log2f(md.y) : 0.f;  // SFU: 2^(z log2 e - log2 d)
        // pass 2, last chunk first: y = e^(x - m) / d
        for (int c = nchunks - 1; c >= 0; --c) {
            if (c * STEP + warp_first >= vo.any) continue;  // nothing to load or store
            Chunk<TI, UNROLL> ch;
            // kept on chip only if this warp took part in chunk c in pass 1
            if (c < NS && c * STEP + warp_first < vl.any) {
#pragma unroll
                for (int k = 0; k < UNROLL; ++k) ch.raw[k] = kept[(c * UNROLL + k) * THREADS + threadIdx.x];
            } else {
                load_chunk(c, drop, ch);  // masked chunks: -inf without a load, written as 0
            }
            float e[EPC];
            if constexpr (SFU) {
                ch.shifted(md.x, e);
#pragma unroll
                for (int i = 0; i < EPC; i += 2) {
                    const float2 p = exp_pair_div(make_float2(e[i], e[i + 1]), neg_log2_d);
                    e[i] = p.x;
                    e[i + 1] = p.y;
                }
            } else if (packed2) {
                if constexpr (FOLD) ch.template folded_scaled<DEG>(lo2r, fs2.k, fscale, e);
                else ch.template biased_scaled<DEG, true>(ms2, lo2r, scale, e);
            } else {
                ch.template biased_scaled<DEG, false>(ms2, lo2r, scale, e);
            }
            store_stream_chunk<TO, THREADS, UNROLL, EPV, ALIGNED>(ys, c, vo, begin, cols, head, yvec, e);
        }
    }
}

// ---------------------------------------------------------------------------
// safe_rows: the three-pass "safe softmax" that the online normalizer
// replaces ("Online normalizer calculation for softmax" (notes), section 2;
// "5.2 CUDA Online Softmax", section 1.1): pass 1 the row maximum m, pass 2
// d = sum e^(x - m), pass 3 y = e^(x - m) / d, each pass reading the row from
// global memory with ordinary (L2-allocating) loads.  A measurement baseline
// (OS_PATH_SAFE), never chosen by AUTO.  One persistent CTA per row.
template <typename TI, typename TO, int THREADS, int UNROLL, bool ALIGNED, bool SFU>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2 > 0 ? 2048 / THREADS / 2 : 1)
safe_rows_kernel(const TI* x, TO* y, int64_t rows, int cols) {
    static_assert(!SFU || sizeof(TO) == 2, "the SFU form serves bf16 results only");
    constexpr int EPV = VecTraits<TI>::EPV, EPC = UNROLL * EPV, NW = THREADS / 32;
    constexpr int DEG = exp_degree<TO>();
    constexpr int STEP = THREADS * UNROLL;
    __shared__ float red[2][NW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int len = row_slots<EPV, ALIGNED>(cols);
    const int nchunks = (len + STEP - 1) / STEP;
    const uint64_t normal = l2_policy_evict_normal();
    int rb = 0;  // alternate reduction buffers: one barrier per reduction
    auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float t = __shfl_xor_sync(kFullMask, v, o);
            v = is_max ? fmaxf(v, t) : v + t;
        }
        if (lane == 0) red[rb][warp] = v;
        __syncthreads();
        float r = red[rb][0];
#pragma unroll
        for (int w = 1; w < NW; ++w) r = is_max ? fmaxf(r, red[rb][w]) : r + red[rb][w];
        rb ^= 1;
        return r;
    };
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const TI* xr = x + row * int64_t(cols);
        TO* yr = y + row * int64_t(cols);
        const int head = ALIGNED ? 0 : row_head(xr);
        const bool yvec = ALIGNED || out_vec_ok<TO, EPV>(yr, head);
        const VecLimits vl = vec_limits<EPV, ALIGNED>(len, 0, cols, head);
        const TI* xs = xr - head;  // the row's first slot
        TO* ys = yr - head;
        float m = kNegInf;
        for (int c = 0; c < nchunks; ++c) {  // pass 1: maximum
            Chunk<TI, UNROLL> ch;
            load_stream_chunk<TI, THREADS, UNROLL, ALIGNED>(xs, c, vl, 0, cols, head, normal, ch,
                                                            int(threadIdx.x));
            m = fmaxf(m, ch.max());
        }
        m = block_reduce(m, true);
        float d = 0.f;
        for (int c = 0; c < nchunks; ++c) {  // pass 2: normalizer
            Chunk<TI, UNROLL> ch;
            load_stream_chunk<TI, THREADS, UNROLL, ALIGNED>(xs, c, vl, 0, cols, head, normal, ch,
                                                            int(threadIdx.x));
            float z[EPC];
            ch.shifted(m, z);
            if constexpr (SFU) d += exp_sum_z<EPC, true>(z);
            else d += exp_biased_sum<EPC, DEG>(z) * expc::kUnbias;
        }
        d = block_reduce(d, false);
        const float2 scale = splat2(expc::kUnbias * (1.0f / d));
        const float neg_log2_d = SFU ? -__log2f(d) : 0.f;
        for (int c = 0; c < nchunks; ++c) {  // pass 3: outputs
            Chunk<TI, UNROLL> ch;
            load_stream_chunk<TI, THREADS, UNROLL, ALIGNED>(xs, c, vl, 0, cols, head, normal, ch,
                                                            int(threadIdx.x));
            float e[EPC];
            ch.shifted(m, e);
            if constexpr (SFU) {
#pragma unroll
                for (int i = 0; i < EPC; i += 2) {
                    const float2 p = exp_pair_div(make_float2(e[i], e[i + 1]), neg_log2_d);
                    e[i] = p.x;
                    e[i + 1] = p.y;
                }
            } else {
                exp_scale_all<EPC, DEG>(e, scale);
            }
            store_stream_chunk<TO, THREADS, UNROLL, EPV, ALIGNED>(ys, c, vl, 0, cols, head, yvec, e);
        }
    }
}

// ---------------------------------------------------------------------------
// stats_rows: the online normalizer's state of each row, without the
// normalisation ("Online normalizer calculation for softmax" (notes), section
// 3): m = max_j x_j and d = sum_j e^(x_j - m) in one read of the row, one
// rescale per chunk, then lse = m + ln d.  GROUP threads share a row: 32 (a
// warp per row, for rows of up to 32 x UNROLL vectors) or THREADS (the CTA).
// Outputs given as NULL are not written.
template <typename TI, int THREADS, int GROUP, int UNROLL, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
stats_rows_kernel(const TI* __restrict__ x, float* __restrict__ m_out, float* __restrict__ d_out,
                  float* __restrict__ lse_out, int64_t rows, int cols) {
    static_assert(GROUP == 32 || GROUP == THREADS, "a warp or the whole CTA per row");
    constexpr int EPV = VecTraits<TI>::EPV, EPC = UNROLL * EPV, STEP = GROUP * UNROLL;
    constexpr int GPC = THREADS / GROUP;  // rows in flight per CTA
    __shared__ RowMergeSmem<THREADS, 1> sm;
    const int t = int(threadIdx.x) % GROUP;
    const int64_t g0 = int64_t(blockIdx.x) * GPC + threadIdx.x / GROUP;
    const int64_t ng = int64_t(gridDim.x) * GPC;
    const int len = row_slots<EPV, ALIGNED>(cols);
    const int nchunks = (len + STEP - 1) / STEP;
    const uint64_t policy = l2_policy_evict_first();  // read once
    int parity = 0;
    for (int64_t row = g0; row < rows; row += ng, parity ^= 1) {  // uniform per group
        const TI* xr = x + row * int64_t(cols);
        const int head = ALIGNED ? 0 : row_head(xr);
        const VecLimits vl = vec_limits<EPV, ALIGNED>(len, 0, cols, head);
        float m = kNegInf, d = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            Chunk<TI, UNROLL> ch;
            load_stream_chunk<TI, GROUP, UNROLL, ALIGNED>(xr - head, c, vl, 0, cols, head, policy, ch, t);
            const float m_new = fmaxf(m, ch.max());
            float z[EPC];
            ch.shifted(m_new, z);
            d = d * rescale(m, m_new) + exp_sum_z<EPC, false>(z);
            m = m_new;
        }
        float2 md;
        if constexpr (GROUP == 32) {
            group_merge<32>(m, d);
            md = make_float2(m, d);
        } else {
            md = merge_row_state<THREADS, 1>(sm, m, d, parity, 0);
        }
        if (t == 0) {
            if (m_out) m_out[row] = md.x;
            if (d_out) d_out[row] = md.y;
            if (lse_out) lse_out[row] = md.x + logf(md.y);  // all -inf: -inf + -inf
        }
    }
}

}  // namespace os
