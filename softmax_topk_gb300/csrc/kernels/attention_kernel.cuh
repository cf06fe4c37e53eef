// attention_kernel.cuh -- attention forward, O = softmax(scale Q K^T) V with the
// per-row logsumexp, on the fifth-generation tensor cores.
//
// What it computes follows "6.2 FlashAttention V2" (section 6.1, forward
// algorithm): for one tile of 128 query rows of one (batch, head) the kernel
// walks the key/value tiles of 128 rows, keeping per query row the running
// maximum m, the running sum l and the unnormalised output; at the end it
// writes O = O~ / l and L = m + ln l.  The recurrence is the (m, d, o) one of
// the "Online normalizer calculation for softmax" notes (FlashAttention
// section): o is rescaled by e^(m_old - m_new) whenever the maximum moves.
// With the causal mask, query i sees keys j <= i and the key walk stops at the
// diagonal tile (section 5 of the same page).
//
// GB300 mapping (persistent CTAs, one per SM, 224 threads, warp-specialised;
// each CTA walks work units round-robin, see work_unit):
//   * warp 4 (one lane) streams the Q tile once and the K/V tiles through a
//     ring of STAGES buffers with TMA tiled loads (128-byte swizzle, rows past
//     the sequence end zero-filled by the copy engine);
//   * warp 5 (one lane) issues S_j = Q K_j^T (tcgen05.mma) into one of two
//     128-column fp32 accumulators in tensor memory;
//   * warp 6 (one lane) issues O += P_j V_j into a D-column accumulator that
//     stays in tensor memory for the whole walk.  The two products touch
//     disjoint tensor-memory columns, and with two issuers one keeps the
//     tensor pipe fed while the other waits on a barrier (the pipe queues
//     only about one instruction ahead of its issuer);
//   * warps 0-3 (the softmax warps) own one query row per thread, which is one
//     tensor-memory lane: they read S_j with tcgen05.ld, mask, update (m, l),
//     write P_j = 2^(S_j scale log2e - m) as packed bf16 pairs into tensor
//     memory with tcgen05.st (the A operand of the P V product is read from
//     there, so P never touches shared memory), and at the end normalise O.
// S_{j+1} is computed while the softmax warps work on S_j, and P_j V_j runs
// while they work on S_{j+1}; the next query tile's loads and first S
// products overlap the end of the current one.
//
// Rescaling differs from the pages' every-tile form: the exponent base m is
// only moved when a tile's maximum exceeds it by more than 2^8 (in the base-2
// exponent), so P stays <= 256 and the tensor-memory O is read and rewritten
// only on those (rare) tiles.  l and O always share one base, so O / l is the
// same quotient in exact arithmetic.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "../ctl.h"
#include "ops.cuh"
#include "umma.cuh"

namespace os {
namespace attn {

constexpr int kBM = 128;  // query rows per CTA (one per tensor-memory lane)
constexpr int kBN = 128;  // keys per tile
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarp = 4;
constexpr int kMmaSWarp = 5;
constexpr int kMmaPVWarp = 6;
constexpr int kThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS1 = 128;         // S accumulators at columns 0 and 128
constexpr uint32_t kTmemO = 256;          // O accumulator, D columns
constexpr uint32_t kTmemP = 384;          // P buffers at columns 384 and 448 (bf16 pairs)
constexpr float kRescaleLog2 = 8.0f;      // move the base when the max grows by more than 2^8
constexpr float kLn2 = 0.693147182f;

// Dynamic shared memory, 1024-byte aligned regions (the 128-byte swizzle
// repeats every 1024 bytes).  A Q/K/V tile is D/64 blocks of [128 rows][64
// bf16].
template <int D, int STAGES>
struct Layout {
    static constexpr int kBlock = kBM * 64 * 2;  // 16 KB
    static constexpr int kTile = kBM * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTile;            // STAGES buffers
    static constexpr int kV = kK + STAGES * kTile;   // STAGES buffers
    static constexpr int kBytes = kV + STAGES * kTile;
    static constexpr int kDynBytes = kBytes + 1024;
};

// Ring depth per head dimension: as deep as shared memory allows.
template <int D> struct Stages;
template <> struct Stages<128> { static constexpr int value = 3; };
template <> struct Stages<64> { static constexpr int value = 5; };

template <int STAGES>
struct Barriers {
    uint64_t q_full;
    uint64_t k_full[STAGES], v_full[STAGES];    // TMA landed (transaction bytes)
    uint64_t k_empty[STAGES], v_empty[STAGES];  // the MMAs reading the stage completed
    uint64_t s_full[2];               // S_j in tensor memory
    uint64_t p_full[2];               // P_j in tensor memory (128 arrivals)
    uint64_t pv_done[2];              // P_j V_j accumulated into O
    uint64_t q_empty;                 // the S products of an item have read its Q tile
    uint64_t o_empty;                 // the softmax warps have read an item's O (128 arrivals)
    uint32_t tmem;
};

// Work unit u of the persistent walk: one query tile (bh, qa) without the
// mask; with it the pair of query tiles qa = nq - 1 - p and qb = p of a slice
// (one tile when they coincide), so every unit walks nq + 1 key tiles and a
// static round-robin over units stays balanced.  Units go slice by slice, so
// the CTAs running together share their K/V tiles in L2.  Returns the number
// of query tiles in the unit.
__device__ __forceinline__ int work_unit(int u, int nq, bool causal, int& bh, int& qa, int& qb) {
    if (!causal) {
        bh = u / nq;
        qa = qb = u % nq;
        return 1;
    }
    const int pairs = (nq + 1) / 2;
    bh = u / pairs;
    const int p = u % pairs;
    qa = nq - 1 - p;
    qb = p;
    return qa == qb ? 1 : 2;
}

// 32 bytes to global memory in one store (p 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                    "r"(w[6]), "r"(w[7]) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, __nv_bfloat16* __restrict__ o,
                     float* __restrict__ lse, int n, int nq, int units, float scale_log2,
                     int causal, KernelCtl ctl) {
    static_assert(D == 64 || D == 128, "head dimension");
    constexpr int STAGES = Stages<D>::value;
    using L = Layout<D, STAGES>;
    extern __shared__ unsigned char dyn_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Barriers<STAGES> bars;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool masked = causal != 0;

    if (tid == 0) {
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        mbar_init(&bars.o_empty, kSoftmaxWarps * 32);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.p_full[s], kSoftmaxWarps * 32);
            mbar_init(&bars.pv_done[s], 1);
        }
        mbar_init_fence();
    }
    if (warp == 0) umma::tmem_alloc(&bars.tmem, kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = bars.tmem;

    // Every role walks the same items in the same order: units blockIdx.x,
    // blockIdx.x + gridDim.x, ...; within a unit its query tiles.  Barrier
    // phases follow item and key-tile counters that run across items, so the
    // next item's loads and S products start while this one finishes.
    if (warp == kLoadWarp) {
        // ---------------------------------------------------------------- loads
        if (lane == 0) {
            umma::prefetch_tensormap(&map_q);
            umma::prefetch_tensormap(&map_k);
            umma::prefetch_tensormap(&map_v);
            int g = 0, it = 0;  // key tiles and items so far
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                int bh, qa, qb;
                const int cnt = work_unit(u, nq, masked, bh, qa, qb);
                for (int e = 0; e < cnt; ++e, ++it) {
                    const int qi = e == 0 ? qa : qb;
                    const int ntiles = masked ? qi + 1 : nq;
                    // the Q buffer is free once the previous item's S products completed
                    if (it > 0) umma::mbar_wait(&bars.q_empty, (it - 1) & 1, ctl);
                    mbar_arrive_expect_tx(&bars.q_full, L::kTile);
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk)
                        umma::tma_load_3d(smem + L::kQ + blk * L::kBlock, &map_q, 64 * blk,
                                          qi * kBM, bh, &bars.q_full);
                    for (int j = 0; j < ntiles; ++j, ++g) {
                        const int st = g % STAGES;
                        const uint32_t reuse_parity = (g / STAGES - 1) & 1;
                        if (g >= STAGES) umma::mbar_wait(&bars.k_empty[st], reuse_parity, ctl);
                        mbar_arrive_expect_tx(&bars.k_full[st], L::kTile);
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            umma::tma_load_3d(smem + L::kK + st * L::kTile + blk * L::kBlock, &map_k,
                                              64 * blk, j * kBN, bh, &bars.k_full[st]);
                        if (g >= STAGES) umma::mbar_wait(&bars.v_empty[st], reuse_parity, ctl);
                        mbar_arrive_expect_tx(&bars.v_full[st], L::kTile);
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            umma::tma_load_3d(smem + L::kV + st * L::kTile + blk * L::kBlock, &map_v,
                                              64 * blk, j * kBN, bh, &bars.v_full[st]);
                    }
                }
            }
        }
    } else if (warp == kMmaSWarp) {
        // ---------------------------------------------------------------- S = Q K^T
        if (lane == 0) {
            constexpr uint32_t id_s = umma::idesc_bf16(kBM, kBN, false);
            const uint32_t q_addr = smem_addr(smem + L::kQ);
            int g = 0, it = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                int bh, qa, qb;
                const int cnt = work_unit(u, nq, masked, bh, qa, qb);
                for (int e = 0; e < cnt; ++e, ++it) {
                    const int qi = e == 0 ? qa : qb;
                    const int ntiles = masked ? qi + 1 : nq;
                    umma::mbar_wait(&bars.q_full, it & 1, ctl);
                    for (int j = 0; j < ntiles; ++j, ++g) {
                        const int st = g & 1, ks = g % STAGES;
                        // S buffer st is free once the softmax warps have turned
                        // S of key tile g - 2 into P
                        if (g >= 2) umma::mbar_wait(&bars.p_full[st], ((g - 2) >> 1) & 1, ctl);
                        umma::mbar_wait(&bars.k_full[ks], (g / STAGES) & 1, ctl);
                        umma::fence_after_sync();
                        const uint32_t k_addr = smem_addr(smem + L::kK + ks * L::kTile);
#pragma unroll
                        for (int s = 0; s < D / 16; ++s) {
                            const uint32_t koff = (s >> 2) * L::kBlock + (s & 3) * 32;
                            umma::mma_bf16(tmem + st * kTmemS1,
                                           umma::desc_sw128(q_addr + koff, 16, 1024),
                                           umma::desc_sw128(k_addr + koff, 16, 1024), id_s, s > 0);
                        }
                        umma::commit(&bars.s_full[st]);
                        umma::commit(&bars.k_empty[ks]);
                    }
                    umma::commit(&bars.q_empty);
                }
            }
        }
    } else if (warp == kMmaPVWarp) {
        // ---------------------------------------------------------------- O += P V
        // P from tensor memory (lane = query row, 16 keys per 8 columns), V
        // MN-major in shared memory (rows = keys)
        if (lane == 0) {
            constexpr uint32_t id_o = umma::idesc_bf16(kBM, D, true);
            int g = 0, it = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                int bh, qa, qb;
                const int cnt = work_unit(u, nq, masked, bh, qa, qb);
                for (int e = 0; e < cnt; ++e, ++it) {
                    const int qi = e == 0 ? qa : qb;
                    const int ntiles = masked ? qi + 1 : nq;
                    // O is overwritten by the item's first product: the softmax
                    // warps must have read the previous item's O
                    if (it > 0) umma::mbar_wait(&bars.o_empty, (it - 1) & 1, ctl);
                    for (int j = 0; j < ntiles; ++j, ++g) {
                        const int b = g & 1, vs = g % STAGES;
                        umma::mbar_wait(&bars.p_full[b], (g >> 1) & 1, ctl);
                        umma::mbar_wait(&bars.v_full[vs], (g / STAGES) & 1, ctl);
                        umma::fence_after_sync();
                        const uint32_t v_addr = smem_addr(smem + L::kV + vs * L::kTile);
#pragma unroll
                        for (int s = 0; s < kBN / 16; ++s) {
                            const uint64_t bd = umma::desc_sw128(v_addr + s * 2048, L::kBlock, 1024);
                            umma::mma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + 64 * b + 8 * s, bd,
                                                  id_o, j > 0 || s > 0);
                        }
                        umma::commit(&bars.pv_done[b]);
                        umma::commit(&bars.v_empty[vs]);
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax
        const int r = tid;  // row of the tile == tensor-memory lane
        const uint32_t lane_addr = tmem + (uint32_t(warp * 32) << 16);
        int g = 0, it = 0;  // key tiles and items so far
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int bh, qa, qb;
        const int cnt = work_unit(u, nq, masked, bh, qa, qb);
        for (int e = 0; e < cnt; ++e, ++it) {
        const int qi = e == 0 ? qa : qb;
        const int ntiles = masked ? qi + 1 : nq;
        const int row_q = qi * kBM + r;
        float m = -INFINITY;  // exponent base, base-2 units of the scaled scores
        float l = 0.f;
        for (int j = 0; j < ntiles; ++j, ++g) {
            const int st = g & 1;
            umma::mbar_wait(&bars.s_full[st], (g >> 1) & 1, ctl);
            umma::fence_after_sync();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) umma::tmem_ld32(lane_addr + st * kTmemS1 + 32 * c, s + 32 * c);
            umma::tmem_wait_ld();

            // keys past the sequence end, and under the mask keys after the query
            int lim = min(kBN, n - j * kBN);
            if (causal) lim = min(lim, row_q - j * kBN + 1);
            if (lim < kBN) {
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c >= lim) s[c] = -INFINITY;
            }
            // P = 2^(s scale log2e - m): fp32 values summed into l, bf16 pairs
            // (even key in the low half) for tensor memory.  Once a base m
            // exists the exponentials are taken against it speculatively,
            // with the tile maximum folded into the same pass (eight chains of
            // three-input maxima hidden under the SFU work); only a warp in
            // which some row's maximum outgrew its base by more than 2^8 does
            // the pass again with the new bases.
            uint32_t pk[kBN / 2];
            auto exp_pass = [&](float base, bool want_max, float& mt) {
                const float2 sl2 = splat2(scale_log2), nb2 = splat2(-base);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                float mx[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) {
                    if (want_max) mx[c & 7] = max3(mx[c & 7], s[2 * c], s[2 * c + 1]);
                    const float2 z = fma2(make_float2(s[2 * c], s[2 * c + 1]), sl2, nb2);
                    const float2 p = make_float2(ex2_sfu(z.x), ex2_sfu(z.y));
                    acc[c & 3] = add2(acc[c & 3], p);
                    pk[c] = pack_bf16x2(p.x, p.y);
                }
                if (want_max)
                    mt = fmaxf(max3(mx[0], mx[1], mx[2]),
                               fmaxf(max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) +
                       (acc[3].x + acc[3].y);
            };
            float mt = -INFINITY, lsum = 0.f;
            bool grow;
            const bool speculate = __all_sync(kFullMask, m != -INFINITY);
            if (speculate) {
                lsum = exp_pass(m, true, mt);
                grow = mt * scale_log2 > m + kRescaleLog2;  // scale > 0
            } else {
                float mx[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) mx[a] = s[a];
#pragma unroll
                for (int c = 8; c < kBN; c += 16) {
#pragma unroll
                    for (int a = 0; a < 8; ++a)
                        mx[a] = max3(mx[a], s[c + a], s[c + 8 + a < kBN ? c + 8 + a : c + a]);
                }
                mt = fmaxf(max3(mx[0], mx[1], mx[2]),
                           fmaxf(max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                grow = true;  // every row takes a new base (a row still at -inf keeps it)
            }
            const float mt2 = mt * scale_log2;
            grow = grow && mt2 > m;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2_sfu(m - mt2);  // +0 when m = -inf
                l *= alpha;
                m = mt2;
            }
            if (__any_sync(kFullMask, grow) || !speculate) {  // without a base: the pass runs once
                float unused;
                lsum = exp_pass(m == -INFINITY ? 0.f : m, false, unused);
                // tcgen05.ld/st are warp-collective: the warp rescales its O
                // rows (rows that kept their base multiply by 1)
                if (j > 0) {
                    umma::mbar_wait(&bars.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, ctl);
                    umma::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float t[32];
                        umma::tmem_ld32(lane_addr + kTmemO + 32 * c, t);
                        umma::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) t[e] *= alpha;
                        umma::tmem_st32(lane_addr + kTmemO + 32 * c, t);
                    }
                }
            }
            l += lsum;
            // the P buffer was last read by the P V product of key tile g - 2
            // (possibly of the previous item)
            if (g >= 2) umma::mbar_wait(&bars.pv_done[st], ((g - 2) >> 1) & 1, ctl);
            umma::tmem_st32(lane_addr + kTmemP + 64 * st, reinterpret_cast<const float*>(pk));
            umma::tmem_st32(lane_addr + kTmemP + 64 * st + 32, reinterpret_cast<const float*>(pk + 32));
            umma::tmem_wait_st();
            umma::fence_before_sync();
            umma::mbar_arrive(&bars.p_full[st]);
        }

        // ---------------------------------------------------------------- epilogue
        // O read into registers, then released to the next item's first P V
        // product before it is normalised and stored
        const int last = g - 1;
        umma::mbar_wait(&bars.pv_done[last & 1], (last >> 1) & 1, ctl);
        umma::fence_after_sync();
        float ov[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) umma::tmem_ld32(lane_addr + kTmemO + 32 * c, ov + 32 * c);
        umma::tmem_wait_ld();
        umma::fence_before_sync();
        umma::mbar_arrive(&bars.o_empty);
        const float inv_l = 1.f / l;
        if (row_q < n) {
            // one row per thread: 32-byte stores when O is 32-byte aligned
            // (rows are D * 2 bytes, so then every row is), else 16-byte ones;
            // each warp-wide store touches 32 rows, so fewer, wider stores
            // shorten this tail of the item
            __nv_bfloat16* orow = o + (int64_t(bh) * n + row_q) * D;
            if ((reinterpret_cast<uintptr_t>(o) & 31) == 0) {
#pragma unroll
                for (int v = 0; v < D / 16; ++v) {
                    uint32_t w[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        w[c] = pack_bf16x2(ov[16 * v + 2 * c] * inv_l, ov[16 * v + 2 * c + 1] * inv_l);
                    st_global_v8(orow + 16 * v, w);
                }
            } else {
#pragma unroll
                for (int v = 0; v < D / 8; ++v) {
                    uint4 w;
                    w.x = pack_bf16x2(ov[8 * v + 0] * inv_l, ov[8 * v + 1] * inv_l);
                    w.y = pack_bf16x2(ov[8 * v + 2] * inv_l, ov[8 * v + 3] * inv_l);
                    w.z = pack_bf16x2(ov[8 * v + 4] * inv_l, ov[8 * v + 5] * inv_l);
                    w.w = pack_bf16x2(ov[8 * v + 6] * inv_l, ov[8 * v + 7] * inv_l);
                    *reinterpret_cast<uint4*>(orow + 8 * v) = w;
                }
            }
            if (lse) lse[int64_t(bh) * n + row_q] = (m + __log2f(l)) * kLn2;
        }
        }  // query tiles of the unit
        }  // units
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace attn
}  // namespace os
