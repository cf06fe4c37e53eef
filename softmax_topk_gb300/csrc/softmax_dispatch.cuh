// softmax_dispatch.cuh -- kernel choice and launch for one (input, output) dtype
// pair.  Included by one translation unit per pair, which instantiates it.
//
// Families by row length, in 16-byte input vectors nv = ceil(cols / EPV);
// AUTO takes WARP for nv <= 256 fp32 / 128 bf16, ONCHIP for nv <= 2048 fp32
// / 1024 bf16 vectors, STREAM beyond:
//   WARP    nv <= 256: L = 1..32 lanes per row with 4 vectors per lane, or 32
//           lanes with 8 vectors (rows of up to 1024 fp32 / 2048 bf16).
//   ONCHIP  nv <= 16 x 512 x VPT (VPT = 32 elements per thread / EPV).
//           * rows longer than 8192 elements whose rows start on 16-byte
//             boundaries: the persistent bulk-copy ring (tma_rows), one CTA
//             or a cluster of 2..16 CTAs of 256 threads per row (32 fp32 or
//             64 bf16 elements per thread: a 32 KB slice per CTA, two CTAs per
//             SM), with row slices prefetched 2 rows ahead in shared memory;
//           * otherwise the register kernel (onchip_rows): one CTA of
//             128/256/512 threads, or a cluster of 512-thread CTAs, per row.
//           Rows of up to 262144 fp32 / 524288 bf16 (16-CTA clusters only
//           where the device can schedule them).
//   STREAM  anything longer: one CTA per row when there are at least as many
//           rows as SMs (CTAs of 256 threads, four per SM, for rows of up to
//           96 KB; of 512 threads, two per SM, beyond), else a cluster of 8
//           CTAs of 512 threads per row.
//   SAFE    the three-pass safe softmax, as a measurement baseline only.
// "5.2 CUDA Online Softmax" (sections 6.3 and 8.3) makes the same split on
// its hardware: the register-cached single read (V3) for short rows, the
// two-pass kernel (V2/V4) beyond the register budget.
#pragma once

#include "host_common.h"
#include "kernels/softmax_kernels.cuh"

namespace os {

constexpr int kWarpThreads = 256;
constexpr int kOnchipThreadsMax = 512;
constexpr int kOnchipElemsPerThread = 32;
constexpr int kStreamThreads = 512;
// Rows of at most this many input bytes stream through CTAs of
// kStreamThreadsShort threads: four rows in flight per SM instead of two,
// each kept on chip whole up to 48 KB.  Measured on GB300 (4096 rows, CUDA
// events): fp32 24000 columns 6030 against 4706 GB/s, bf16 24000 5263
// against 4592; from 128 KB rows on the 512-thread CTAs are as fast or faster.
constexpr int kStreamThreadsShort = 256;
constexpr int64_t kStreamShortRowBytes = 96 * 1024;
// vectors per thread per chunk: 8 fp32 or 4 bf16 (32 elements either way; measured best)
template <typename TI> constexpr int stream_unroll() { return sizeof(TI) == 4 ? 8 : 4; }
constexpr int kTmaMinCols = 8192;
// AUTO sends rows longer than this many 16-byte vectors (8192 elements of
// either dtype) to the two-pass streaming kernel: measured on GB300 (1 GB
// inputs) the register kernel wins up to there with CTAs of at most 256
// threads (fp32 8192 columns: 7146 against 6413 GB/s; bf16 8192: 6704
// against 6432; bf16 6000: 5585 against 5230), the streaming kernel beyond
// (fp32 8193: 4689 against 3437 with a 512-thread CTA; bf16 8193: 4098
// against 1593; the bulk-copy ring kernel 3780-5465 GB/s on fp32 rows of
// 10000-16384 columns against the streaming kernel's 4497-6342).
template <typename TI> constexpr int64_t auto_onchip_max_vectors() { return sizeof(TI) == 4 ? 2048 : 1024; }
// AUTO's WARP family: rows of up to 256 fp32 / 128 bf16 vectors (1024
// elements either way: 32 per thread); longer bf16 rows run the register
// kernel with 128-thread CTAs (2048 columns: 4673 against 3340 GB/s).
template <typename TI> constexpr int64_t auto_warp_max_vectors() { return sizeof(TI) == 4 ? 256 : 128; }
// The bulk-copy ring kernel runs CTAs of 256 threads, two per SM, so one
// CTA's reductions and exchange overlap the other's loads and arithmetic.
// Elements per thread: 32 fp32 or 64 bf16, so a CTA's slice is 32 KB of input
// either way and its 3-stage ring 96 KB.
constexpr int kTmaThreads = 256;
template <typename TI> constexpr int tma_ept() { return sizeof(TI) == 4 ? 32 : 64; }

template <typename TI, typename TO>
struct SoftmaxFamily {
    using Kernel = void (*)(const TI*, TO*, int64_t, int, int);
    using WarpKernel = void (*)(const TI*, TO*, int64_t, int, int, int64_t, int64_t);
    using TmaKernel = void (*)(const TI*, TO*, int64_t, int, KernelCtl);
    static constexpr int EPV = VecTraits<TI>::EPV;
    static constexpr int VPT = kOnchipElemsPerThread / EPV;
    static constexpr int TMA_STAGES = 3;
    static constexpr int TMA_EPT = tma_ept<TI>();
    using Ring = TmaRing<TI, kTmaThreads, TMA_EPT, TMA_STAGES>;

    // PEEL: rows that are not all 16-byte aligned whole vectors move as the
    // 16-byte blocks they cover (see warp_rows_kernel)
    template <bool PEEL>
    static WarpKernel warp_as(int lanes, int vpt) {
        if (vpt == 8) {
            switch (lanes) {
                case 4: return warp_rows_kernel<TI, TO, 4, 8, kWarpThreads, PEEL>;
                case 8: return warp_rows_kernel<TI, TO, 8, 8, kWarpThreads, PEEL>;
                case 16: return warp_rows_kernel<TI, TO, 16, 8, kWarpThreads, PEEL>;
                default: return warp_rows_kernel<TI, TO, 32, 8, kWarpThreads, PEEL>;
            }
        }
        switch (lanes) {
            case 1: return warp_rows_kernel<TI, TO, 1, 4, kWarpThreads, PEEL>;
            case 2: return warp_rows_kernel<TI, TO, 2, 4, kWarpThreads, PEEL>;
            case 4: return warp_rows_kernel<TI, TO, 4, 4, kWarpThreads, PEEL>;
            case 8: return warp_rows_kernel<TI, TO, 8, 4, kWarpThreads, PEEL>;
            case 16: return warp_rows_kernel<TI, TO, 16, 4, kWarpThreads, PEEL>;
            default: return warp_rows_kernel<TI, TO, 32, 4, kWarpThreads, PEEL>;
        }
    }
    static WarpKernel warp(int lanes, int vpt, bool peel = false) {
        return peel ? warp_as<true>(lanes, vpt) : warp_as<false>(lanes, vpt);
    }
    template <bool PEEL>
    static Kernel onchip_as(int threads, int cluster) {
        if (cluster == 1) {
            switch (threads) {
                case 128: return onchip_rows_kernel<TI, TO, 128, VPT, 1, PEEL>;
                case 256: return onchip_rows_kernel<TI, TO, 256, VPT, 1, PEEL>;
                default: return onchip_rows_kernel<TI, TO, 512, VPT, 1, PEEL>;
            }
        }
        switch (cluster) {
            case 2: return onchip_rows_kernel<TI, TO, 512, VPT, 2, PEEL>;
            case 4: return onchip_rows_kernel<TI, TO, 512, VPT, 4, PEEL>;
            case 8: return onchip_rows_kernel<TI, TO, 512, VPT, 8, PEEL>;
            default: return onchip_rows_kernel<TI, TO, 512, VPT, 16, PEEL>;
        }
    }
    static Kernel onchip(int threads, int cluster, bool peel = false) {
        return peel ? onchip_as<true>(threads, cluster) : onchip_as<false>(threads, cluster);
    }
    static TmaKernel tma(int cluster) {
        constexpr int T = kTmaThreads, E = TMA_EPT, S = TMA_STAGES;
        switch (cluster) {
            case 1: return tma_rows_kernel<TI, TO, T, E, 1, S>;
            case 2: return tma_rows_kernel<TI, TO, T, E, 2, S>;
            case 4: return tma_rows_kernel<TI, TO, T, E, 4, S>;
            case 8: return tma_rows_kernel<TI, TO, T, E, 8, S>;
            default: return tma_rows_kernel<TI, TO, T, E, 16, S>;
        }
    }
    static constexpr int STREAM_UNROLL = stream_unroll<TI>();
    using SafeKernel = void (*)(const TI*, TO*, int64_t, int);
    using StreamKernel = void (*)(const TI*, TO*, int64_t, int, int64_t, int64_t);
    // bf16 results take the SFU exponential in STREAM (and in the SAFE
    // baseline measured against it); STREAM_POLY and fp32 results the
    // library's FMA-pipe exponential
    static constexpr bool SFU_DEFAULT = sizeof(TO) == 2;
    static SafeKernel safe(bool aligned) {
        constexpr int T = kStreamThreads, U = STREAM_UNROLL;
        return aligned ? safe_rows_kernel<TI, TO, T, U, true, SFU_DEFAULT>
                       : safe_rows_kernel<TI, TO, T, U, false, SFU_DEFAULT>;
    }
    static constexpr int stream_smem_bytes(int threads) {
        return stream_kept_chunks<TI, kStreamThreads, STREAM_UNROLL>() * threads * STREAM_UNROLL * 16;
    }
    // threads 256 (cluster 1 only) or 512
    template <bool SFU>
    static StreamKernel streaming_as(int threads, int cluster, bool aligned) {
        constexpr int T = kStreamThreads, TS = kStreamThreadsShort, U = STREAM_UNROLL;
        if (threads == TS)
            return aligned ? stream_rows_kernel<TI, TO, TS, U, 1, true, SFU>
                           : stream_rows_kernel<TI, TO, TS, U, 1, false, SFU>;
        if (aligned)
            return cluster == 1 ? stream_rows_kernel<TI, TO, T, U, 1, true, SFU>
                                : stream_rows_kernel<TI, TO, T, U, 8, true, SFU>;
        return cluster == 1 ? stream_rows_kernel<TI, TO, T, U, 1, false, SFU>
                            : stream_rows_kernel<TI, TO, T, U, 8, false, SFU>;
    }
    static StreamKernel streaming(int threads, int cluster, bool aligned, bool poly = false) {
        if (poly || !SFU_DEFAULT) return streaming_as<false>(threads, cluster, aligned);
        return streaming_as<SFU_DEFAULT>(threads, cluster, aligned);
    }

    // Largest cluster size of the ONCHIP family the current device can run.
    static int onchip_cluster_limit(const DeviceInfo& dev) {
        static int cache[64] = {0};
        int& c = cache[dev.device & 63];
        if (c == 0) {
            const bool reg16 = max_active_clusters(onchip(512, 16), 512, 16) > 0;
            const bool tma16 = max_active_clusters(tma(16), kTmaThreads, 16, Ring::SMEM_BYTES) > 0;
            c = reg16 && tma16 ? 16 : 8;
        }
        return c;
    }

    // Clusters of the bulk-copy ring kernel resident at once (its persistent grid).
    static int tma_resident_clusters(const DeviceInfo& dev, int cluster) {
        static int cache[64][5] = {{0}};
        const int slot = cluster == 1 ? 0 : cluster == 2 ? 1 : cluster == 4 ? 2 : cluster == 8 ? 3 : 4;
        int& c = cache[dev.device & 63][slot];
        if (c == 0) {
            if (cluster == 1) {
                c = blocks_per_sm(tma(1), kTmaThreads, Ring::SMEM_BYTES) * dev.sms;
            } else {
                c = max_active_clusters(tma(cluster), kTmaThreads, cluster, Ring::SMEM_BYTES);
            }
            if (c <= 0) c = -1;
        }
        return c;
    }

    // `aligned`: x and y 16-byte aligned (then rows are aligned iff cols is a
    // multiple of the vector width).
    static os_status plan(int64_t rows, int64_t cols, os_path path, bool aligned, os_plan* p) {
        const DeviceInfo* dev = device_info();
        if (!dev) return OS_ERR_CUDA;
        // vector slots a row needs: one more for rows that are not 16-byte
        // aligned whole vectors, whose first and last blocks are partial
        const int64_t nv = (aligned && cols % EPV == 0) ? ceil_div(cols, EPV)
                                                        : ceil_div(cols + EPV - 1, EPV);
        const bool warp_ok = nv <= 256;
        const int64_t cta_cap = int64_t(kOnchipThreadsMax) * VPT;
        const bool onchip_ok = nv <= int64_t(onchip_cluster_limit(*dev)) * cta_cap;
        if (path == OS_PATH_AUTO)
            path = nv <= auto_warp_max_vectors<TI>() ? OS_PATH_WARP
                 : (nv <= auto_onchip_max_vectors<TI>() && onchip_ok) ? OS_PATH_ONCHIP : OS_PATH_STREAM;
        os_plan q = {};
        q.path = path;
        switch (path) {
            case OS_PATH_WARP: {
                if (!warp_ok) return OS_ERR_PATH;
                // 32 elements per thread where the row allows it: fp32 rows of
                // 32-256 vectors take 8 vectors per thread (measured on GB300,
                // 1048576x128: 6460 against 6060 GB/s with 4), bf16 rows 4
                // (8 measured far slower: 64 values per thread)
                q.vectors_per_thread = nv > 128 || (sizeof(TI) == 4 && nv >= 32) ? 8 : 4;
                q.lanes_per_row = pow2_at_least(ceil_div(nv, q.vectors_per_thread));
                q.threads = kWarpThreads;
                q.cluster = 1;
                const int64_t rows_per_cta = kWarpThreads / q.lanes_per_row;
                const int occ = blocks_per_sm(warp(q.lanes_per_row, q.vectors_per_thread,
                                                   !(aligned && cols % EPV == 0)),
                                              kWarpThreads);
                q.grid = min64(ceil_div(rows, rows_per_cta), int64_t(dev->sms) * (occ > 0 ? occ : 1));
                break;
            }
            case OS_PATH_ONCHIP: {
                if (!onchip_ok) return OS_ERR_PATH;
                q.vectors_per_thread = VPT;
                const bool rows_aligned = aligned && cols % EPV == 0;
                const int64_t tma_cap = int64_t(kTmaThreads) * TMA_EPT / EPV;
                if (rows_aligned && cols > kTmaMinCols &&
                    nv <= int64_t(onchip_cluster_limit(*dev)) * tma_cap) {
                    q.threads = kTmaThreads;
                    q.vectors_per_thread = TMA_EPT / EPV;
                    q.cluster = pow2_at_least(ceil_div(nv, tma_cap));
                    const int resident = tma_resident_clusters(*dev, q.cluster);
                    if (resident > 0) {
                        q.stages = TMA_STAGES;
                        q.grid = min64(rows, resident) * q.cluster;
                        break;
                    }
                }
                q.vectors_per_thread = VPT;
                if (nv <= cta_cap) {
                    q.cluster = 1;
                    q.threads = nv <= 128 * VPT ? 128 : nv <= 256 * VPT ? 256 : 512;
                } else {
                    q.cluster = pow2_at_least(ceil_div(nv, cta_cap));
                    q.threads = kOnchipThreadsMax;
                }
                q.grid = min64(rows, kMaxClustersPerLaunch) * q.cluster;
                break;
            }
            case OS_PATH_STREAM:
            case OS_PATH_STREAM_POLY: {
                q.vectors_per_thread = STREAM_UNROLL;
                q.cluster = rows >= int64_t(dev->sms) ? 1 : 8;  // measured: 1 CTA per row wins from one row per SM up
                q.threads = q.cluster == 1 && cols * int64_t(sizeof(TI)) <= kStreamShortRowBytes
                    ? kStreamThreadsShort : kStreamThreads;
                {
                    const int occ = blocks_per_sm(streaming(q.threads, q.cluster, true), q.threads,
                                                  stream_smem_bytes(q.threads));
                    const int64_t resident = q.cluster == 1
                        ? int64_t(dev->sms) * (occ > 0 ? occ : 1)
                        : kMaxClustersPerLaunch;
                    q.grid = min64(rows, resident) * q.cluster;
                }
                break;
            }
            case OS_PATH_SAFE: {
                q.threads = kStreamThreads;
                q.vectors_per_thread = STREAM_UNROLL;
                q.cluster = 1;
                const int occ = blocks_per_sm(safe(true), kStreamThreads);
                q.grid = min64(rows, int64_t(dev->sms) * (occ > 0 ? occ : 1));
                break;
            }
            default:
                return OS_ERR_PATH;
        }
        *p = q;
        return OS_OK;
    }

    // period > 0: causal mask (columns c > (row mod period) + offset masked);
    // only the WARP and STREAM families take one.
    static cudaError_t launch(const os_plan& p, const void* x, void* y, int64_t rows, int cols,
                              bool aligned, int64_t period, int64_t offset, const KernelCtl& ctl,
                              cudaStream_t stream) {
        const TI* xi = static_cast<const TI*>(x);
        TO* yo = static_cast<TO*>(y);
        if (p.path == OS_PATH_ONCHIP && p.stages > 0) {
            TmaKernel k = tma(p.cluster);
            if (!prepare_kernel(k, p.cluster, Ring::SMEM_BYTES)) return cudaErrorInvalidValue;
            return launch_kernel(k, p.grid, p.threads, p.cluster, Ring::SMEM_BYTES, stream, xi, yo,
                                 rows, cols, ctl);
        }
        if (p.path == OS_PATH_SAFE) {
            SafeKernel k = safe(aligned);
            if (!prepare_kernel(k, 1, 0)) return cudaErrorInvalidValue;
            return launch_kernel(k, p.grid, p.threads, 1, 0, stream, xi, yo, rows, cols);
        }
        if (p.path == OS_PATH_STREAM || p.path == OS_PATH_STREAM_POLY) {
            StreamKernel k = streaming(p.threads, p.cluster, aligned, p.path == OS_PATH_STREAM_POLY);
            const int smem = stream_smem_bytes(p.threads);
            if (!prepare_kernel(k, p.cluster, smem)) return cudaErrorInvalidValue;
            return launch_kernel(k, p.grid, p.threads, p.cluster, smem, stream, xi, yo, rows, cols,
                                 period, offset);
        }
        if (p.path == OS_PATH_WARP) {
            WarpKernel k = warp(p.lanes_per_row, p.vectors_per_thread, !aligned);
            if (!prepare_kernel(k, 1, 0)) return cudaErrorInvalidValue;
            return launch_kernel(k, p.grid, p.threads, 1, 0, stream, xi, yo, rows, cols,
                                 aligned ? 1 : 0, period, offset);
        }
        Kernel k = onchip(p.threads, p.cluster, !aligned);
        if (!prepare_kernel(k, p.cluster, 0)) return cudaErrorInvalidValue;
        return launch_kernel(k, p.grid, p.threads, p.cluster, 0, stream, xi, yo, rows, cols,
                             aligned ? 1 : 0);
    }
};

}  // namespace os

// One translation unit per dtype pair defines these two entry points.
#define OS_DEFINE_SOFTMAX_PAIR(NAME, TI, TO)                                                   \
    namespace os {                                                                             \
    os_status plan_softmax_##NAME(int64_t rows, int64_t cols, os_path path, bool aligned,      \
                                  os_plan* p) {                                                \
        return SoftmaxFamily<TI, TO>::plan(rows, cols, path, aligned, p);                      \
    }                                                                                          \
    cudaError_t launch_softmax_##NAME(const os_plan& p, const void* x, void* y, int64_t rows,  \
                                      int cols, bool aligned, int64_t period, int64_t offset,  \
                                      const KernelCtl& ctl, cudaStream_t stream) {             \
        return SoftmaxFamily<TI, TO>::launch(p, x, y, rows, cols, aligned, period, offset, ctl, \
                                             stream);                                          \
    }                                                                                          \
    }
