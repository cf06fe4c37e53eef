// ops.cuh -- device building blocks shared by the softmax and TopK kernels.
//
//  * packed fp32 pair arithmetic (the sm_100-family f32x2 FMA/ADD/MUL forms),
//  * exponentials: the library's own FMA-pipe fp32 exponential and the SFU's ex2,
//  * the (m, d) online-normalizer state and its merge over lanes,
//  * 128-bit vector loads/stores with bf16 <-> fp32 conversion,
//  * thread-block-cluster helpers (rank, barrier, distributed shared memory).
//
// The (m, d) state and its operator follow "Online normalizer calculation for
// softmax" (notes), section 3.3: (m1,d1) (+) (m2,d2) = (max, d1 e^(m1-max) +
// d2 e^(m2-max)), associative and commutative, identity (-inf, 0) (Lesson 7
// "Online Softmax and associative state", section 3).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../ctl.h"

namespace os {

constexpr unsigned kFullMask = 0xffffffffu;

// ------------------------------------------------------------------ f32x2
// One instruction operates on two fp32 lanes held in a 64-bit register pair,
// halving the issue slots of the exponential's FMA chain.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// Three-input maximum (one instruction on sm_100-family GPUs).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------ exp
// e^z for z <= 88, in fp32, on the FMA pipe only: the library's accurate
// exponential (os_exp_f32) and the rescale factors of the (m, d) merges.
//
//   z := max(z, -88)                      (-inf and NaN become -88: result 0)
//   n  = rint(z log2 e)                   via the 1.5*2^23 rounding constant
//   r  = (z - n ln2_hi) - n ln2_lo        Cody & Waite reduction, |r| <~ ln2/2
//   p  = 1 + c1 r + ... + c6 r^6          minimax fit of e^r on that interval
//   e^z = p * 2^n                         2^n written into the exponent field
//
// For z >= -87.33 the result is within about 1 ulp of e^z; for z in
// [-88, -87.33) it is 0 or a value below FLT_MIN (e^z itself is below FLT_MIN
// there); z = -inf gives exactly +0.  The polynomial coefficients come from
// the Lawson fit in csrc/fit_exp_poly.py, not from any library.
namespace expc {
constexpr float kLog2e = 1.442695022e+00f;   // fp32(log2 e)
constexpr float kRound = 12582912.0f;        // 1.5 * 2^23: adding it rounds to an integer
constexpr float kLn2Hi = 0.693145751953125f; // ln 2 with its low bits cleared (exact n*ln2_hi)
constexpr float kLn2Lo = 1.428606765e-06f;   // ln 2 - kLn2Hi
constexpr float kFloor = -88.0f;
constexpr float c1 = 1.0f;
constexpr float c2 = 0.49999994f;
constexpr float c3 = 0.1666643f;
constexpr float c4 = 0.041668005f;
constexpr float c5 = 0.008374209f;
constexpr float c6 = 0.0013843592f;
}  // namespace expc

// 2^n from t = kRound + n: the low bits of t's pattern hold n; shifting them
// into the exponent field and adding the bias gives 2^n (n = -127 -> +0).
// Written as one integer multiply-add (t_bits * 2^23 + bias, modulo 2^32),
// which the FMA pipe executes, leaving the integer ALU pipe to other work.
__device__ __forceinline__ float pow2_from_rounded(float t) {
    uint32_t b;
    asm("mad.lo.u32 %0, %1, 8388608, 1065353216;" : "=r"(b) : "r"(__float_as_uint(t)));
    return __uint_as_float(b);
}

__device__ __forceinline__ float exp1(float z) {
    using namespace expc;
    z = fmaxf(z, kFloor);
    const float t = fmaf(z, kLog2e, kRound);
    const float n = t - kRound;
    float r = fmaf(n, -kLn2Hi, z);
    r = fmaf(n, -kLn2Lo, r);
    float p = fmaf(c6, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, c1);
    p = fmaf(p, r, 1.0f);
    return p * pow2_from_rounded(t);
}

// ------------------------------------------------------------------ exp (pairs)
// The per-element exponentials of the two-pass streaming kernel (and of the
// three-pass baseline measured against it), the two lanes of a packed f32x2
// at a time, on the FMA and integer pipes only (no ex2.approx):
//
//   z := max(z, -110)                  (-inf included)
//   u  = z log2e + (1.5*2^23 + 66)     one FMA; the rounding constant makes u
//                                      hold n + 66 in its low bits, n = rint(z log2e)
//   f  = z log2e - n                   two FMAs (the constant minus u is -n
//                                      exactly); fp32 results add z log2e_lo
//   p  = 2^f                           minimax fit on [-1/2, 1/2]: degree 5
//                                      (1.1e-7) for fp32 results, degree 3
//                                      (1.0e-4) for bf16 results
//   q  = p 2^(n + 66)                  n + 66 added to p's exponent field: one
//                                      integer shift-add of u's bits
//
// The caller multiplies q by 2^-66 -- and the output pass by 2^-66 / d, so
// the normalisation costs nothing extra -- or sums q first (pass 1 sums a
// chunk, then scales once).  The +66 keeps q a normal number for every
// z >= -110 (n >= -159, so the exponent field of q stays >= 2); the clamp
// makes e^-inf (and anything below e^-110) come out as 0 or a subnormal
// after the scale, below FLT_MIN as e^z itself is.  e^0 is exactly 1.
namespace expc {
constexpr float kLog2eLo = 1.925963034e-08f;  // log2 e - kLog2e
constexpr float kZClamp = -110.0f;
constexpr float kBiasedRound = 12582978.0f;   // 1.5 * 2^23 + 66
constexpr float kUnbias = 1.35525271560688054e-20f;  // 2^-66
// 2^f = 1 + f (e1 + f (e2 + ...)) on [-1/2, 1/2], max relative error 1.1e-7
constexpr float e5_1 = 0.693147f, e5_2 = 0.24022242f, e5_3 = 0.055507336f,
                e5_4 = 0.009671513f, e5_5 = 0.0013264726f;
// the same, degree 3, max relative error 1.0e-4 (results rounded to bf16,
// whose own rounding is 2^-8 relative)
constexpr float e3_1 = 0.69328296f, e3_2 = 0.24221098f, e3_3 = 0.055008918f;
// degree 2, max relative error 2.0e-3: the normaliser sum of rows whose
// results are rounded to bf16 (it adds at most 2.0e-3 to every result's
// error, which with the degree-3 output pass and bf16's rounding stays below
// 6e-3)
constexpr float e2_1 = 0.70294195f, e2_2 = 0.23986399f;
constexpr float kLn2 = 0.693147182f;
}  // namespace expc

// 2^f of a pair for |f| <= 1/2 by the fit of degree DEG (2, 3 or 5).
template <int DEG>
__device__ __forceinline__ float2 exp2_poly(float2 f) {
    using namespace expc;
    float2 p;
    if constexpr (DEG == 5) {
        p = fma2(splat2(e5_5), f, splat2(e5_4));
        p = fma2(p, f, splat2(e5_3));
        p = fma2(p, f, splat2(e5_2));
        p = fma2(p, f, splat2(e5_1));
    } else if constexpr (DEG == 3) {
        p = fma2(splat2(e3_3), f, splat2(e3_2));
        p = fma2(p, f, splat2(e3_1));
    } else {
        static_assert(DEG == 2, "fitted degrees");
        p = fma2(splat2(e2_2), f, splat2(e2_1));
    }
    return fma2(p, f, splat2(1.0f));
}

// p * 2^k where u = 1.5 * 2^23 + k (an integer-valued float, |k| < 2^22):
// p's bits plus u's bits times 2^23, one integer multiply-add.
__device__ __forceinline__ float add_exponent(float p, float u) {
    uint32_t r;
    asm("mad.lo.u32 %0, %1, 8388608, %2;" : "=r"(r) : "r"(__float_as_uint(u)), "r"(__float_as_uint(p)));
    return __uint_as_float(r);
}

// q = 2^(z log2 e + 66) of a pair, -126 <= z <= 43 after the clamp; DEG 5
// (fp32 results) or 3 (bf16).  CLAMP = false: the caller has already bounded
// z from below (at -110 or lower, but not below -126), e.g. on packed bf16
// inputs.  Above, z up to 43 keeps q (and a sum of 32 such) finite.
template <int DEG, bool CLAMP = true>
__device__ __forceinline__ float2 exp_biased_pair(float2 z) {
    using namespace expc;
    if constexpr (CLAMP) z = make_float2(fmaxf(z.x, kZClamp), fmaxf(z.y, kZClamp));
    const float2 K = splat2(kBiasedRound);
    const float2 u = fma2(z, splat2(kLog2e), K);
    const float2 neg_n = fma2(u, splat2(-1.0f), K);  // exact: both near 1.5 * 2^23
    float2 f = fma2(z, splat2(kLog2e), neg_n);
    if constexpr (DEG == 5) f = fma2(z, splat2(kLog2eLo), f);
    const float2 p = exp2_poly<DEG>(f);
    // u's bits are those of 1.5 * 2^23 plus n + 66; times 2^23 (modulo 2^32)
    // the constant part leaves the word and n + 66 lands on the exponent field
    return make_float2(add_exponent(p.x, u.x), add_exponent(p.y, u.y));
}

// The two bf16 values of a word as exact fp32 values, by byte permutes (on
// the integer pipe, off the FMA pipe that the exponential keeps busy).
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(lo) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x3244;" : "=r"(hi) : "r"(w));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// Shift m folded into the exponential: for a reference m (finite, |m| <
// 2^21), 2^((x - m) log2 e) = q(x) * frac with q(x) = 2^(x log2 e + c_int +
// 66) from exp_folded_pair and k = 1.5 * 2^23 + 66 + c_int, where
// -m log2 e = c_int + c_frac (c_int an integer, |c_frac| <= 1/2 + 2^-20,
// m log2 e carried in two fp32 parts) and frac = 2^c_frac * 2^-66.  log2 e's
// own fp32 rounding enters only through (x - m).
struct FoldedShift {
    float2 k;
    float frac;
};
__device__ __forceinline__ FoldedShift folded_shift(float m) {
    using namespace expc;
    const float b_hi = m * kLog2e;
    const float b_lo = fmaf(m, kLog2e, -b_hi);  // exact residual of the product
    const float c_int = rintf(-b_hi);
    const float c_frac = (-b_hi - c_int) - b_lo;
    return {splat2(kBiasedRound + c_int), exp1(c_frac * kLn2) * kUnbias};
}

// q = 2^(x log2 e + c_int + 66) of a pair of inputs x (not x - m), for
// -126 <= x - m <= 43 (the caller clamps below): the rounding constant k of
// folded_shift(m) takes the place of the subtraction of m.  DEG 2 or 3.
template <int DEG>
__device__ __forceinline__ float2 exp_folded_pair(float2 x, float2 k) {
    using namespace expc;
    const float2 u = fma2(x, splat2(kLog2e), k);
    const float2 neg_n = fma2(u, splat2(-1.0f), k);  // exact
    const float2 f = fma2(x, splat2(kLog2e), neg_n);   // x log2 e - rint(x log2 e)
    const float2 p = exp2_poly<DEG>(f);
    return make_float2(add_exponent(p.x, u.x), add_exponent(p.y, u.y));
}

__device__ __forceinline__ float ex2_sfu(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// e^z of a pair on the SFU (the register, on-chip and statistics kernels):
// accurate (FAST = false: log2 e carried in two fp32 parts, for fp32 results)
// or with log2 e rounded to fp32 (FAST = true, for results rounded to bf16
// afterwards).  Error of e^z: the product t =
// z log2 e rounded once (2^-24 |z| relative) plus ex2's few ulp.
template <bool FAST>
__device__ __forceinline__ float2 exp_pair(float2 z) {
    float2 t;
    if constexpr (FAST) t = mul2(z, splat2(expc::kLog2e));
    else t = fma2(z, splat2(expc::kLog2e), mul2(z, splat2(expc::kLog2eLo)));
    return make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
}

// e^z / d of a pair on the SFU for results rounded to bf16, folded into one
// exponent: 2^(z log2 e - log2 d), with neg_log2_d = -log2 d.
__device__ __forceinline__ float2 exp_pair_div(float2 z, float neg_log2_d) {
    const float2 t = fma2(z, splat2(expc::kLog2e), splat2(neg_log2_d));
    return make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
}

// ------------------------------------------------------------------ (m, d)
// Rescale factor e^(m - M) of a state with maximum m into a merge whose
// maximum is M >= m.  m == M gives 1 (also when both are -inf: the NaN of
// -inf - -inf becomes 0 inside exp1, and such a state has d = 0 anyway).
__device__ __forceinline__ float rescale(float m, float M) {
    return m == M ? 1.0f : exp1(m - M);
}

// n-ary (+) over aligned groups of G lanes (G a power of two <= 32): the
// maxima are max-reduced, every lane rescales its own d once to the group
// maximum, and the rescaled d are sum-reduced.  By associativity this equals
// folding the pairwise operator over the group; every lane ends with the
// group's state.  All 32 lanes of the warp must call it together.
template <int G>
__device__ __forceinline__ void group_merge(float& m, float& d) {
    float M = m;
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
    d *= rescale(m, M);
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) d += __shfl_xor_sync(kFullMask, d, o);
    m = M;
}

// ------------------------------------------------------------------ vectors
// A 16-byte input vector holds EPV = 16 / sizeof(T) elements.
template <typename T> struct VecTraits;
template <> struct VecTraits<float> { static constexpr int EPV = 4; };
template <> struct VecTraits<__nv_bfloat16> { static constexpr int EPV = 8; };

// L2 eviction policies for loads that will be read again soon (pass 1 of a
// two-pass kernel) and for last reads (pass 2).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_policy_v4(const void* p, uint64_t policy) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(policy));
    return v;
}

// Coherent (not read-only-path) 16-byte loads, with and without an L2 policy,
// for inputs that the same launch may overwrite: softmax exactly in place,
// where y == x.  In every softmax kernel an element is written only by the
// thread that read it (or, for rows staged in shared memory, by that CTA),
// after reading it, and the value written depends on the value read, so no
// load can move past the store to its own address.  The loads therefore need
// neither `volatile` nor a memory clobber, and the compiler stays free to
// schedule them.
__device__ __forceinline__ uint4 ld_coherent_policy_v4(const void* p, uint64_t policy) {
    uint4 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint4 ld_coherent_v4(const void* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Unpack one 16-byte vector of T into EPV floats.
__device__ __forceinline__ void unpack(const uint4& v, float* out, float) {
    out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float* out, __nv_bfloat16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// (lo - m, hi - m) of a word holding two bf16 values, widened exactly and
// subtracted in one mixed-precision instruction each (no separate unpack).
__device__ __forceinline__ float2 sub_bf16x2(uint32_t w, float m) {
    float2 z;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(z.x), "=f"(z.y) : "r"(w), "f"(m));
    return z;
}

// Lane-wise maximum of two words of two bf16 values each.
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16x2_max_to_f32(uint32_t w) {
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Store N consecutive outputs (N = EPV of the input type) with the widest
// aligned vector stores; streaming (evict-first) cache hint.
template <typename TO, int N> struct VecStore;
template <> struct VecStore<float, 4> {
    __device__ __forceinline__ static void run(float* p, const float* v) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
};
template <> struct VecStore<float, 8> {
    __device__ __forceinline__ static void run(float* p, const float* v) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
};
template <> struct VecStore<__nv_bfloat16, 4> {
    __device__ __forceinline__ static void run(__nv_bfloat16* p, const float* v) {
        uint2 w = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        __stcs(reinterpret_cast<uint2*>(p), w);
    }
};
template <> struct VecStore<__nv_bfloat16, 8> {
    __device__ __forceinline__ static void run(__nv_bfloat16* p, const float* v) {
        uint4 w = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                             pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        __stcs(reinterpret_cast<uint4*>(p), w);
    }
};

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Full barrier over all threads of all CTAs of the cluster; the release /
// acquire pair orders shared-memory writes to peers before their reads.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `local` (a __shared__ object of this CTA) in CTA `rank`'s
// shared memory window of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void* local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(addr), "f"(v.x), "f"(v.y)
                 : "memory");
}

// ------------------------------------------------------------------ async copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// One poll of phase `parity`: the thread may sleep in the instruction until
// the phase completes or about kSuspendHintNs pass, so waiting warps issue
// (almost) nothing while a copy is in flight.
constexpr uint32_t kSuspendHintNs = 200000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
                 : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most ctl.timeout_ns
// (and at most 2^24 polls).  On giving up, records kErrWaitTimeout in the
// device status word and returns false; the caller carries on with whatever
// is in the buffer, so a lost copy corrupts outputs but never hangs the GPU.
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint64_t* bar, uint32_t parity,
                                                     unsigned long long timeout_ns,
                                                     unsigned int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) break;
    }
    atomicOr(err, kErrWaitTimeout);
    return false;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const KernelCtl& ctl) {
    return mbar_wait_bounded_ns(bar, parity, ctl.timeout_ns, ctl.err);
}

// Bound of the wait, before a CTA exits, for its own bulk copies still in
// flight (only after a data wait gave up).  Fixed and long: a copy that has
// been issued lands within microseconds, and a CTA must not exit while one
// can still write its shared memory; the caller-set data-wait bound (which
// may be as short as a millisecond) does not apply here.
constexpr unsigned long long kDrainTimeoutNs = 4000000000ull;

// CTA-wide bounded wait: thread 0 polls (the other threads sleep in the CTA
// barrier instead of spinning), then the result is shared through flag[which]
// (a __shared__ int[2]); callers alternate `which` between consecutive waits
// so a slow reader never sees the next wait's result.  Every thread of the
// CTA must call it.
__device__ __forceinline__ bool cta_wait_bounded(uint64_t* bar, uint32_t parity,
                                                 const KernelCtl& ctl, int* flag, int which) {
    if (threadIdx.x == 0) flag[which] = mbar_wait_bounded(bar, parity, ctl) ? 1 : 0;
    __syncthreads();
    return flag[which] != 0;
}

// Asks L2 to fetch [src, src + bytes) from memory ahead of its use, with an
// eviction policy; nothing reaches this SM and nothing waits for it.  src
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
                 :: "l"(src), "r"(bytes), "l"(policy) : "memory");
}

// One bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// 8 bytes into the shared memory of a CTA of the cluster (`remote`, a
// shared::cluster address from map_to_rank), completing `bytes` of the
// transaction count of that CTA's barrier `remote_bar`.
__device__ __forceinline__ void st_async_b64(uint32_t remote, uint32_t lo, uint32_t hi,
                                             uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
                 :: "r"(remote), "r"(lo), "r"(hi), "r"(remote_bar) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
    return v;
}

}  // namespace os
