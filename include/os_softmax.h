/*
 * os_softmax.h -- C ABI of libos_softmax.so: row-wise online-normalizer
 * softmax and fused softmax+TopK on one NVIDIA GB300 GPU (sm_103a), with the
 * attention forward that the same (m, d) recurrence carries onto the tensor
 * cores (os_attention_fwd).
 *
 * Operations (statement of the problem):
 *   softmax : for each row r of x[rows, cols], y[r, i] = e^(x[r,i] - m_r) / d_r
 *             with m_r = max_j x[r,j] and d_r = sum_j e^(x[r,j] - m_r)
 *             ("Online normalizer calculation for softmax" notes, section 2,
 *             safe softmax; computed with the single-pass online normalizer of
 *             its section 3 and the (m, d) combine of section 3.3).
 *   topk    : for each row, the K largest probabilities v and their column
 *             indices z, without writing the full probability row (same notes,
 *             section 4, "Softmax and top-k fusion": select the K largest
 *             logits u in the normalizer's single pass, then
 *             v_i = e^(u_i - m_r) / d_r).
 *   attention : softmax(scale Q K^T) V per (batch, head) slice and its
 *             logsumexp (see os_attention_fwd).
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers into dense row-major buffers (row stride =
 *     cols elements) that the caller allocates, owns and frees.  The library
 *     allocates no device or host memory and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  The return value reports argument errors and launch
 *     errors (the return code of the CUDA launch); a fault inside a kernel
 *     surfaces at the caller's next synchronisation, as for any CUDA launch.
 *   - rows == 0 is a no-op returning OS_OK.  cols must be in [1, 2^31 - 1].
 *   - Inputs are assumed free of NaN.  -inf entries are allowed and get
 *     probability exactly +0; a row whose entries are ALL -inf has no defined
 *     softmax and its outputs are unspecified (NaN in practice).
 *   - Arithmetic: fp32 throughout (bf16 inputs widened exactly, fp32
 *     accumulation, bf16 outputs rounded to nearest even).  Per-element
 *     exponentials: the two-pass streaming kernel (AUTO's choice for rows
 *     longer than 8192 fp32 / 4096 bf16 elements) and the three-pass
 *     baseline use the library's own FMA-pipe exponential for fp32 results
 *     (no ex2.approx: base-2 reduction, a degree-5 polynomial, 2^n added to
 *     the exponent field), and for bf16 results too under
 *     OS_PATH_STREAM_POLY (degree 2 for the normaliser, 3 for the outputs);
 *     bf16 results on OS_PATH_STREAM and the register, on-chip, statistics
 *     and TopK kernels use the SFU's 2^x (ex2.approx) of (x - m) log2 e,
 *     log2 e in two fp32 parts for fp32 results.  A value
 *     that carries a whole row (a merge's rescale factor, a TopK output
 *     value) uses the library's accurate exponential (os_exp_f32).
 *   - Work runs on the device current at the call (cudaGetDevice); the
 *     pointers and the stream must belong to it.  There is no CPU fallback.
 */
#ifndef OS_SOFTMAX_H
#define OS_SOFTMAX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. */
typedef struct CUstream_st *os_stream_t;

typedef enum {
    OS_F32 = 0,  /* IEEE binary32 */
    OS_BF16 = 1  /* bfloat16 */
} os_dtype;

typedef enum {
    OS_OK = 0,
    OS_ERR_NULL = 1,    /* a required pointer is NULL (with rows > 0) */
    OS_ERR_SHAPE = 2,   /* rows < 0, cols outside [1, 2^31 - 1] */
    OS_ERR_DTYPE = 3,   /* dtype value not in os_dtype */
    OS_ERR_K = 4,       /* K outside [1, min(cols, 256)] */
    OS_ERR_ALIAS = 5,   /* an output overlaps an input or another output */
    OS_ERR_CUDA = 6,    /* the CUDA runtime reported an error (launch or device query) */
    OS_ERR_TIMEOUT = 7, /* a device-side bounded wait gave up (os_device_status) */
    OS_ERR_PATH = 8,    /* the requested kernel family cannot run this shape */
    OS_ERR_ALIGN = 9,   /* a pointer is not aligned to its element size */
    OS_ERR_VALUE = 10   /* a scalar argument outside its range (attention scale, causal flag) */
} os_status;

/* Kernel families (see os_softmax_fwd_path). */
typedef enum {
    OS_PATH_AUTO = 0,   /* choose by row length, dtype and device */
    OS_PATH_WARP = 1,   /* 1..32 lanes per row, row held in registers; short rows */
    OS_PATH_ONCHIP = 2, /* one CTA or a thread-block cluster per row, row held
                           in registers across the cluster; one HBM read */
    OS_PATH_STREAM = 3, /* two passes over the row (running (m, d), then
                           normalise); any row length */
    OS_PATH_SAFE = 4,   /* baseline: the three-pass safe softmax (maximum;
                           sum of e^(x - m); normalise), each pass reading the
                           row from memory ("Online normalizer calculation for
                           softmax", section 2); any row length; never chosen
                           by AUTO */
    OS_PATH_STREAM_POLY = 5 /* OS_PATH_STREAM with the library's FMA-pipe
                           exponential for every output dtype (no
                           ex2.approx anywhere in the kernel).  For fp32
                           results this is the STREAM kernel itself; for bf16
                           results it replaces the SFU's 2^x (STREAM's and
                           AUTO's choice there, about 20 % faster on GB300)
                           by degree-2 (normaliser) and degree-3 (outputs)
                           fits of 2^f; never chosen by AUTO */
} os_path;

/* Launch configuration chosen for a call (see os_softmax_plan / os_topk_plan). */
typedef struct {
    int32_t path;               /* os_path actually used (never AUTO) */
    int32_t threads;            /* threads per CTA */
    int32_t vectors_per_thread; /* 16-byte input vectors held per thread (per chunk for STREAM) */
    int32_t cluster;            /* CTAs per row (thread-block cluster size), 1 if none */
    int32_t lanes_per_row;      /* WARP path: lanes that share one row; else 0 */
    int32_t stages;             /* ONCHIP path with bulk-copy staging: row slices
                                   prefetched in shared memory; 0 = registers only */
    int64_t grid;               /* CTAs launched */
} os_plan;

/*
 * y = softmax(x) row by row.
 *   x         device pointer, rows*cols elements of in_dtype, read only.
 *   y         device pointer, rows*cols elements of out_dtype, written.
 *             Either y == x with out_dtype == in_dtype (in place: x is
 *             overwritten by its softmax) or no overlap with x at all; any
 *             other overlap is OS_ERR_ALIAS.
 *   in_dtype, out_dtype: OS_F32 or OS_BF16, in any combination.
 * Pointers must be aligned to their element size (OS_ERR_ALIGN).  Rows move
 * as the aligned 16-byte blocks they cover (128-bit loads, and 128-bit stores
 * when y's rows have x's offset inside their 16-byte blocks), with element
 * access only for the partial block at each end of a row.  A row that does
 * not start on a 16-byte boundary can need one 16-byte slot more than
 * cols / (16/sizeof(in)), which the choice of kernel family accounts for.
 */
os_status os_softmax_fwd(const void *x, void *y, int64_t rows, int64_t cols,
                         os_dtype in_dtype, os_dtype out_dtype, os_stream_t stream);

/*
 * Fused softmax + TopK: for each row the K largest probabilities, best first.
 *   x     device pointer, rows*cols fp32 logits, read only (4-byte aligned is
 *         enough; rows need not start on 16-byte boundaries).
 *   vals  device pointer, rows*K fp32: vals[r*K + k] = e^(x[r,z] - m_r) / d_r
 *         of the k-th best column z.
 *   idx   device pointer, rows*K int32: the column indices z.
 *   K     1 <= K <= min(cols, 256).
 * Order: larger logit first; equal logits (ties) go to the LOWER column index.
 * Selection compares the input logits, so distinct logits whose probabilities
 * round to the same fp32 value keep their logit order.  vals and idx must not
 * overlap x or each other (OS_ERR_ALIAS).
 */
os_status os_softmax_topk(const float *x, float *vals, int32_t *idx, int64_t rows,
                          int64_t cols, int32_t K, os_stream_t stream);

/*
 * TopK of x itself (no softmax): for each row the K largest values and their
 * columns, best first, with the same order, ties rule, arguments, checks and
 * kernel as os_softmax_topk; vals[r*K + k] = x[r, idx[r*K + k]] exactly.
 * With y = softmax(x) from os_softmax_fwd it forms the unfused softmax-then-
 * TopK pipeline that "Online normalizer calculation for softmax" (section 4)
 * compares the fused kernel with; it is also a plain row TopK.
 */
os_status os_topk(const float *x, float *vals, int32_t *idx, int64_t rows, int64_t cols,
                  int32_t K, os_stream_t stream);

/*
 * y = softmax(x) row by row under a causal mask applied inside the kernel:
 * in row r the columns c > (r mod period) + offset are masked (treated as
 * -inf, never read, written as exactly 0), the attention mask of a query at
 * position r mod period over keys with `offset` extra leading positions
 * ("6.2 FlashAttention V2": the causal mask applied while the row is
 * processed rather than stored in the input).
 *   period >= 1, offset >= 0 (so every row keeps at least column 0), else
 *   OS_ERR_SHAPE.  Other arguments, checks and layout as os_softmax_fwd.
 * Rows of up to 256 16-byte vectors run on the WARP family, longer ones on
 * STREAM; masked columns cost no reads.
 */
os_status os_softmax_causal_fwd(const void *x, void *y, int64_t rows, int64_t cols,
                                int64_t period, int64_t offset, os_dtype in_dtype,
                                os_dtype out_dtype, os_stream_t stream);

/*
 * The online normalizer's state of every row, without normalising ("Online
 * normalizer calculation for softmax", section 3): m[r] = max_j x[r, j],
 * d[r] = sum_j e^(x[r, j] - m[r]) (so 1 <= d[r] <= the number of finite
 * entries), and lse[r] = m[r] + ln d[r], the row's log-sum-exp ("6.2
 * FlashAttention V2" keeps it per row for the backward pass).  One read of x.
 *   x    device pointer, rows*cols of in_dtype (OS_F32 or OS_BF16).
 *   m, d, lse  device pointers to rows fp32 each, written; any of them may be
 *        NULL (not written) but not all three (OS_ERR_NULL).  They must not
 *        overlap x or one another (OS_ERR_ALIAS).
 * Rows that are all -inf give m = -inf, d = 0, lse = -inf.
 */
os_status os_softmax_stats(const void *x, float *m, float *d, float *lse, int64_t rows,
                           int64_t cols, os_dtype in_dtype, os_stream_t stream);

/*
 * Top-K sampling after the fused pass ("Online normalizer calculation for
 * softmax", section 4, names sampling from the top K as what the fused kernel
 * feeds): for each row one column drawn from its K entries with probability
 * proportional to their values, i.e. from the top-K distribution
 * renormalised.
 *   vals, idx  device pointers, rows*K: the outputs of os_softmax_topk (or
 *              os_topk on probabilities), best first; values >= 0.
 *   u          device pointer, rows fp32 uniform numbers in [0, 1), one per
 *              row, supplied by the caller (the random source stays outside).
 *   out        device pointer, rows int32, written: out[r] = idx[r*K + k] for
 *              the smallest k with p_0 + ... + p_k > u[r] * (p_0 + ... +
 *              p_{K-1}), every sum and the product rounded to fp32 in index
 *              order (u >= 1 gives the last entry).  Must not overlap the
 *              inputs (OS_ERR_ALIAS).
 *   K          1 <= K <= 256 (OS_ERR_K).
 */
os_status os_topk_sample(const float *vals, const int32_t *idx, const float *u, int32_t *out,
                         int64_t rows, int32_t K, os_stream_t stream);

/* Attention forward on the tensor cores ("6.2 FlashAttention V2", section 6.1,
 * forward algorithm; the (m, d, o) recurrence of the "Online normalizer
 * calculation for softmax" notes, FlashAttention section):
 *   O[s, i, :] = sum_j softmax_j(scale * q_i . k_j) v_j,
 *   L[s, i]    = ln sum_j e^(scale * q_i . k_j)  (the logsumexp kept for a backward pass),
 * over the keys j that query i sees: all n of them, or j <= i when `causal`
 * is 1.  s runs over the bh (batch x head) slices.
 *   q, k, v    [bh][n][head_dim] bf16, row-major, 16-byte aligned (OS_ERR_ALIGN).
 *   o          [bh][n][head_dim] bf16 output, 16-byte aligned; must not overlap
 *              q, k or v (OS_ERR_ALIAS).
 *   lse        [bh][n] fp32 output, 4-byte aligned, or NULL (not written); must
 *              not overlap any other argument (OS_ERR_ALIAS).
 *   bh >= 0 and n >= 0 (either 0: no-op); n <= 2^31 - 1 and bh * ceil(n/128)
 *   <= 2^31 - 1; head_dim 64 or 128 (OS_ERR_SHAPE otherwise).
 *   scale      finite and > 0, usually 1/sqrt(head_dim) (OS_ERR_VALUE).
 *   causal     0 or 1 (OS_ERR_VALUE).
 * Arithmetic: scores Q K^T in fp32 on the tensor cores from bf16 operands;
 * probabilities e^(scale s - m) in fp32, summed into l in fp32 and rounded to
 * bf16 for the P V product (fp32 accumulation); O = (P V) / l rounded to bf16;
 * L = m + ln l in fp32.  The buffers are the caller's; the
 * library allocates nothing. */
os_status os_attention_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t bh, int64_t n, int32_t head_dim, float scale, int32_t causal,
                           os_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *os_status_string(os_status status);

/*
 * os_softmax_fwd with the kernel family fixed by the caller (tests and
 * benchmarks use it to exercise every family on the same shape).
 * OS_PATH_AUTO behaves exactly like os_softmax_fwd.  A family that cannot
 * hold the row (WARP beyond 32 x 8 vectors, ONCHIP beyond the largest
 * cluster the device can launch) returns OS_ERR_PATH and launches nothing.
 */
os_status os_softmax_fwd_path(const void *x, void *y, int64_t rows, int64_t cols,
                              os_dtype in_dtype, os_dtype out_dtype, os_path path,
                              os_stream_t stream);

/*
 * The launch configuration os_softmax_fwd_path would use for this shape on the
 * current device, written to *plan; nothing is launched.  Same argument
 * checks as the launching call, minus the pointer checks; x and y are assumed
 * 16-byte aligned (the choice can differ for other pointers).
 */
os_status os_softmax_plan(int64_t rows, int64_t cols, os_dtype in_dtype, os_dtype out_dtype,
                          os_path path, os_plan *plan);

/* The launch configuration os_softmax_topk would use; nothing is launched. */
os_status os_topk_plan(int64_t rows, int64_t cols, int32_t K, os_plan *plan);

/*
 * out[i] = e^(z[i]) for n fp32 values with the library's own exponential
 * (Cody-Waite reduction z = n ln2 + r, a degree-6 minimax polynomial for e^r,
 * 2^n written into the exponent field; no ex2.approx).  The kernels above use
 * it where one value carries a whole row (the rescale factors of the merges,
 * the TopK output values).  Defined
 * for z <= 88: within about 1 ulp of e^z for
 * z >= -87.33, 0 or a value below FLT_MIN for smaller z, exactly +0 for
 * z = -inf.  Exposed so the routine can be tested on its own.
 *   z, out  device pointers to n fp32 values (may be the same buffer).
 */
os_status os_exp_f32(const float *z, float *out, int64_t n, os_stream_t stream);

/*
 * out[i] = e^(z[i]) for n fp32 values with the per-element exponential of the
 * two-pass streaming kernel's fp32 results: two values at a time on packed
 * fp32 FMAs, no ex2.approx (n = rint(z log2 e) from one FMA with a rounding
 * constant, f = z log2 e - n with log2 e in two fp32 parts, a degree-5
 * minimax polynomial for 2^f, n + 66 added to its exponent field by an
 * integer shift-add, then one multiply by 2^-66, which the kernel shares with
 * its 1/d).  Defined for z <= 0, the softmax domain x - max: within 3e-7
 * relative of e^z for z >= -87.33, 0 or a value below FLT_MIN for smaller z
 * (exactly +0 below -110 and for z = -inf), exactly 1 for z = 0.  Exposed so
 * the routine can be tested on its own; arguments and checks as os_exp_f32
 * (n may be odd).
 */
os_status os_exp_pairs_f32(const float *z, float *out, int64_t n, os_stream_t stream);

/*
 * The same for the streaming kernel's bf16 results, before their rounding to
 * bf16: log2 e in one fp32 part and a degree-3 polynomial for 2^f (1.0e-4),
 * so within 1.2e-4 relative of e^z for z >= -87.33 (bf16 itself rounds at
 * 2^-9 = 2.0e-3); the other properties as os_exp_pairs_f32.
 */
os_status os_exp_pairs_coarse_f32(const float *z, float *out, int64_t n, os_stream_t stream);

/*
 * Device-side waits.  Kernels that stage rows in shared memory wait on
 * hardware barriers for their bulk copies; every such wait is bounded (by
 * default 1 s).  A wait that gives up does not hang or fault the GPU: the
 * kernel finishes with garbage in the affected outputs and records the event
 * in a per-device status word.
 *
 * os_device_status reads and clears the word in one atomic exchange (a
 * one-thread kernel on `stream`), synchronises `stream`, and returns
 * OS_ERR_TIMEOUT if any kernel of this library on the current device gave up
 * a wait since the previous call, OS_OK otherwise.  A kernel on another stream
 * that records a timeout concurrently is reported by this call or the next,
 * never lost.  Host callers are serialised inside the call.
 *
 * Two bounds apply.  The data wait (a copy or a peer's message that a CTA
 * needs before it can go on) is bounded by os_set_wait_timeout_ns.  The drain
 * wait (a CTA whose data wait gave up waits, before it exits, for its own
 * bulk copies still in flight so none lands after it has gone) has its own
 * fixed bound of 4 s, which no setting shortens.
 */
os_status os_device_status(os_stream_t stream);

/*
 * Testing controls, process-wide, read at every launch.
 *   os_set_wait_timeout_ns: bound of each device-side data wait, 1 ms .. 10 s
 *     (OS_ERR_SHAPE outside that range).
 *   os_set_fault_injection: 0 = off (default); 1 = in every following launch
 *     one CTA withholds data that another CTA waits for, so that wait must run
 *     out (exercises the bounded-wait path; the outputs of that launch are
 *     garbage): in the bulk-copy ring softmax (OS_PATH_ONCHIP rows held in
 *     shared memory) the first CTA never issues its first copy; in the fused
 *     TopK, when a row is split over a cluster, CTA 1 of the first cluster
 *     never sends its list to CTA 0.  Other values: OS_ERR_SHAPE.
 */
os_status os_set_wait_timeout_ns(uint64_t ns);
os_status os_set_fault_injection(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* OS_SOFTMAX_H */
