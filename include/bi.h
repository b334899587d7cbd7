/*
 * bi.h - batch-invariant verify pass for GB300 (sm_103a), C ABI.
 *
 * The library computes the linear layers of an LLM decode or speculative
 * verify pass (M = 1 .. K+1 tokens against a large int8 weight matrix) so that
 * every output row is bitwise identical whatever M is and whatever else shares
 * the pass; with them the LM-head argmax, greedy verification, a block-scaled
 * variant of the linear and the verify queries' split-KV attention, each with
 * the same guarantee.  Greedy speculative decoding then keeps exactly the target's own
 * argmax ("why speculative decoding changed my output", introduction: the
 * guarantee needs a position's logits inside a batch to equal its logits
 * decoded alone).
 *
 * Arithmetic (W8A8 as in "Deterministic LLM Inference Across GPU Kernels:
 * Power-of-Two INT8 Quantization Scales and the Limits of Tolerance-Based
 * Conformance", Abstract, Fig. 1, Table II):
 *   s_a[m]   = absmax_k |x[m,k]| / 127  (IEEE fp32 division; 1 if absmax = 0)
 *   q[m,k]   = clamp(rne(x[m,k] / s_a[m]), -127, 127)
 *   acc[m,n] = sum_k q[m,k] * W[n,k]       exact in int32 (K * 127^2 < 2^31)
 *   y[m,n]   = bf16_rne((float(acc) * s_a[m]) * s_w[n])
 * The integer sum is exact and independent of summation order ("The Integer
 * Alibi", abstract), so the kernels may split K in any way; the epilogue is
 * fixed element by element.  Hence rows do not depend on M.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers, allocated and owned by the caller; the
 *    library allocates nothing and keeps no pointer after returning.
 *  - bf16 values are passed as their uint16_t bit patterns.
 *  - Matrices are row-major: x [M, ldx] (ldx >= K), q [M, K], W [N, K]
 *    (K contiguous), y / logits [M, N].
 *  - Work is enqueued on `stream` (NULL = legacy default stream) and the call
 *    returns without waiting.  Calls are reentrant; calls that may run
 *    concurrently on the device must not share output or workspace buffers.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error status and enqueues nothing.  No call
 *    aborts, throws, or writes to stderr.
 *  - Shape limits: 1 <= M <= 65535, 1 <= N <= 2^31-1, 16 <= K, K % 16 == 0,
 *    K * 127^2 < 2^31 (K <= 133144).  Base pointers of x, q and w_q must be
 *    16-byte aligned, and ldx % 8 == 0 (16-byte aligned rows).
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BI_API __attribute__((visibility("default")))
#else
#define BI_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bi_stream_t;

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1, /* null pointer, bad shape, ldx < K, K % 16 != 0 */
    BI_ERR_ALIGNMENT = 2,   /* a base pointer or row stride not 16-byte aligned */
    BI_ERR_INT32_BOUND = 3, /* K * 127^2 >= 2^31: the int32 sum could overflow */
    BI_ERR_WORKSPACE = 4,   /* workspace null or smaller than the queried size */
    BI_ERR_UNSUPPORTED = 5, /* no usable sm_103a device, or a feature missing */
    BI_ERR_TIMEOUT = 6,     /* a kernel gave up a bounded wait (see bi_workspace_status) */
    BI_ERR_CUDA = 7         /* a CUDA runtime/driver call failed */
} bi_status;

/* Flags for the calls that take `flags`. */
enum {
    /* Programmatic dependent launch.  The call may begin while the kernel
     * that precedes it on `stream` is still running: it waits for that kernel
     * before reading any of its inputs except the weight codes w_q, which it
     * may start streaming early, and it lets the next kernel on the stream
     * launch early in the same way.  Use it only when w_q is not written by
     * the immediately preceding kernel (weights are constants of the model).
     * Results are bitwise identical with and without the flag. */
    BI_FLAG_PDL = 1u
};

/* Human-readable name of a status (static string, never NULL). */
BI_API const char *bi_status_string(bi_status s);

/*
 * Per-token activation quantisation.
 *   x    bf16 [M, ldx], first K columns used (read only)
 *   q    int8 [M, K] out, s_a fp32 [M] out
 * s_a[m] = absmax/127 by IEEE division (1 for an all-zero row); q by IEEE
 * division x/s_a, round-to-nearest-even, clamp to [-127, 127].  Subnormal
 * inputs are honoured (no flush to zero).  With BI_FLAG_PDL the kernel waits
 * for the preceding kernel before reading x.
 */
BI_API bi_status bi_quantize_act(const uint16_t *x, int64_t ldx, int M, int K,
                          int8_t *q, float *s_a, unsigned flags, bi_stream_t stream);

/*
 * Chained verify pass: the two elementwise steps between a layer's linears,
 * each fused with the activation quantisation of the linear that reads it.
 * A decode/verify pass chains its linears through the residual stream ("why
 * speculative decoding changed my output", "the mat-vec kernel"; "My
 * speculative decoder got slower", "The physics"); the pages print no layer
 * body, so the steps are this library's reading, both exact roundings of
 * fp32 operations on bf16 values (fp32 has enough bits that an fp32 add or
 * multiply of two bf16 values, then bf16 rounding, equals one rounding of
 * the exact result):
 *
 * bi_residual_quantize: the residual update after the o and down projections.
 *   h    bf16 [M, K] (row stride K), read and written in place
 *   y    bf16 [M, ldy], first K columns added (read only; must not overlap h)
 *   h'   = bf16_rne(h + y)  (fp32 add);  e = floor(log2 max_k |h'[m, k]|),
 *          0 for an all-zero row;  h = bf16_rne(h' * 2^-e)
 *   q, s_a = bi_quantize_act of the new h (the power-of-two rescale keeps a
 *          deep stack finite and changes no code: per-row absmax quantisation
 *          is exactly invariant to scaling a row by a power of two)
 *
 * bi_relu_mul_quantize: the gated MLP product feeding the down projection.
 *   gu   bf16 [M, ldgu] (ldgu >= 2K): gate g = gu[:, 0:K], up u = gu[:, K:2K]
 *        (the output of one packed gate/up linear), read only
 *   m    = bf16_rne(relu(g) * u), relu(g) = g if g > 0 else +0 (fp32 multiply)
 *   q, s_a = bi_quantize_act of m;  m_out bf16 [M, K] (row stride K) receives
 *          m unless it is NULL (it must not overlap gu)
 *
 * Both: 16-byte aligned h, y, gu, m_out and q; row strides multiples of 8
 * elements; K % 16 == 0.  One CTA per row; with BI_FLAG_PDL the kernel waits
 * for the preceding kernel before reading.
 */
BI_API bi_status bi_residual_quantize(uint16_t *h, const uint16_t *y, int64_t ldy, int M, int K,
                                      int8_t *q, float *s_a, unsigned flags, bi_stream_t stream);
BI_API bi_status bi_relu_mul_quantize(const uint16_t *gu, int64_t ldgu, int M, int K, int8_t *q, float *s_a,
                                      uint16_t *m_out, unsigned flags, bi_stream_t stream);

/*
 * Checkpoint-style per-output-channel weight quantisation (offline, not part
 * of the verify pass): the same rule as bi_quantize_act applied to each row of
 * an fp32 matrix.
 *   w    fp32 [N, ldw] (ldw >= K, ldw % 4 == 0, 16-byte aligned), read only
 *   w_q  int8 [N, K] out, s_w fp32 [N] out
 */
BI_API bi_status bi_quantize_weight(const float *w, int64_t ldw, int N, int K,
                             int8_t *w_q, float *s_w, bi_stream_t stream);

/*
 * Power-of-two scale requantisation ("Deterministic LLM Inference ...",
 * Abstract and Fig. 1: every weight scale is moved to its nearest power of
 * two and the codes are requantised to it, not merely relabelled).
 *   s'   = 2^round(log2 s_w[n])   (nearest in the log domain; never a tie)
 *   w_q' = clamp(rne(w_q * s_w[n] / s'), -127, 127), computed exactly
 * A scale whose power of two would exceed fp32 is held at 2^127; rows whose
 * scale is not a positive finite number are copied unchanged.  Outputs may
 * alias the inputs exactly (w_q_out == w_q, s_w_out == s_w) for an in-place
 * update; partial overlap is not allowed.
 */
BI_API bi_status bi_requant_pow2(const int8_t *w_q, const float *s_w, int N, int K,
                          int8_t *w_q_out, float *s_w_out, bi_stream_t stream);

/*
 * Workspace bytes needed by bi_linear_w8a8 for this shape (> 0).  The
 * workspace holds split-K partial sums, their counters and a status word.  It
 * must be zero-filled before its first use (cudaMemset); every call that
 * completes leaves it zero-filled again, so one workspace can serve a whole
 * sequence of calls on one stream.  For M > 16 it is larger: about 12.6 MB
 * for the int32 partial sums of prefill tiles split along K to fill the GPU's
 * last wave (scratch: every call overwrites what it reads) and their counters
 * (zero between calls).  For M > 256 it also holds 2 * (M + N) * K bytes
 * (each part rounded up to 256) for exact f16 copies of q and w_q that the
 * tensor cores read by TMA (scratch).  A smaller workspace still works for
 * M > 16, with the same results: without the f16 room the kernel converts
 * the codes in its tile loop (slower above 256 tokens), and with only the
 * M <= 16 size it also runs without the split.
 */
BI_API size_t bi_linear_workspace_size(int M, int N, int K);

/*
 * y = the W8A8 linear layer above.
 *   q    int8 [M, K], s_a fp32 [M]          (from bi_quantize_act)
 *   w_q  int8 [N, K], s_w fp32 [N]          (per-output-channel codes/scales)
 *   y    bf16 [M, N] out (row stride N)
 *   ws   workspace of ws_bytes >= bi_linear_workspace_size(M, N, K)
 * M <= 16 runs the weight-streaming kernel (TMA-staged int8 weight tiles,
 * int8 tensor-core dot products, int32 partial sums reduced exactly across
 * CTAs); larger M runs the tiled prefill kernel.  Both give the same bits for
 * every row.  Any outputs that do not fit bf16 become +-Inf by round to
 * nearest even.
 */
BI_API bi_status bi_linear_w8a8(const int8_t *q, const float *s_a, int M, int K,
                         const int8_t *w_q, const float *s_w, int N,
                         uint16_t *y, void *ws, size_t ws_bytes,
                         unsigned flags, bi_stream_t stream);

/* Workspace bytes needed by bi_lmhead_argmax (same zero-fill rule). */
BI_API size_t bi_lmhead_workspace_size(int M, int N, int K);

/*
 * Greedy LM head: the logits of bi_linear_w8a8 (optionally written to
 * `logits`, bf16 [M, N]) and, per row, argmax[m] = the lowest n whose bf16
 * logit is the row maximum, logits compared as real numbers (-0 == +0).
 * ("My speculative decoder got slower", "We're nowhere near SOL": a head that
 * computes only the winning token; "Why the decoders disagreed?": bf16 logits
 * do tie.)  M <= 16.
 *   logits  bf16 [M, N] out, or NULL to skip writing them
 *   argmax  int32 [M] out
 */
BI_API bi_status bi_lmhead_argmax(const int8_t *q, const float *s_a, int M, int K,
                           const int8_t *w_q, const float *s_w, int N,
                           uint16_t *logits, int32_t *argmax,
                           void *ws, size_t ws_bytes, unsigned flags, bi_stream_t stream);

/*
 * Device-side status of a workspace: waits for `stream`, reads the status word
 * that kernels set when a bounded wait gives up, clears it, and returns BI_OK
 * or BI_ERR_TIMEOUT (or BI_ERR_CUDA if the stream itself reports an error).
 * After BI_ERR_TIMEOUT the workspace must be zero-filled again before reuse.
 */
BI_API bi_status bi_workspace_status(void *ws, size_t ws_bytes, bi_stream_t stream);

/*
 * Greedy verification of a verify pass, the step after the LM head.  Greedy
 * speculative decoding keeps exactly the tokens plain greedy decoding would
 * produce ("why speculative decoding changed my output", introduction; "My
 * speculative decoder got slower", "Speculative decoding (SD)").  The pass
 * ran the target on the last accepted token followed by the drafted tokens
 * d_1 .. d_{M-1}; argmax[i] is the target's choice after input i.
 *   argmax int32 [M] (from bi_lmhead_argmax), draft int32 [M - 1] (NULL when
 *   M == 1), out int32 [2] receives L = the length of the longest prefix with
 *   argmax[i] == draft[i], and argmax[L] (the correction, or the bonus token
 *   when all M - 1 drafts are accepted).  Device pointers, 4-byte aligned.
 * One warp; M <= 65535.  In a program, the same result is produced by an
 * LM-head op whose `draft` and `accept` fields are set, in the CTA that
 * finishes the argmax.
 */
BI_API bi_status bi_greedy_verify(const int32_t *argmax, const int32_t *draft, int M, int32_t *out,
                                  bi_stream_t stream);

/*
 * Test of the failure path: launches one thread that waits, with the same
 * bounded wait the kernels use, on a barrier phase that nothing completes.
 * After the wait limit (2 s of GPU time) it gives up and sets the status
 * word of `ws` (a linear workspace, >= bi_linear_workspace_size(1, 1, 16)
 * bytes), so that bi_workspace_status then returns BI_ERR_TIMEOUT.  With
 * ws = NULL (ws_bytes ignored) the status word is that of the fixed scratch
 * of bi_linear_w8a8_noalloc, read back by bi_linear_w8a8_noalloc_status.
 * Nothing faults or hangs; the context stays usable.
 */
BI_API bi_status bi_selftest_wait_timeout(void *ws, size_t ws_bytes, bi_stream_t stream);

/*
 * Block-scaled variant: the mat-vec of "why speculative decoding changed my
 * output", section "the mat-vec kernel" (q6_k-style weight blocks of 256,
 * int8 activation blocks of 32, integer products per block, fp32 per-block
 * scale-and-add in an order fixed for every number of tokens).  The pages
 * print no storage layout or quantiser; this library's are:
 *
 * Weights, K % 256 == 0.  Super-blocks of 256 = 16 sub-blocks of 16; code
 * c in [-32, 31], int8 sub-scale sc per sub-block, fp32 scale d per
 * super-block; w ~ c * (d * sc).  Per row n:
 *   ql [K/2]  low 4 bits of c + 32, element k in byte k/2, bits 4 (k & 1)
 *   qh [K/4]  high 2 bits of c + 32, element k in byte k/4, bits 2 (k & 3)
 *   sc [K/16], d [K/256]
 * Quantiser, per super-block: t_j = absmax_j / 31 (IEEE fp32 division);
 * d = max_j t_j / 127 (1 if all zero); sc_j = clamp(rne(t_j / d), 0, 127);
 * e_j = d * sc_j (fp32); c = clamp(rne(w / e_j), -32, 31), 0 where e_j = 0.
 *   w  fp32 [N, K] (row stride ldw >= K, ldw % 4 == 0), device.
 *   ql, qh, sc, d  device outputs, row-major as above (16-byte aligned; d 4).
 * Returns BI_ERR_INVALID_ARG for K not a positive multiple of 256.
 */
BI_API bi_status bi_quantize_weight_q6(const float *w, int64_t ldw, int N, int K, uint8_t *ql, uint8_t *qh,
                                       int8_t *sc, float *d, bi_stream_t stream);

/*
 * Activation blocks of 32 for the block-scaled linear: the per-token rule of
 * bi_quantize_act applied to each block of 32 (d_a = absmax / 127, 1 for an
 * all-zero block; q = clamp(rne(x / d_a), -127, 127), IEEE division).
 *   x    bf16 [M, K] (row stride ldx >= K), K % 32 == 0
 *   q    int8 [M, K] out;  d_a  fp32 [M, K/32] out (4-byte aligned)
 */
BI_API bi_status bi_quantize_act_blocks(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *d_a,
                                        bi_stream_t stream);

/*
 * y = the block-scaled linear, fp32 [M, N] (row stride N), 1 <= M <= 16.
 * For token m and row n, 32-block b (of K/32) of super-block s = b / 8 holds
 * sub-blocks j = 2b and 2b + 1:
 *   isum_b = sc_j * sum(c * q) over its first 16 elements
 *          + sc_(j+1) * sum over the next 16               (exact integer)
 *   v_b    = ((float)isum_b * d_a[m][b]) * d[n][s]          (fp32, RNE)
 * Partial l (l = 0 .. 31) adds v_l, v_(l+32), v_(l+64), ... in that order
 * starting from +0; then, for offsets 16, 8, 4, 2, 1, every partial becomes
 * p[l] + p[l xor offset]; y[m][n] = p[0].  The order depends on K only, so
 * every row is bitwise the same for any M and any other rows in the pass.
 *   q, d_a  from bi_quantize_act_blocks (q rows 16-byte aligned)
 *   ql, qh, sc, d  from bi_quantize_weight_q6
 *   flags   BI_FLAG_PDL or 0
 */
BI_API bi_status bi_linear_q6(const int8_t *q, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                              const int8_t *sc, const float *d, int N, float *y, unsigned flags, bi_stream_t stream);

/*
 * Split-KV attention of a verify pass, batch-invariant ("My speculative
 * decoder got slower", split-KV attention in 256-token chunks with a merge;
 * "why speculative decoding changed my output", "attention").  Query m
 * (0 .. M-1) attends to cache positions 0 .. T0 + m; query head h reads kv
 * head h / (Hq / Hkv).  Per query, head and chunk c (positions 256c ..
 * 256c + 255 of those), fp32, every operation rounded once:
 *   s_t = (sum over d in order of q_d k_td, from +0) * scale
 *   mx  = max s_t,  p_t = e(s_t - mx),  l = sum of p_t in position order,
 *   a_d = sum of p_t v_td in position order;
 * then over the query's chunks in order: mx* = max mx_c, w_c = e(mx_c - mx*),
 * L = sum w_c l_c, o_d = bf16_rne((sum w_c a_cd) / L).  e(x) for x <= 0:
 * t = x log2(e) (fp32 constant 0x3FB8AA3B); 0 if t < -126; else n = rne(t),
 * f = t - n, 2^f by the degree-6 Taylor polynomial of e^(f ln 2) in Horner
 * form with c_0 = 1, c_k = (c_(k-1) ln 2) / k (ln 2 = 0x3F317218), times 2^n.
 * Every step acc <- acc + x * y is one fused multiply-add.  A query's result
 * depends only on its own positions: the same bits for any M, for any T0
 * that leaves it the same cache positions, alone or in a batch.
 *   q      bf16 [M, Hq, D]          k, v  bf16 [S, Hkv, D]
 *   o      bf16 [M, Hq, D] out      D = 64 or 128; Hq % Hkv == 0; T0 + M <= S
 *   ws     device workspace of at least bi_attention_workspace_size(M, Hq,
 *          D, T0) bytes (null when that size is 0); its contents need no
 *          initialisation and are overwritten.
 * Device pointers, all 16-byte aligned; M <= 4096, Hq <= 65535, T0 + M <=
 * 2^20 positions, M * Hq / Hkv <= 65535 * 32.
 * One or two launches on `stream` (the second merges when the last query
 * covers more than one chunk).  Returns BI_ERR_INVALID_ARG for a null
 * pointer or an out-of-range size, BI_ERR_ALIGNMENT, BI_ERR_WORKSPACE.
 */
BI_API size_t bi_attention_workspace_size(int M, int Hq, int D, int T0);
BI_API bi_status bi_attention_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v, int M, int Hq, int Hkv,
                                     int D, int T0, int S, float scale, uint16_t *o, void *ws, size_t ws_bytes,
                                     bi_stream_t stream);

/*
 * Bandwidth probes, for measurement only: the device's own read-only and copy
 * ceilings with 16-byte streaming loads (8 in flight per thread) over a grid
 * of four 512-thread CTAs per SM.  A weight stream only reads, so the
 * read-only ceiling is the one it is measured against.
 *   bi_probe_read: reads `bytes` of `buf` once; *out (device, 8-byte aligned)
 *     = the xor of all its 64-bit words (a check that every byte was read).
 *   bi_probe_copy: dst = src, `bytes` bytes; src and dst must not overlap.
 * Device pointers, 16-byte aligned; bytes a positive multiple of 16.
 * Returns BI_ERR_INVALID_ARG or BI_ERR_ALIGNMENT for bad arguments.
 */
BI_API bi_status bi_probe_read(const void *buf, size_t bytes, unsigned long long *out, bi_stream_t stream);
BI_API bi_status bi_probe_copy(const void *src, void *dst, size_t bytes, bi_stream_t stream);

/*
 * Exhaustive check of the quotient the verify-pass executor quantises with.
 * Codes are clamp(rne(v / s), -127, 127) with v / s an IEEE fp32 division
 * (the per-token absmax quantisation of the W8A8 page, "Quantization").  The
 * executor forms v / s from r = RN(1/s) by one fused-multiply-add correction
 * instead of dividing.  This runs, for every positive finite bf16 row maximum
 * amax (scale s = RN(amax / 127) >= 2^-64) and every bf16 v with |v| <= amax
 * (about 0.99e9 pairs), that quotient and the IEEE division, and counts the
 * pairs whose codes differ or whose quotients differ at |v / s| >= 2^-8
 * (smaller quotients have code 0 either way).
 *   out  device, 8-byte aligned, 3 x uint64, overwritten: [0] pairs checked,
 *        [1] mismatches, [2] one mismatching pair (amax bits << 16 | v bits)
 *        or 0.  Read it after the stream completes.
 * Returns BI_ERR_INVALID_ARG for a null or misaligned `out`.
 */
BI_API bi_status bi_selftest_quotient(unsigned long long *out, bi_stream_t stream);

/*
 * Verify-pass executor: a program of ops run by one persistent kernel.
 *
 * A decode or verify pass is a chain of small dependent steps (quantise an
 * activation, stream a weight matrix, ...).  Launched one call at a time each
 * step pays a launch, a ramp to full memory bandwidth and a tail, which for
 * the smaller projections cost more than the weight read itself.  A program
 * runs all of them in one cooperative launch (two CTAs per SM): op i starts
 * only after every op before it has completed on the whole GPU (a grid-wide
 * barrier), so an op may read anything earlier ops wrote, while the weight
 * tiles of the ops ahead keep streaming into shared memory across the
 * barriers (weights never depend on earlier ops).  Every op gives exactly
 * the bits of the corresponding single call.
 *
 * Build once, run many times: bi_program_build validates the ops, encodes
 * the TMA descriptors and copies the program (bi_program_bytes(n_ops) bytes,
 * caller-allocated device memory, 128-byte aligned) synchronously; the
 * program refers to the ops' buffers by address, so their contents may
 * change between runs but not their addresses.  bi_program_run is one
 * asynchronous launch on `stream` (capturable in a CUDA graph once the
 * program is built); `max_tokens` is the largest M of the program's linear
 * and LM-head ops (1..16) and must be the value the program was built for.
 * The workspace follows the zero-fill rule of bi_linear_workspace_size.
 * A mismatched program or max_tokens is reported by bi_workspace_status as
 * BI_ERR_INVALID_ARG; a bounded wait that gives up as BI_ERR_TIMEOUT.
 */
typedef enum {
    BI_OP_QUANTIZE_ACT = 1, /* x, ldx, M, K -> q, s_a        (bi_quantize_act)  */
    BI_OP_LINEAR = 2,       /* q, s_a, M, K, w_q, s_w, N -> y (bi_linear_w8a8, M <= 16) */
    BI_OP_LMHEAD = 3,       /* ... -> y (logits, may be NULL), argmax (bi_lmhead_argmax) */
    BI_OP_RESIDUAL_QUANT = 4, /* y = h [M, K] in/out, x = addend (ldx), M, K -> q, s_a
                                 (bi_residual_quantize) */
    BI_OP_RELU_MUL_QUANT = 5  /* x = packed gate|up [M, ldx >= 2K], M, K -> q, s_a,
                                 y = m or NULL (bi_relu_mul_quantize) */
} bi_op_kind;

typedef struct {
    int kind;               /* bi_op_kind */
    int M, N, K;            /* N unused by the three quantising kinds */
    const uint16_t *x;      /* quantising kinds: input rows (see above) */
    int64_t ldx;
    int8_t *q;              /* quantise: output; linear / head: input */
    float *s_a;             /* quantise: output; linear / head: input */
    const int8_t *w_q;      /* linear / head weights [N, K] */
    const float *s_w;       /* [N] */
    uint16_t *y;            /* linear: output [M, N]; head: logits or NULL;
                               residual: the stream h; relu-mul: m or NULL */
    int32_t *argmax;        /* head: output [M] */
    const int32_t *draft;   /* head, optional: drafted tokens [M - 1] (see bi_greedy_verify) */
    int32_t *accept;        /* head, optional: [2] accepted count and next token, or NULL */
} bi_op;

BI_API size_t bi_program_bytes(int n_ops);
BI_API size_t bi_program_workspace_size(void);
BI_API bi_status bi_program_build(const bi_op *ops, int n_ops, void *program, size_t program_bytes);
BI_API bi_status bi_program_run(const void *program, int max_tokens, void *ws, size_t ws_bytes,
                                bi_stream_t stream);

/*
 * bi_linear_w8a8 for callers that cannot allocate device memory.
 *
 * No counterpart in the papers: this is a deployment variant.  Some callers
 * cannot call cudaMalloc or any allocating routine: code running inside a
 * custom allocator or memory-pool callback, plugins that their host framework
 * hands only input and output pointers, and processes that must not grow
 * their device memory after start-up.  This entry point allocates nothing.
 * The weight-streaming kernel's scratch (split-K partial sums, their
 * counters, a status word) is a fixed array of BI_NOALLOC_SCRATCH_BYTES
 * inside the library, present on every GPU that loads the library until the
 * process exits.  The caller still passes all inputs and outputs.
 *
 *   Arguments, layouts, results and the errors found before any launch are
 *   those of bi_linear_w8a8; there is no workspace argument.
 *   M must be <= BI_NOALLOC_MAX_M (the most the fixed scratch holds); larger
 *   M returns BI_ERR_UNSUPPORTED without launching anything.
 *   The first call on each device (and the first after the device's context
 *   was replaced, for instance by cudaDeviceReset) looks up the scratch
 *   array's device address with that device current; make that first call
 *   before any stream capture.
 *   Every call shares the one array.  The kernel leaves the scratch's counters
 *   and partial sums at zero when it completes, so a call launches with no
 *   clearing (BI_FLAG_PDL keeps its effect).  Calls that may overlap on the
 *   GPU (other streams, other host threads) race on the array and must not
 *   be issued; calls in order on one stream are fine.
 *   A wait inside the kernel that gives up (after 2 s) is recorded in the
 *   scratch's status word and leaves y partly written; later calls are then
 *   not reliable until bi_linear_w8a8_noalloc_status has reported it.
 *   Results are bitwise identical to bi_linear_w8a8.
 *
 * bi_linear_w8a8_noalloc_status: waits for `stream`, then reads the status
 * word of the scratch on the current device: BI_OK, or BI_ERR_TIMEOUT if a
 * wait of an earlier call (or of bi_selftest_wait_timeout with a NULL
 * workspace) gave up.  After a timeout it restores the whole scratch to zero,
 * so that the next call is reliable again.  Allocates nothing.
 */
#define BI_NOALLOC_MAX_M 16
#define BI_NOALLOC_SCRATCH_BYTES 2164992
BI_API bi_status bi_linear_w8a8_noalloc(const int8_t *q, const float *s_a, int M, int K,
                                        const int8_t *w_q, const float *s_w, int N,
                                        uint16_t *y, unsigned flags, bi_stream_t stream);
BI_API bi_status bi_linear_w8a8_noalloc_status(bi_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_H */
