/*
 * CPU oracle for the batch-invariant verify pass: the W8A8 linear layer and
 * LM-head argmax, the chained pass's elementwise steps, the block-scaled
 * variant and the split-KV attention of the verify queries.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header or table with the CUDA library and calls nothing in it.
 *
 * Plain scalar C, built with -O2 -ffp-contract=off and no fast-math, so every
 * float operation below is one IEEE-754 operation rounded to nearest-even; an
 * explicit fmaf (the attention's multiply-accumulate steps) is one fused
 * operation with one rounding.
 * Sums of int8 products are carried in int64 (exact) and checked against the
 * int32 range.  Loops run in the textbook order; the only parallelism is an
 * OpenMP loop over independent output elements, which cannot change a result.
 *
 * Sources (page title, section / table):
 *  [chen]   "Deterministic LLM Inference Across GPU Kernels: Power-of-Two INT8
 *           Quantization Scales and the Limits of Tolerance-Based Conformance",
 *           Abstract, Fig. 1, Table II (epilogue faults F1-F5).
 *  [alibi]  "The Integer Alibi: Localizing Cross-Kernel Divergence in
 *           INT8-Quantized LLM Inference" (abstract on the same page).
 *  [cintu]  "why speculative decoding changed my output", sections
 *           "floats care about order" and "the mat-vec kernel".
 *  [goyal]  "My speculative decoder got slower", sections "Why the decoders
 *           disagreed?" (bf16 tie 30.0 / 29.875) and "We're nowhere near SOL"
 *           (a vocab head that computes only the winning token).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 -> fp32 is exact: a bf16 value is the top half of an fp32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/*
 * fp32 -> bf16, round to nearest, ties to even (the output rounding the
 * epilogue must use; output truncation is fault F4 in [chen] Table II).
 * Written from the definition: the two bf16 neighbours of f are the pattern
 * with the low 16 bits cleared (toward zero) and the next pattern away from
 * zero; pick the one nearer to f, and the one with an even last bit on a tie.
 * The distances are exact in double (f has 24 significant bits).  Overflow
 * rounds to infinity exactly as IEEE round-to-nearest does; NaN becomes the
 * quiet NaN 0x7FC0 (the oracle never produces one from finite inputs).
 */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f))
        return 0x7FC0;
    uint16_t toward0 = (uint16_t)(u >> 16);
    if ((u & 0xFFFFu) == 0)
        return toward0;                      /* already a bf16 value */
    uint16_t away = (uint16_t)(toward0 + 1); /* next magnitude (may be Inf) */
    double vf = (double)f;
    double v0 = (double)oracle_bf16_to_f32(toward0);
    double v1;
    if ((away & 0x7FFFu) == 0x7F80u) {
        /* the next magnitude is infinity: compare with 2^128, the value the
           unbounded-exponent format would hold there */
        v1 = (away & 0x8000u) ? -ldexp(1.0, 128) : ldexp(1.0, 128);
    } else {
        v1 = (double)oracle_bf16_to_f32(away);
    }
    double d0 = fabs(vf - v0), d1 = fabs(v1 - vf);
    if (d0 < d1) return toward0;
    if (d1 < d0) return away;
    return (toward0 & 1u) ? away : toward0;   /* tie: even last bit */
}

/* Array form of oracle_f32_to_bf16_rne, for exhaustive checks. */
void oracle_f32_to_bf16_rne_array(const float *f, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16_rne(f[i]);
}

/* Round a double to the nearest integer, ties to even, written out. */
static double rne_to_int(double v)
{
    double fl = floor(v);
    double frac = v - fl;                   /* exact for |v| < 2^52 */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

static int8_t clamp127(double r)
{
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

/* ------------------------------------------------ per-row absmax quantisation
 *
 * W8A8 (the "INT8 pipeline" of [chen] Abstract / Fig. 1; the scale rule is the
 * plain absmax one): s = absmax / 127 as one IEEE fp32 division (s = 1 for an
 * all-zero row), q = clamp(rne(v / s), -127, 127) with the quotient an IEEE
 * fp32 division.  -128 is never produced.
 */
static void quantize_row_f32(const float *v, int K, int8_t *q, float *s_out)
{
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
        float a = fabsf(v[k]);
        if (a > amax) amax = a;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 127.0f;
    for (int k = 0; k < K; ++k) {
        float t = v[k] / s;                 /* fp32 division, RNE */
        q[k] = clamp127(rne_to_int((double)t));
    }
    *s_out = s;
}

/* A1: per-token activation quantisation of bf16 x [M, K] (row stride ldx). */
void oracle_quantize_act(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *s_a)
{
    float *row = (float *)malloc(sizeof(float) * (size_t)K);
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < K; ++k)
            row[k] = oracle_bf16_to_f32(x[(int64_t)m * ldx + k]);
        quantize_row_f32(row, K, q + (int64_t)m * K, &s_a[m]);
    }
    free(row);
}

/* Checkpoint-style per-output-channel weight quantisation of fp32 W [N, K]. */
void oracle_quantize_weight(const float *w, int N, int K, int8_t *wq, float *s_w)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        quantize_row_f32(w + (int64_t)n * K, K, wq + (int64_t)n * K, &s_w[n]);
}

/* --------------------------------------------- power-of-two requantisation
 *
 * [chen] Abstract and Fig. 1: every weight scale moves to its nearest power
 * of two, and the weights are requantised to the new scale (rewriting the
 * scale alone is the artefact the paper warns about).
 *
 * Reading: "nearest" is taken in the log domain, s' = 2^round(log2 s).  With
 * s = m * 2^E, m in [0.5, 1) (frexp), log2 s = E + log2 m and log2 m is in
 * [-1, 0), so s' = 2^E when m >= 2^-1/2, else 2^(E-1).  m >= 2^-1/2 is decided
 * exactly as m*m >= 0.5 (m has 24 bits, m*m is exact in double).  A tie would
 * need m = 2^-1/2, which is irrational, so none exists.  The new codes are
 * clamp(rne(q * s / s'), -127, 127), each product exact in double.  A scale
 * whose power of two would overflow fp32 is held at 2^127.  Rows whose scale
 * is not a positive finite number are copied unchanged.
 */
void oracle_requant_pow2(const int8_t *wq, const float *s_w, int N, int K,
                         int8_t *wq_out, float *s_out)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        float s = s_w[n];
        const int8_t *src = wq + (int64_t)n * K;
        int8_t *dst = wq_out + (int64_t)n * K;
        if (!(s > 0.0f) || isinf(s)) {
            memmove(dst, src, (size_t)K);
            s_out[n] = s;
            continue;
        }
        int E;
        double m = frexp((double)s, &E);
        int e2 = (m * m >= 0.5) ? E : E - 1;
        if (e2 > 127) e2 = 127;
        double sp = ldexp(1.0, e2);
        for (int k = 0; k < K; ++k) {
            double v = (double)src[k] * (double)s / sp;
            dst[k] = clamp127(rne_to_int(v));
        }
        s_out[n] = (float)sp;
    }
}

/* ------------------------------------------------------- linear + epilogue
 *
 * acc[m,n] = sum_k q[m,k] * W[n,k]   exact integer sum ([alibi]: for shared
 *            int8 operands under a no-overflow bound the int32 dot product is
 *            exact and independent of order; K * 127^2 < 2^31).
 * y[m,n]   = bf16_rne( (float(acc) * s_a[m]) * s_w[n] )
 *            [chen] Table II read as the correct epilogue: scales stay fp32
 *            (not F1), the two multiplies are separate fp32 roundings with no
 *            bf16 rounding between them (not F2), acc*s_a first, then *s_w
 *            (not F3), one final round-to-nearest-even (not F4), scales never
 *            enter the integer sum (not F5).  int32 -> fp32 rounds to nearest
 *            even (C conversion in the default rounding mode).
 * Returns 0, or -1 if some |acc| reached 2^31 (the overflow precondition).
 */
int oracle_linear_w8a8(const int8_t *q, const float *s_a, int M, int K,
                       const int8_t *wq, const float *s_w, int N, uint16_t *y)
{
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int n = 0; n < N; ++n) {
        const int8_t *w = wq + (int64_t)n * K;
        for (int m = 0; m < M; ++m) {
            const int8_t *a = q + (int64_t)m * K;
            int64_t acc = 0;
            for (int k = 0; k < K; ++k)
                acc += (int64_t)a[k] * (int64_t)w[k];
            if (acc >= 2147483648LL || acc <= -2147483648LL) {
                bad = 1;
                acc = 0;
            }
            float f = (float)(int32_t)acc;
            f = f * s_a[m];
            f = f * s_w[n];
            y[(int64_t)m * N + n] = oracle_f32_to_bf16_rne(f);
        }
    }
    return bad ? -1 : 0;
}

/*
 * Greedy LM-head argmax over the bf16 logits of each row: the lowest index n
 * whose logit equals the row maximum, logits compared as real numbers (so -0
 * equals +0).  Greedy decoding keeps the target's own argmax ([cintu] intro,
 * [goyal] "Speculative decoding (SD)"); [goyal] shows bf16 logits tying
 * (29.875 vs 29.875), so the tie rule is part of the contract.  The head
 * reuses oracle_linear_w8a8 for the logits; `logits` may be NULL.
 */
int oracle_lmhead_argmax(const int8_t *q, const float *s_a, int M, int K,
                         const int8_t *wq, const float *s_w, int N,
                         uint16_t *logits, int32_t *argmax)
{
    uint16_t *y = logits ? logits : (uint16_t *)malloc(sizeof(uint16_t) * (size_t)M * (size_t)N);
    int rc = oracle_linear_w8a8(q, s_a, M, K, wq, s_w, N, y);
    for (int m = 0; m < M; ++m) {
        int32_t best = 0;
        float bv = oracle_bf16_to_f32(y[(int64_t)m * N]);
        for (int n = 1; n < N; ++n) {
            float v = oracle_bf16_to_f32(y[(int64_t)m * N + n]);
            if (v > bv) {
                bv = v;
                best = n;
            }
        }
        argmax[m] = best;
    }
    if (!logits) free(y);
    return rc;
}

/* ------------------------------------------- chained verify pass (elementwise)
 *
 * The pages measure a decode/verify pass as a chain of layers whose linears
 * read the previous ones' outputs ([cintu] "the mat-vec kernel", [goyal]
 * "The physics"), but print no layer body.  Reading (no attention): the q
 * slice of the packed q/k/v output stands in for the attention output; the
 * residual stream h is updated twice per layer; the MLP gate is a ReLU (no
 * transcendental, so both sides round identically).  Each step below is one
 * IEEE fp32 operation on bf16 inputs followed by one bf16 rounding.  Because
 * fp32 has 24 >= 2*8+2 significand bits, an fp32 add or multiply of bf16
 * values followed by bf16 rounding equals a single rounding of the exact
 * result, so these have a plain definition (checked against exact rationals).
 */

/*
 * Residual add with a power-of-two row rescale, in place on h [M, K] (row
 * stride K):  h' = bf16_rne(h + y)  (fp32 add);  e = ilogb(max_k |h'|)
 * (e = 0 for an all-zero row);  h = bf16_rne(h' * 2^-e).  The rescale keeps a
 * 36-layer stack finite and changes no quantisation code: per-row absmax
 * quantisation is exactly invariant to multiplying a row by a power of two.
 * The product is formed in double (exact) and rounded to fp32 then bf16; it is
 * exact except below 2^-142, where both roundings give a signed zero.
 */
void oracle_residual_rescale(uint16_t *h, const uint16_t *y, int64_t ldy, int M, int K)
{
    uint16_t *t = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K);
    for (int m = 0; m < M; ++m) {
        uint16_t *hr = h + (int64_t)m * K;
        const uint16_t *yr = y + (int64_t)m * ldy;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float sum = oracle_bf16_to_f32(hr[k]) + oracle_bf16_to_f32(yr[k]);
            t[k] = oracle_f32_to_bf16_rne(sum);
            float a = fabsf(oracle_bf16_to_f32(t[k]));
            if (a > amax) amax = a;
        }
        int e = (amax == 0.0f) ? 0 : ilogbf(amax);
        for (int k = 0; k < K; ++k) {
            double scaled = ldexp((double)oracle_bf16_to_f32(t[k]), -e);
            hr[k] = oracle_f32_to_bf16_rne((float)scaled);
        }
    }
    free(t);
}

/*
 * MLP product: out[m, k] = bf16_rne(relu(g) * u) with g = gu[m, k] and
 * u = gu[m, K + k] (the gate and up halves of one packed gate/up output, row
 * stride ld >= 2K), relu(g) = g if g > 0 else +0, the product one fp32
 * multiply (exact for two bf16 values in the normal range).
 */
void oracle_relu_mul(const uint16_t *gu, int64_t ld, int M, int K, uint16_t *out)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t *r = gu + (int64_t)m * ld;
        for (int k = 0; k < K; ++k) {
            float g = oracle_bf16_to_f32(r[k]);
            float u = oracle_bf16_to_f32(r[K + k]);
            float gr = (g > 0.0f) ? g : 0.0f;
            out[(int64_t)m * K + k] = oracle_f32_to_bf16_rne(gr * u);
        }
    }
}

/* ------------------------------------------------------- greedy verification
 *
 * Greedy speculative decoding keeps exactly the tokens plain greedy decoding
 * would produce ([cintu] introduction; [goyal] "Speculative decoding (SD)"):
 * the verify pass runs the target on the last accepted token followed by the
 * M - 1 drafted tokens d_1 .. d_{M-1}; row i's argmax a_i is the target's
 * choice for the token after input i.  Drafted token d_{i+1} is accepted
 * while it equals a_i, so the accepted count L is the length of the longest
 * prefix with a_i == d_{i+1} (0 <= L <= M - 1), and the next token is a_L
 * (the correction after a rejection, or the bonus token when every draft is
 * accepted).  out[0] = L, out[1] = a_L.
 */
void oracle_greedy_verify(const int32_t *argmax, const int32_t *draft, int M, int32_t *out)
{
    int L = 0;
    while (L < M - 1 && argmax[L] == draft[L])
        ++L;
    out[0] = L;
    out[1] = argmax[L];
}

/* ------------------------------------------------ block-scaled variant
 *
 * The mat-vec of [cintu] "the mat-vec kernel": a weight row of K inputs is cut
 * into blocks of 256 weights, the activations into int8 blocks of 32; the
 * products inside a block are integer (exact in any order), and each block's
 * integer result is scaled and added into an fp32 accumulator, whose order
 * of adds must be the same for every number of tokens in the pass.
 *
 * The pages name the formats (q6_k weights, int8 activation blocks of 32) but
 * print no layout and no quantiser, so this library defines its own:
 *  - weights: super-blocks of 256 = 16 sub-blocks of 16.  Code c in [-32, 31]
 *    (6 bits), int8 sub-scale sc per sub-block, fp32 scale d per super-block;
 *    w ~ c * (d * sc).  Stored as ql [N][K/2] (low 4 bits of c + 32; element k
 *    in byte k/2, bits 4 * (k & 1)), qh [N][K/4] (high 2 bits of c + 32;
 *    element k in byte k/4, bits 2 * (k & 3)), sc [N][K/16], d [N][K/256].
 *  - quantiser, per super-block: t_j = absmax_j / 31 (fp32 division) for each
 *    sub-block j; d = max_j t_j / 127 (1 if all zero); sc_j = clamp(rne(t_j /
 *    d), 0, 127); e_j = d * sc_j (fp32); c = clamp(rne(w / e_j), -32, 31), or 0
 *    when e_j = 0.
 *  - activations: blocks of 32 with the per-token rule of A1 applied to each
 *    block: d_a = absmax / 127 (1 if zero), q = clamp(rne(x / d_a), +-127).
 *  - the sum: 32-block b (of K / 32) of super-block s = b / 8 holds sub-blocks
 *    j = 16 s + 2 (b % 8) and j + 1; isum_b = sc_j * sum(c * q) over its first
 *    16 elements + sc_(j+1) * sum over the next 16 (|isum| < 2^24, exact in
 *    fp32); contribution v_b = ((float)isum_b * d_a[b]) * d[s].  Lane l
 *    (0..31) adds v_l, v_(l+32), v_(l+64), ... in that order into a partial
 *    starting at +0; then, for offsets 16, 8, 4, 2, 1, every partial becomes
 *    p[l] + p[l xor offset]; y = p[0] (fp32, not rounded further).  The order
 *    depends on K only, so every token of every pass gets the same adds.
 */
static float rne_f(double v) { return (float)rne_to_int(v); }

void oracle_quantize_q6(const float *w, int N, int K, uint8_t *ql, uint8_t *qh, int8_t *sc, float *d)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const float *wr = w + (int64_t)n * K;
        for (int s = 0; s < K / 256; ++s) {
            float t[16], tmax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float amax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    float a = fabsf(wr[256 * s + 16 * j + i]);
                    if (a > amax) amax = a;
                }
                t[j] = amax / 31.0f;
                if (t[j] > tmax) tmax = t[j];
            }
            float ds = (tmax == 0.0f) ? 1.0f : tmax / 127.0f;
            d[(int64_t)n * (K / 256) + s] = ds;
            for (int j = 0; j < 16; ++j) {
                float r = rne_f((double)(t[j] / ds));
                if (r > 127.0f) r = 127.0f;
                if (r < 0.0f) r = 0.0f;
                int8_t scj = (int8_t)r;
                sc[(int64_t)n * (K / 16) + 16 * s + j] = scj;
                float e = ds * (float)scj;
                for (int i = 0; i < 16; ++i) {
                    int64_t k = 256 * s + 16 * j + i;
                    int c = 0;
                    if (e != 0.0f) {
                        float v = rne_f((double)(wr[k] / e));
                        if (v > 31.0f) v = 31.0f;
                        if (v < -32.0f) v = -32.0f;
                        c = (int)v;
                    }
                    unsigned u = (unsigned)(c + 32);
                    uint8_t *bl = &ql[(int64_t)n * (K / 2) + k / 2];
                    uint8_t *bh = &qh[(int64_t)n * (K / 4) + k / 4];
                    if ((k & 1) == 0) *bl = (uint8_t)((*bl & 0xF0u) | (u & 0xFu));
                    else *bl = (uint8_t)((*bl & 0x0Fu) | ((u & 0xFu) << 4));
                    unsigned sh = 2u * (unsigned)(k & 3);
                    *bh = (uint8_t)((*bh & ~(3u << sh)) | (((u >> 4) & 3u) << sh));
                }
            }
        }
    }
}

/* The code of weight k in row n of a block-scaled matrix (layout above). */
int oracle_q6_code(const uint8_t *ql, const uint8_t *qh, int K, int n, int k)
{
    unsigned lo = (ql[(int64_t)n * (K / 2) + k / 2] >> (4 * (k & 1))) & 0xFu;
    unsigned hi = (qh[(int64_t)n * (K / 4) + k / 4] >> (2 * (k & 3))) & 3u;
    return (int)(lo | (hi << 4)) - 32;
}

void oracle_quantize_act_blocks(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *d_a)
{
    float row[32];
    for (int m = 0; m < M; ++m)
        for (int b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i)
                row[i] = oracle_bf16_to_f32(x[(int64_t)m * ldx + 32 * b + i]);
            quantize_row_f32(row, 32, q + (int64_t)m * K + 32 * b, &d_a[(int64_t)m * (K / 32) + b]);
        }
}

void oracle_linear_q6(const int8_t *qa, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                      const int8_t *sc, const float *d, int N, float *y)
{
    const int nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m) {
            float p[32];
            for (int l = 0; l < 32; ++l) {
                p[l] = 0.0f;
                for (int b = l; b < nb; b += 32) {
                    int s = b / 8, j = 16 * s + 2 * (b % 8);
                    int64_t part[2] = {0, 0};
                    for (int i = 0; i < 32; ++i) {
                        int k = 32 * b + i;
                        part[i / 16] += (int64_t)oracle_q6_code(ql, qh, K, n, k) * qa[(int64_t)m * K + k];
                    }
                    int64_t isum = (int64_t)sc[(int64_t)n * (K / 16) + j] * part[0] +
                                   (int64_t)sc[(int64_t)n * (K / 16) + j + 1] * part[1];
                    float v = ((float)isum * d_a[(int64_t)m * nb + b]) * d[(int64_t)n * (K / 256) + s];
                    p[l] = p[l] + v;
                }
            }
            for (int off = 16; off > 0; off /= 2) {
                float q2[32];
                for (int l = 0; l < 32; ++l) q2[l] = p[l] + p[l ^ off];
                memcpy(p, q2, sizeof(p));
            }
            y[(int64_t)m * N + n] = p[0];
        }
}

/* ------------------------------------------------ split-KV attention
 *
 * The verify pass's attention, batch-invariant: "My speculative decoder got
 * slower" (the split-KV attention: the cache cut into 256-token chunks, one
 * partial result per chunk, then a merge; one chunk writes the output
 * directly) and "why speculative decoding changed my output" (section
 * "attention": a batch of queries must use the one-query geometry).
 *
 * Readings used on both sides:
 *  - every step acc <- acc + x * y below is one fused multiply-add
 *    (fmaf: one rounding); every other operation is one fp32 operation;
 *  - query m (of M) attends to cache positions 0 .. T0 + m (causal);
 *    head h uses kv head h / (Hq / Hkv); s_t = (sum over d in order of
 *    q_d * k_td, fp32, from +0) * scale;
 *  - chunk c holds positions 256 c .. 256 c + 255 of those; per chunk:
 *    mx = max s_t; p_t = e(s_t - mx); l = sum of p_t in position order;
 *    a_d = sum of p_t * v_td in position order (fp32, from +0);
 *  - merge over chunks in order: mx* = max mx_c; w_c = e(mx_c - mx*);
 *    L = sum w_c * l_c; o_d = (sum w_c * a_cd) / L; o is rounded to bf16.
 *    With one chunk w_0 = e(0) = 1 and the merge changes nothing.
 *  - e(x), x <= 0: t = x * log2(e); 0 if t < -126; else n = rne(t),
 *    f = t - n (exact, |f| <= 1/2), 2^f by the Taylor polynomial of
 *    e^(f ln 2) to degree 6, times 2^n (one rounding).  ln 2 and log2(e) are
 *    their fp32 roundings (0x3F317218, 0x3FB8AA3B); the coefficients come
 *    from the recurrence c_0 = 1, c_k = (c_(k-1) * ln 2) / k in fp32; the
 *    polynomial is evaluated by Horner, p <- p * f + c_k (fused) per step.
 * The chunk count follows the positions a query sees, never the allocated
 * cache size.
 */
static const float kLn2 = 0.693147182464599609375f;    /* ln 2 rounded to fp32 (0x3F317218) */
static const float kLog2e = 1.44269502162933349609375f; /* log2(e) rounded to fp32 (0x3FB8AA3B) */

static float e_f32(float x)
{
    float c[7];
    c[0] = 1.0f;
    for (int k = 1; k < 7; ++k) {
        float u = c[k - 1] * kLn2;
        c[k] = u / (float)k;
    }
    float t = x * kLog2e;
    if (t < -126.0f) return 0.0f;
    float n = rne_f((double)t);
    float f = t - n;
    float p = c[6];
    for (int k = 5; k >= 0; --k) p = fmaf(p, f, c[k]);
    return ldexpf(p, (int)n);
}

float oracle_attn_exp(float x) { return e_f32(x); }

/* One chunk: positions t0 .. t1 - 1 (t1 - t0 <= 256) of kv head hk for the
 * query row qr [D]: its maximum score mx, weight sum l and weighted values a [D]. */
void oracle_attention_chunk(const uint16_t *qr, const uint16_t *kc, const uint16_t *vc, int Hkv, int hk, int D,
                            int t0, int t1, float scale, float *mx_out, float *l_out, float *a)
{
    float s[256];
    float mx = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        const uint16_t *kr = kc + ((int64_t)t * Hkv + hk) * D;
        float acc = 0.0f;
        for (int d = 0; d < D; ++d) acc = fmaf(oracle_bf16_to_f32(qr[d]), oracle_bf16_to_f32(kr[d]), acc);
        s[t - t0] = acc * scale;
        if (s[t - t0] > mx) mx = s[t - t0];
    }
    float l = 0.0f;
    for (int d = 0; d < D; ++d) a[d] = 0.0f;
    for (int t = t0; t < t1; ++t) {
        const float p = e_f32(s[t - t0] - mx);
        l = l + p;
        const uint16_t *vr = vc + ((int64_t)t * Hkv + hk) * D;
        for (int d = 0; d < D; ++d) a[d] = fmaf(p, oracle_bf16_to_f32(vr[d]), a[d]);
    }
    *mx_out = mx;
    *l_out = l;
}

/* The merge of C chunk results (mxc [C], lc [C], ac [C][D]) into o [D] (bf16). */
void oracle_attention_merge(int C, const float *mxc, const float *lc, const float *ac, int D, uint16_t *o)
{
    float mx = mxc[0];
    for (int c = 1; c < C; ++c)
        if (mxc[c] > mx) mx = mxc[c];
    float L = 0.0f;
    for (int c = 0; c < C; ++c) L = fmaf(e_f32(mxc[c] - mx), lc[c], L);
    for (int d = 0; d < D; ++d) {
        float num = 0.0f;
        for (int c = 0; c < C; ++c) num = fmaf(e_f32(mxc[c] - mx), ac[(size_t)c * D + d], num);
        o[d] = oracle_f32_to_bf16_rne(num / L);
    }
}

void oracle_attention(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, int M, int Hq, int Hkv, int D,
                      int T0, float scale, uint16_t *o)
{
    const int g = Hq / Hkv;
#pragma omp parallel for schedule(static) collapse(2)
    for (int m = 0; m < M; ++m)
        for (int h = 0; h < Hq; ++h) {
            const int T = T0 + m + 1;                  /* positions 0 .. T0 + m */
            const int C = (T + 255) / 256;
            float *mxc = (float *)malloc(sizeof(float) * C), *lc = (float *)malloc(sizeof(float) * C);
            float *ac = (float *)malloc(sizeof(float) * (size_t)C * D);
            for (int c = 0; c < C; ++c) {
                const int t0 = 256 * c, t1 = (t0 + 256 < T) ? t0 + 256 : T;
                oracle_attention_chunk(q + ((int64_t)m * Hq + h) * D, kc, vc, Hkv, h / g, D, t0, t1, scale, &mxc[c],
                                       &lc[c], ac + (size_t)c * D);
            }
            oracle_attention_merge(C, mxc, lc, ac, D, o + ((int64_t)m * Hq + h) * D);
            free(mxc);
            free(lc);
            free(ac);
        }
}

/* Number of OpenMP threads the parallel loops above use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the parallel loops above (timing only: every result is the same
 * for any thread count, each output element being computed by one thread). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
