// Row-wise quantisation kernels: per-token activation quantisation (bf16 in),
// checkpoint-style weight quantisation (fp32 in) and power-of-two scale
// requantisation of int8 weights.
//
// Arithmetic follows the W8A8 pipeline of "Deterministic LLM Inference Across
// GPU Kernels: Power-of-Two INT8 Quantization Scales and the Limits of
// Tolerance-Based Conformance" (Abstract, Fig. 1): s = absmax/127 by IEEE
// division, q = clamp(rne(v/s), -127, 127); power-of-two scales are built by
// requantising the codes, not by rewriting the scales.
#include "kernels.cuh"
#include "ptx.cuh"
#include "row_ops.cuh"

namespace bi {

namespace {

constexpr int kQuantThreads = 256;

enum RowMode { kRowPlain = 0, kRowResidual = 1, kRowReluMul = 2 };

template <int THREADS = kQuantThreads>
__device__ __forceinline__ float block_max(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = (lane < THREADS / 32) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

__device__ __forceinline__ int8_t quant1(float v, float s)
{
    int r = __float2int_rn(__fdiv_rn(v, s));  // IEEE division, round half to even
    r = max(-127, min(127, r));
    return static_cast<int8_t>(r);
}

// Load 16 consecutive elements of a row as fp32 (exact widening for bf16).
template <bool BF16>
__device__ __forceinline__ void load16(const void *row, int k, float (&v)[16])
{
    if constexpr (BF16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + k);
        uint4 a = p[0], b = p[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(row) + k);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 t = p[i];
            v[4 * i] = t.x;
            v[4 * i + 1] = t.y;
            v[4 * i + 2] = t.z;
            v[4 * i + 3] = t.w;
        }
    }
}

// One CTA per row.  Pass 1: absmax (exact; max is order-free).  Pass 2:
// quantise 16 elements per thread per step and store them as one 16-byte word.
template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(const void *__restrict__ x, int64_t ld,
                                                                      int K, int8_t *__restrict__ q,
                                                                      float *__restrict__ s_out, int pdl)
{
    __shared__ float red[kQuantThreads / 32];
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t row = blockIdx.x;
    const size_t esz = BF16 ? 2 : 4;
    const void *xr = static_cast<const char *>(x) + row * ld * esz;

    float amax = 0.0f;
    for (int k = threadIdx.x * 16; k < K; k += kQuantThreads * 16) {
        float v[16];
        load16<BF16>(xr, k, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = block_max<kQuantThreads>(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);

    int8_t *qr = q + row * K;
    for (int k = threadIdx.x * 16; k < K; k += kQuantThreads * 16) {
        float v[16];
        load16<BF16>(xr, k, v);
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t b0 = static_cast<uint8_t>(quant1(v[4 * i], s));
            uint32_t b1 = static_cast<uint8_t>(quant1(v[4 * i + 1], s));
            uint32_t b2 = static_cast<uint8_t>(quant1(v[4 * i + 2], s));
            uint32_t b3 = static_cast<uint8_t>(quant1(v[4 * i + 3], s));
            w[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
        *reinterpret_cast<uint4 *>(qr + k) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (threadIdx.x == 0) s_out[row] = s;
}

// Activation rows: one CTA of 256 threads per row.  For rows up to 16384
// elements each thread holds C chunks of 8 bf16 values in registers, so the
// row is read from memory once and the kernel is one load, one block
// reduction and one store deep; longer rows (C = 0) are read twice.  The CTA
// is small so that it fits beside a running linear-layer CTA when launched as
// a programmatic dependent.
//
// MODE selects the row's input (the elementwise steps of row_ops.cuh):
//   kRowPlain     x[row]
//   kRowResidual  bf16_rne(h[row] + x[row]), rescaled by 2^-ilogb(absmax) and
//                 written back to h (in place, row stride K)
//   kRowReluMul   bf16_rne(relu(x[row, :K]) * x[row, K:2K]), written to h if
//                 h is not null
// and the quantised codes are those of that input.
constexpr int kActThreads = 256;

struct RowArgs {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *h;
    int K;
    int8_t *q;
    float *s_a;
};

__device__ __forceinline__ uint4 ld16(const uint16_t *p) { return *reinterpret_cast<const uint4 *>(p); }

template <int MODE>
__device__ __forceinline__ uint4 row_in8(const RowArgs &a, int64_t row, int k)
{
    const uint16_t *xr = a.x + row * a.ldx;
    if constexpr (MODE == kRowResidual) return residual8(ld16(a.h + row * a.K + k), ld16(xr + k));
    if constexpr (MODE == kRowReluMul) return relu_mul8(ld16(xr + k), ld16(xr + a.K + k));
    return ld16(xr + k);
}

template <int C, int MODE>
__global__ void __launch_bounds__(kActThreads) row_quant_kernel(RowArgs a, int pdl)
{
    __shared__ float red[kActThreads / 32];
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t row = blockIdx.x;
    const int K = a.K;
    uint4 v[C > 0 ? C : 1];
    float amax = 0.0f;
    if constexpr (C > 0) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int k = (c * kActThreads + threadIdx.x) * 8;
            v[c] = (k < K) ? row_in8<MODE>(a, row, k) : make_uint4(0, 0, 0, 0);
            amax = absmax8(v[c], amax);
        }
    } else {
        for (int k = threadIdx.x * 8; k < K; k += kActThreads * 8) amax = absmax8(row_in8<MODE>(a, row, k), amax);
    }
    amax = block_max<kActThreads>(amax, red);
    int p = 0;
    if constexpr (MODE == kRowResidual) {
        p = rescale_shift(amax);
        amax = scale_pow2(amax, p);   // exact: the row's largest magnitude, rescaled
    }
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
    int8_t *qr = a.q + row * K;
    // Each thread writes only the chunks it read itself, so the in-place
    // residual update never overwrites a value another thread has yet to read.
    auto emit = [&](uint4 t, int k) {
        if constexpr (MODE == kRowResidual) {
            t = rescale8(t, p);
            *reinterpret_cast<uint4 *>(a.h + row * K + k) = t;
        }
        if constexpr (MODE == kRowReluMul) {
            if (a.h) *reinterpret_cast<uint4 *>(a.h + row * K + k) = t;
        }
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
        uint32_t o[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = static_cast<uint8_t>(quant1(bf16_lo(w[i]), s));
            const uint32_t hi = static_cast<uint8_t>(quant1(bf16_hi(w[i]), s));
            o[i >> 1] |= (lo | (hi << 8)) << (16 * (i & 1));
        }
        *reinterpret_cast<uint2 *>(qr + k) = make_uint2(o[0], o[1]);
    };
    if constexpr (C > 0) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int k = (c * kActThreads + threadIdx.x) * 8;
            if (k < K) emit(v[c], k);
        }
    } else {
        for (int k = threadIdx.x * 8; k < K; k += kActThreads * 8) emit(row_in8<MODE>(a, row, k), k);
    }
    if (threadIdx.x == 0) a.s_a[row] = s;
}

template <int MODE>
cudaError_t launch_rows(const RowArgs &a, int M, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(kActThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int p = pdl ? 1 : 0;
    const int chunks = (a.K + kActThreads * 8 - 1) / (kActThreads * 8);
    switch (chunks) {
    case 1: return cudaLaunchKernelEx(&cfg, row_quant_kernel<1, MODE>, a, p);
    case 2: return cudaLaunchKernelEx(&cfg, row_quant_kernel<2, MODE>, a, p);
    case 3: return cudaLaunchKernelEx(&cfg, row_quant_kernel<3, MODE>, a, p);
    case 4: return cudaLaunchKernelEx(&cfg, row_quant_kernel<4, MODE>, a, p);
    case 5: return cudaLaunchKernelEx(&cfg, row_quant_kernel<5, MODE>, a, p);
    case 6: return cudaLaunchKernelEx(&cfg, row_quant_kernel<6, MODE>, a, p);
    case 7: return cudaLaunchKernelEx(&cfg, row_quant_kernel<7, MODE>, a, p);
    case 8: return cudaLaunchKernelEx(&cfg, row_quant_kernel<8, MODE>, a, p);
    default: return cudaLaunchKernelEx(&cfg, row_quant_kernel<0, MODE>, a, p);
    }
}

// Round the integer p / 2^sh to nearest, ties to even (sh >= 1), symmetric in sign.
__device__ __forceinline__ int64_t rne_shift(int64_t p, int sh)
{
    const bool neg = p < 0;
    uint64_t a = static_cast<uint64_t>(neg ? -p : p);
    uint64_t fl = a >> sh;
    uint64_t rem = a & ((1ull << sh) - 1);
    uint64_t half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (fl & 1ull))) ++fl;
    return neg ? -static_cast<int64_t>(fl) : static_cast<int64_t>(fl);
}

// One CTA per row.  The scale s = mant * 2^(e - 150) (mant a 24-bit integer
// with its top bit set, after normalising subnormals) has frexp form
// m = mant / 2^24 in [0.5, 1), E = e - 126.  Its nearest power of two in the
// log domain is 2^E when m^2 >= 1/2, i.e. mant^2 >= 2^47 (exact in 64 bits),
// else 2^(E-1).  The new code is q * s / s' = q * mant / 2^(24 - (E - e2)),
// an integer divided by a power of two, rounded half to even and clamped.
__global__ void __launch_bounds__(kQuantThreads) requant_pow2_kernel(const int8_t *w_q, const float *s_w, int K,
                                                                     int8_t *w_q_out, float *s_w_out)
{
    __shared__ float s_sh;
    const int64_t row = blockIdx.x;
    if (threadIdx.x == 0) s_sh = s_w[row];
    __syncthreads();
    const float s = s_sh;
    const int8_t *src = w_q + row * K;
    int8_t *dst = w_q_out + row * K;
    const uint32_t bits = __float_as_uint(s);
    const bool usable = (s > 0.0f) && (((bits >> 23) & 0xFFu) != 0xFFu);

    float s_new = s;
    if (usable) {
        int e = static_cast<int>((bits >> 23) & 0xFFu);
        uint32_t mant = bits & 0x7FFFFFu;
        if (e == 0) {  // subnormal: normalise so bit 23 is set
            int lz = __clz(mant) - 8;
            mant <<= lz;
            e = 1 - lz;
        } else {
            mant |= 0x800000u;
        }
        const int E = e - 126;
        const uint64_t m2 = static_cast<uint64_t>(mant) * mant;
        int e2 = (m2 >= (1ull << 47)) ? E : E - 1;
        if (e2 > 127) e2 = 127;
        const int sh = 24 - (E - e2);  // 24 or 23
        s_new = (e2 >= -126) ? __uint_as_float(static_cast<uint32_t>(e2 + 127) << 23)
                             : __uint_as_float(1u << (e2 + 149));
        for (int k = threadIdx.x * 16; k < K; k += kQuantThreads * 16) {
            uint4 in = *reinterpret_cast<const uint4 *>(src + k);
            uint32_t wv[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t o = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    int c = static_cast<int8_t>((wv[i] >> (8 * b)) & 0xFFu);
                    int64_t r = rne_shift(static_cast<int64_t>(c) * mant, sh);
                    r = r > 127 ? 127 : (r < -127 ? -127 : r);
                    o |= (static_cast<uint32_t>(r) & 0xFFu) << (8 * b);
                }
                wv[i] = o;
            }
            *reinterpret_cast<uint4 *>(dst + k) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    } else if (dst != src) {
        for (int k = threadIdx.x * 16; k < K; k += kQuantThreads * 16)
            *reinterpret_cast<uint4 *>(dst + k) = *reinterpret_cast<const uint4 *>(src + k);
    }
    __syncthreads();
    if (threadIdx.x == 0) s_w_out[row] = s_new;
}

// L = first i < M - 1 with argmax[i] != draft[i] (M - 1 if none); out = {L, argmax[L]}.
__global__ void greedy_verify_kernel(const int32_t *argmax, const int32_t *draft, int M, int32_t *out)
{
    const int lane = threadIdx.x;
    int L = M - 1;
    for (int base = 0; base < M - 1; base += 32) {
        const int i = base + lane;
        const bool miss = i < M - 1 && argmax[i] != draft[i];
        const unsigned b = __ballot_sync(0xffffffffu, miss);
        if (b) {
            L = base + __ffs(b) - 1;
            break;
        }
    }
    if (lane == 0) {
        out[0] = L;
        out[1] = argmax[L];
    }
}

// One thread waits, with the library's bounded wait, on a barrier phase that
// nothing will complete; when the wait gives up it reports a timeout in the
// status word, as the linear and program kernels do.
__global__ void wait_selftest_kernel(int *status)
{
    __shared__ uint64_t bar;
    __shared__ int never;
    mbar_init(&bar, 1);
    never = 0;
    fence_mbarrier_init();
    if (!mbar_wait_bounded(&bar, 0, &never)) atomicExch(status, DEV_TIMEOUT);
}

// Every (v, amax) a quantisation row can meet: amax a positive finite bf16
// value, v a bf16 value with |v| <= amax.  For every row scale s =
// RN(amax / 127) >= kQuotientMinScale, quotient_rn(v, s, RN(1/s)) is compared
// with IEEE division: the code always, the value wherever IEEE division's
// quotient is at least 2^-8.  One block per amax bit pattern.
// out[0] += pairs checked, out[1] += mismatches, out[2] = a mismatch found
// (amax bits << 16 | v bits), if any.
__global__ void __launch_bounds__(256) quotient_selftest_kernel(unsigned long long *out)
{
    const uint32_t a_bits = blockIdx.x + 1u;   // 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(a_bits << 16);
    const float s = __fdiv_rn(amax, 127.0f);
    if (s < kQuotientMinScale) return;
    const float r = __frcp_rn(s);
    unsigned long long checked = 0, bad = 0;
    for (uint32_t vb = threadIdx.x; vb <= a_bits; vb += blockDim.x)
        for (uint32_t sign = 0; sign < 2; ++sign) {
            const uint32_t v_bits = vb | (sign << 15);
            const float v = __uint_as_float(v_bits << 16);
            const float q = quotient_rn(v, s, r);
            const float q_ref = __fdiv_rn(v, s);
            ++checked;
            // codes always; quotients from 2^-8 up, where every code is
            // decided (smaller quotients round to code 0 either way)
            if (code_byte(q) != code_byte(q_ref) || (fabsf(q_ref) >= 0x1p-8f && q != q_ref)) {
                ++bad;
                out[2] = (static_cast<unsigned long long>(a_bits) << 16) | v_bits;
            }
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        checked += __shfl_xor_sync(0xffffffffu, checked, o);
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&out[0], checked);
        if (bad) atomicAdd(&out[1], bad);
    }
}

}  // namespace

cudaError_t launch_quotient_selftest(unsigned long long *out, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(out, 0, 3 * sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return e;
    quotient_selftest_kernel<<<0x7F7Fu, 256, 0, stream>>>(out);
    return cudaGetLastError();
}

cudaError_t launch_quantize_act(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *s_a, bool pdl,
                                cudaStream_t stream)
{
    const RowArgs a = {x, ldx, nullptr, K, q, s_a};
    return launch_rows<kRowPlain>(a, M, pdl, stream);
}

cudaError_t launch_residual_quantize(uint16_t *h, const uint16_t *y, int64_t ldy, int M, int K, int8_t *q,
                                     float *s_a, bool pdl, cudaStream_t stream)
{
    const RowArgs a = {y, ldy, h, K, q, s_a};
    return launch_rows<kRowResidual>(a, M, pdl, stream);
}

cudaError_t launch_relu_mul_quantize(const uint16_t *gu, int64_t ldgu, int M, int K, int8_t *q, float *s_a,
                                     uint16_t *m_out, bool pdl, cudaStream_t stream)
{
    const RowArgs a = {gu, ldgu, m_out, K, q, s_a};
    return launch_rows<kRowReluMul>(a, M, pdl, stream);
}

cudaError_t launch_greedy_verify(const int32_t *argmax, const int32_t *draft, int M, int32_t *out,
                                 cudaStream_t stream)
{
    greedy_verify_kernel<<<1, 32, 0, stream>>>(argmax, draft, M, out);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int *status, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 1, 0, stream>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_quantize_weight(const float *w, int64_t ldw, int N, int K, int8_t *w_q, float *s_w,
                                   cudaStream_t stream)
{
    quantize_rows_kernel<false><<<static_cast<unsigned>(N), kQuantThreads, 0, stream>>>(w, ldw, K, w_q, s_w, 0);
    return cudaGetLastError();
}

cudaError_t launch_requant_pow2(const int8_t *w_q, const float *s_w, int N, int K, int8_t *w_q_out, float *s_w_out,
                                cudaStream_t stream)
{
    requant_pow2_kernel<<<static_cast<unsigned>(N), kQuantThreads, 0, stream>>>(w_q, s_w, K, w_q_out, s_w_out);
    return cudaGetLastError();
}

}  // namespace bi
