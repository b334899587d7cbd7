// Elementwise steps of a chained verify pass on packed bf16 (8 values in a
// uint4), shared by the stand-alone row kernels and the program executor.
//
// A decode or verify pass chains its linears through the residual stream
// ("why speculative decoding changed my output", "the mat-vec kernel"; "My
// speculative decoder got slower", "The physics").  The pages print no layer
// body; the steps here are the chained pass this library runs:
//   residual:  h' = bf16_rne(h + y), then h = bf16_rne(h' * 2^-e) with
//              e = ilogb(max |h'|) over the row (0 for an all-zero row);
//   MLP gate:  m = bf16_rne(relu(g) * u), relu(g) = g if g > 0 else +0.
// Every step is one IEEE fp32 operation on bf16 values and one bf16 rounding;
// fp32 carries 24 >= 2*8+2 bits, so that equals one rounding of the exact
// result.  The power-of-two rescale changes no code of the per-row absmax
// quantisation that follows it.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace bi {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 bit pattern, round to nearest, ties to even, in integer
// arithmetic (conversion instructions issue at a fraction of the ALU rate).
// Adding 0x7FFF plus the pattern's lowest kept bit carries into the kept half
// exactly when the dropped half is above the midpoint, or at it with an odd
// kept half; a carry out of the significand moves to the next binade or to
// infinity, as IEEE rounding does.  NaN gives 0x7FC0 (never produced here:
// the steps see finite values only).
__device__ __forceinline__ uint32_t bf16_rne_bits(float f)
{
    const uint32_t u = __float_as_uint(f);
    const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return (u & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC0u : r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return bf16_rne_bits(lo) | (bf16_rne_bits(hi) << 16);
}

__device__ __forceinline__ float absmax8(const uint4 &t, float amax)
{
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        amax = fmaxf(amax, fabsf(bf16_lo(w[e])));
        amax = fmaxf(amax, fabsf(bf16_hi(w[e])));
    }
    return amax;
}

// bf16_rne(h + y) elementwise (one fp32 add each).
__device__ __forceinline__ uint4 residual8(const uint4 &h, const uint4 &y)
{
    const uint32_t a[4] = {h.x, h.y, h.z, h.w};
    const uint32_t b[4] = {y.x, y.y, y.z, y.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16x2(__fadd_rn(bf16_lo(a[e]), bf16_lo(b[e])), __fadd_rn(bf16_hi(a[e]), bf16_hi(b[e])));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float relu_pos(float g) { return g > 0.0f ? g : 0.0f; }

// bf16_rne(relu(g) * u) elementwise (one fp32 multiply each).
__device__ __forceinline__ uint4 relu_mul8(const uint4 &g, const uint4 &u)
{
    const uint32_t a[4] = {g.x, g.y, g.z, g.w};
    const uint32_t b[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16x2(__fmul_rn(relu_pos(bf16_lo(a[e])), bf16_lo(b[e])),
                           __fmul_rn(relu_pos(bf16_hi(a[e])), bf16_hi(b[e])));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// floor(log2 a) for a positive finite fp32 value (subnormals included).
__device__ __forceinline__ int ilog2_pos(float a)
{
    const uint32_t b = __float_as_uint(a);
    const int ex = static_cast<int>((b >> 23) & 0xFFu);
    if (ex != 0) return ex - 127;
    return (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// 2^p as fp32 for p in [-149, 127] (exact).
__device__ __forceinline__ float pow2f(int p)
{
    return p >= -126 ? __uint_as_float(static_cast<uint32_t>(p + 127) << 23) : __uint_as_float(1u << (p + 149));
}

// The residual rescale exponent of a row with absmax `amax` (bf16 values):
// returns p = -e, with e = floor(log2 amax), or 0 for a zero row.  p lies in
// [-127, 133] (bf16 magnitudes span [2^-133, 2^128)).
__device__ __forceinline__ int rescale_shift(float amax) { return amax == 0.0f ? 0 : -ilog2_pos(amax); }

// v * 2^p rounded once to fp32.  For p <= 127 one multiply by the exact power;
// above that (a row whose absmax is subnormal) two exact multiplies, since the
// values grow and every product is exact.
__device__ __forceinline__ float scale_pow2(float v, int p)
{
    return p <= 127 ? __fmul_rn(v, pow2f(p)) : __fmul_rn(__fmul_rn(v, pow2f(64)), pow2f(p - 64));
}

// bf16_rne(t * 2^p) elementwise.  t holds bf16 values (8 significant bits), so
// the fp32 product is exact unless it falls below 2^-142, where the fp32 and
// the bf16 rounding both give a signed zero.
__device__ __forceinline__ uint4 rescale8(const uint4 &t, int p)
{
    const uint32_t a[4] = {t.x, t.y, t.z, t.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(scale_pow2(bf16_lo(a[e]), p), scale_pow2(bf16_hi(a[e]), p));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// bf16_rne(t * f) elementwise for an exact power of two f (a normal or
// subnormal fp32 value): the form of rescale8 for shifts p <= 127.
__device__ __forceinline__ uint4 scale8(const uint4 &t, float f)
{
    const uint32_t a[4] = {t.x, t.y, t.z, t.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(__fmul_rn(bf16_lo(a[e]), f), __fmul_rn(bf16_hi(a[e]), f));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Correctly rounded fp32 quotient v / s, given r = RN(1/s), by one
// fused-multiply-add correction (Markstein's division step; P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(v r) is within one ulp
// of v / s, the remainder v - q0 s is exact in one fma, and RN(q0 + rem r)
// is RN(v / s) when nothing underflows.  It is used for rows whose scale s is
// at least 2^-64, where the remainder of any quotient from 2^-8 up is a
// normal number; smaller quotients may differ from IEEE division's in their
// last bits, but round to code 0 either way.  The library's self-test checks
// codes for every bf16 v and every bf16 row maximum, and quotients from 2^-8
// up.
__device__ __forceinline__ float quotient_rn(float v, float s, float r)
{
    const float q0 = __fmul_rn(v, r);
    const float rem = __fmaf_rn(-q0, s, v);
    return __fmaf_rn(rem, r, q0);
}

// The smallest row scale whose codes take quotient_rn.
constexpr float kQuotientMinScale = 0x1p-64f;

// clamp(rne(q), -127, 127) for |q| < 2^22 by one fp32 add: q + 1.5 * 2^23 lies
// in [2^23, 2^24), where the fp32 spacing is 1, so the add rounds q to the
// nearest integer, ties to even, and that integer is the sum's bit pattern
// minus the pattern of 1.5 * 2^23.
__device__ __forceinline__ uint32_t code_byte(float q)
{
    const float u = __fadd_rn(q, 12582912.0f);   // 1.5 * 2^23, bit pattern 0x4B400000
    return static_cast<uint32_t>(max(-127, min(127, __float_as_int(u) - 0x4B400000))) & 0xFFu;
}

// Codes clamp(rne(v / s), -127, 127) of one chunk (8 bf16 values), packed as 8
// bytes in element order; s >= kQuotientMinScale, r = RN(1/s).
__device__ __forceinline__ uint2 quant8(const uint4 &t, float s, float r)
{
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e >> 1] |= (code_byte(quotient_rn(bf16_lo(w[e]), s, r)) | (code_byte(quotient_rn(bf16_hi(w[e]), s, r)) << 8))
                     << (16 * (e & 1));
    return make_uint2(o[0], o[1]);
}

// The same codes by IEEE division (any s > 0); rows with s below
// kQuotientMinScale take it.
__device__ __forceinline__ uint2 quant8_div(const uint4 &t, float s)
{
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e >> 1] |= (code_byte(__fdiv_rn(bf16_lo(w[e]), s)) | (code_byte(__fdiv_rn(bf16_hi(w[e]), s)) << 8))
                     << (16 * (e & 1));
    return make_uint2(o[0], o[1]);
}

}  // namespace bi
