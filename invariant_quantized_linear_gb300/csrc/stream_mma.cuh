// Shared pieces of the weight-streaming kernels: the unit geometry, the
// partition of units over CTAs, and the per-stage tensor-core work of one
// consumer warp.
//
// A unit is 64 weight rows x 256 bytes of K (two 128-byte swizzled TMA boxes)
// plus the matching 256 bytes of every token row.  Consumer warps form four
// 16-row groups; each row group's 256 bytes per stage are split between KS
// warps (32-byte groups of K, 8 / KS per warp).
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"

namespace bi {
namespace stream {

constexpr int kRowGroups = 4;                       // 16-row groups per 64-row block
constexpr int kNch = 2;                             // 128-byte chunks of K per unit
constexpr int kUnitK = kNch * 128;                  // bytes of K per unit
constexpr int kWChunkBytes = kBM * 128;             // 8 KB: 64 rows x 128 B

// Consumer-warp geometry for KS warps sharing each row group's K per stage.
template <int KS>
struct Geo {
    static constexpr int kKSplit = KS;
    static constexpr int kConsumerWarps = kRowGroups * KS;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;  // plus one producer warp
    static constexpr int kGroups = kNch * 4 / KS;                // 32-byte K groups per warp per stage
};

// First unit of CTA i when `units` are cut into G near-equal contiguous ranges.
__device__ __forceinline__ long long range_start(long long i, long long units, int G)
{
    return (i * units) / G;
}

// CTA whose range holds unit u: the largest i with range_start(i) <= u.
__device__ __forceinline__ int unit_owner(long long u, long long units, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / units);
}

// Order-preserving key of a bf16 logit (no NaN): larger value, larger key;
// -0 is folded onto +0.  The low 32 bits hold ~index so that, for equal
// values, the lower index has the larger key.
__device__ __forceinline__ unsigned long long argmax_key(uint16_t b, int n)
{
    if (b == 0x8000u) b = 0;
    uint32_t k16 = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
    return (static_cast<unsigned long long>(k16) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(n));
}

// Which 32-byte groups of K run on the int8 MMA (no conversion; a separate,
// slower pipe) and which on the f16 MMA (fast, but each int8 operand is first
// converted).  Measured on the 36-layer verify pass: with one token tile every
// group on the int8 MMA is fastest (2.31 ms against 2.36 with half and 2.44
// with a quarter: the conversions cost more than the int8 pipe's rate); with
// two token tiles, where the int8 MMA does twice the work per group, the share
// made no difference, and a quarter is kept.
template <int MT>
__device__ __forceinline__ constexpr bool imma_group(int t)
{
    return MT == 1 ? true : (t & 3) == 0;
}

// Lane constants of a consumer warp for ldmatrix and the MMA fragments.
struct Lane {
    int g, tq;        // MMA fragment row group / thread in group
    int rg, kq;       // 16-row group inside the 64-row block, share of K
    uint32_t a_row;   // weight row this lane addresses for ldmatrix
    int a_hi;         // 16-byte chunk X or Y of a 32-byte group (weights)
    uint32_t b_tok;   // token row this lane addresses for ldmatrix
    int b_hi;         // chunk X or Y (tokens)
};

template <int MT, int KS>
__device__ __forceinline__ Lane lane_setup(int warp, int lane)
{
    Lane L;
    L.g = lane >> 2;
    L.tq = lane & 3;
    const int mat = lane >> 3, r8 = lane & 7;
    L.rg = warp % kRowGroups;
    L.kq = warp / kRowGroups;
    L.a_row = L.rg * 16 + ((mat & 1) ? 8 : 0) + r8;
    L.a_hi = (mat & 2) ? 1 : 0;
    L.b_tok = (MT == 2 && (lane >> 4)) ? 8 + r8 : r8;
    L.b_hi = (lane >> 3) & 1;
    return L;
}

// One stage of one consumer warp: the warp's 16 rows x (256 / KS) bytes of K
// against every token row, added exactly into the int32 accumulators
//   v[t][i] = (row g (+8 for i >= 2), token 8t + 2tq + (i & 1)).
// All int8 fragments are loaded first (the loads overlap).  Int8-MMA groups
// accumulate straight into v; f16-MMA groups convert the codes exactly to
// f16 and accumulate in fp32, whose partials (at most 64 bytes of K: integers
// below 2^20) are moved into v at the end.  The logical k order inside an
// MMA is a fixed permutation of the bytes, the same for both operands, so the
// integer dot product is unchanged.
template <int MT, int KS>
__device__ __forceinline__ void consume_stage(uint32_t wbase, uint32_t abase, uint32_t a_chunk_bytes,
                                              const Lane &L, int32_t (&v)[MT][4])
{
    constexpr int kGroups = Geo<KS>::kGroups;
    uint32_t fa[kGroups][4];
    uint32_t fb[kGroups][2 * MT];
#pragma unroll
    for (int tt = 0; tt < kGroups; ++tt) {
        const int t = L.kq * kGroups + tt;
        const int ch = t >> 2, ks = t & 3;
        ldmatrix_x4(wbase + ch * kWChunkBytes + swz128(L.a_row, 2 * ks + L.a_hi), fa[tt][0], fa[tt][1], fa[tt][2],
                    fa[tt][3]);
        if constexpr (MT == 1)
            ldmatrix_x2(abase + ch * a_chunk_bytes + swz128(L.b_tok, 2 * ks + L.b_hi), fb[tt][0], fb[tt][1]);
        else
            ldmatrix_x4(abase + ch * a_chunk_bytes + swz128(L.b_tok, 2 * ks + L.b_hi), fb[tt][0], fb[tt][1],
                        fb[tt][2], fb[tt][3]);
    }
    float facc[2][MT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < MT; ++m) facc[h][m][0] = facc[h][m][1] = facc[h][m][2] = facc[h][m][3] = 0.0f;
#pragma unroll
    for (int t = 0; t < kGroups; ++t) {
        if (imma_group<MT>(t)) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                mma_s8_16832(v[m], fa[t][0], fa[t][1], fa[t][2], fa[t][3], fb[t][2 * m], fb[t][2 * m + 1]);
            continue;
        }
#pragma unroll
        for (int xy = 0; xy < 2; ++xy) {  // chunk X, then chunk Y
            uint32_t a0, a1, a2, a3;
            i8x4_to_f16x2x2(fa[t][2 * xy], a0, a2);      // row g
            i8x4_to_f16x2x2(fa[t][2 * xy + 1], a1, a3);  // row g + 8
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint32_t b0, b1;
                i8x4_to_f16x2x2(fb[t][2 * m + xy], b0, b1);
                mma_f16_16816(facc[xy][m], a0, a1, a2, a3, b0, b1);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[m][i] += f2i_exact(facc[0][m][i]) + f2i_exact(facc[1][m][i]);
}

}  // namespace stream
}  // namespace bi
