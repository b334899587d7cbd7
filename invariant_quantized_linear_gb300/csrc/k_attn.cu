// Batch-invariant split-KV attention for a verify pass: "My speculative
// decoder got slower" (split-KV attention: the cache cut into 256-token
// chunks, one partial result per chunk, a merge; one chunk writes the output
// directly) and "why speculative decoding changed my output" ("attention": a
// batch of queries must use the one-query geometry).
//
// Query m of M attends to cache positions 0 .. T0 + m; q head h reads kv head
// h / (Hq / Hkv).  Per query, head and chunk c (positions 256 c .. 256 c +
// 255 of those), in fp32 with every operation rounded once:
//   s_t = (sum over d in order of q_d k_td, from +0) * scale
//   mx  = max s_t;  p_t = e(s_t - mx)
//   l   = sum of p_t in position order;  a_d = sum of p_t v_td in position order
// then over the query's chunks in order: mx* = max mx_c, w_c = e(mx_c - mx*),
// L = sum w_c l_c, o_d = bf16((sum w_c a_cd) / L).  With one chunk w_0 = 1 and
// the chunk kernel writes o itself.  Nothing depends on M or on other queries:
// chunks are counted from the positions a query sees.
//
// e(x), x <= 0: t = x log2(e); 0 if t < -126; n = rne(t), f = t - n; 2^f by
// the degree-6 Taylor polynomial of e^(f ln 2), Horner, coefficients c_0 = 1,
// c_k = (c_(k-1) ln 2) / k; times 2^n.  ln 2 and log2(e) are their fp32
// roundings.  (A definition shared with the oracle, not CUDA's expf.)
#include "attn.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kChunk = 256;       // positions per chunk
constexpr int kAttnThreads = 256;

struct ExpCoef {
    float c[7];
};

__device__ __forceinline__ ExpCoef exp_coef()
{
    const float ln2 = __uint_as_float(0x3F317218u);
    ExpCoef e;
    e.c[0] = 1.0f;
#pragma unroll
    for (int k = 1; k < 7; ++k) e.c[k] = __fdiv_rn(__fmul_rn(e.c[k - 1], ln2), static_cast<float>(k));
    return e;
}

__device__ __forceinline__ float attn_e(float x, const ExpCoef &e)
{
    const float t = __fmul_rn(x, __uint_as_float(0x3FB8AA3Bu));
    if (t < -126.0f) return 0.0f;
    const int n = __float2int_rn(t);
    const float f = __fsub_rn(t, static_cast<float>(n));     // exact
    float p = e.c[6];
#pragma unroll
    for (int k = 5; k >= 0; --k) p = __fadd_rn(__fmul_rn(p, f), e.c[k]);
    return __fmul_rn(p, __int_as_float((n + 127) << 23));    // 2^n, n in [-126, 0]
}

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// One CTA per (chunk, head, query).  ws holds, per (query, head, chunk):
// mx, l, a[D] (fp32), for queries with more than one chunk.
template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(AttnArgs a)
{
    __shared__ float sq[D];
    __shared__ float sp[kChunk];
    __shared__ float red[kAttnThreads / 32];
    const int c = blockIdx.x, h = blockIdx.y, m = blockIdx.z;
    const int T = a.T0 + m + 1;
    const int C = (T + kChunk - 1) / kChunk;
    if (c >= C) return;
    const int tid = threadIdx.x;
    const int hk = h / (a.Hq / a.Hkv);
    const int t0 = kChunk * c, n = min(kChunk, T - t0);
    const ExpCoef ec = exp_coef();
    const uint16_t *qr = a.q + (static_cast<size_t>(m) * a.Hq + h) * D;
    for (int d = tid; d < D; d += kAttnThreads) sq[d] = bf(qr[d]);
    __syncthreads();
    // scores: thread i holds position t0 + i
    float s = -INFINITY;
    if (tid < n) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(a.k + (static_cast<size_t>(t0 + tid) * a.Hkv + hk) * D);
        float acc = 0.0f;
#pragma unroll 4
        for (int j = 0; j < D / 8; ++j) {
            const uint4 w = __ldg(kr + j);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = __fadd_rn(acc, __fmul_rn(sq[8 * j + 2 * e], __uint_as_float(u[e] << 16)));
                acc = __fadd_rn(acc, __fmul_rn(sq[8 * j + 2 * e + 1], __uint_as_float(u[e] & 0xFFFF0000u)));
            }
        }
        s = __fmul_rn(acc, a.scale);
    }
    // the chunk's maximum (exact in any order)
    float mx = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kAttnThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    if (tid < n) sp[tid] = attn_e(__fsub_rn(s, mx), ec);
    __syncthreads();
    // l (one thread) and a_d (thread d), in position order
    float l = 0.0f;
    if (tid == kAttnThreads - 1) {
#pragma unroll 8
        for (int i = 0; i < n; ++i) l = __fadd_rn(l, sp[i]);
    }
    float acc = 0.0f;
    if (tid < D) {
        const uint16_t *vr = a.v + (static_cast<size_t>(t0) * a.Hkv + hk) * D + tid;
        const size_t stride = static_cast<size_t>(a.Hkv) * D;
#pragma unroll 8
        for (int i = 0; i < n; ++i) acc = __fadd_rn(acc, __fmul_rn(sp[i], bf(__ldg(vr + i * stride))));
    }
    __syncthreads();
    if (tid == kAttnThreads - 1) red[0] = l;
    __syncthreads();
    l = red[0];
    if (C == 1) {
        if (tid < D)
            a.o[(static_cast<size_t>(m) * a.Hq + h) * D + tid] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(acc, l)));
    } else {
        float *part = a.ws + ((static_cast<size_t>(m) * a.Hq + h) * a.Cmax + c) * (D + 2);
        if (tid == 0) {
            part[0] = mx;
            part[1] = l;
        }
        if (tid < D) part[2 + tid] = acc;
    }
}

// One CTA per (head, query) with more than one chunk; thread d makes o_d.
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(AttnArgs a)
{
    const int h = blockIdx.x, m = blockIdx.y, d = threadIdx.x;
    const int T = a.T0 + m + 1;
    const int C = (T + kChunk - 1) / kChunk;
    if (C == 1) return;
    const ExpCoef ec = exp_coef();
    const float *part = a.ws + (static_cast<size_t>(m) * a.Hq + h) * a.Cmax * (D + 2);
    float mx = part[0];
    for (int c = 1; c < C; ++c) mx = fmaxf(mx, part[static_cast<size_t>(c) * (D + 2)]);
    float L = 0.0f, num = 0.0f;
    for (int c = 0; c < C; ++c) {
        const float *pc = part + static_cast<size_t>(c) * (D + 2);
        const float w = attn_e(__fsub_rn(pc[0], mx), ec);
        L = __fadd_rn(L, __fmul_rn(w, pc[1]));
        num = __fadd_rn(num, __fmul_rn(w, pc[2 + d]));
    }
    a.o[(static_cast<size_t>(m) * a.Hq + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(num, L)));
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t stream)
{
    attn_chunk_kernel<D><<<dim3(static_cast<unsigned>(a.Cmax), static_cast<unsigned>(a.Hq), static_cast<unsigned>(a.M)),
                           kAttnThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.Cmax == 1) return e;
    attn_merge_kernel<D><<<dim3(static_cast<unsigned>(a.Hq), static_cast<unsigned>(a.M)), D, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

int attn_chunks(int T0, int M) { return (T0 + M + kChunk - 1) / kChunk; }

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t stream)
{
    return a.D == 64 ? launch_d<64>(a, stream) : launch_d<128>(a, stream);
}

}  // namespace bi
