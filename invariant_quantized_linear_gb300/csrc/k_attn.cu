// Batch-invariant split-KV attention for a verify pass: "My speculative
// decoder got slower" (split-KV attention: the cache cut into 256-token
// chunks, one partial result per chunk, a merge; one chunk writes the output
// directly) and "why speculative decoding changed my output" ("attention": a
// batch of queries must use the one-query geometry).
//
// Query m of M attends to cache positions 0 .. T0 + m; q head h reads kv head
// h / (Hq / Hkv).  Per query, head and chunk c (positions 256 c .. 256 c +
// 255 of those), in fp32, every operation rounded once (a multiply-accumulate
// step is one fused multiply-add):
//   s_t = (sum over d in order of q_d k_td, from +0) * scale
//   mx  = max s_t;  p_t = e(s_t - mx)
//   l   = sum of p_t in position order;  a_d = sum of p_t v_td in position order
// then over the query's chunks in order: mx* = max mx_c, w_c = e(mx_c - mx*),
// L = sum w_c l_c, o_d = bf16((sum w_c a_cd) / L).  With one chunk w_0 = 1 and
// the chunk kernel writes o itself.  Nothing depends on M or on other queries:
// chunks are counted from the positions a query sees.
//
// e(x), x <= 0: t = x log2(e); 0 if t < -126; n = rne(t), f = t - n; 2^f by
// the degree-6 Taylor polynomial of e^(f ln 2), Horner (one fused multiply-add
// a step), coefficients c_0 = 1, c_k = (c_(k-1) ln 2) / k; times 2^n.  ln 2
// and log2(e) are their fp32 roundings.  (Not CUDA's expf.)
//
// Every step acc <- acc + x * y of the sums is one fused multiply-add.
#include "attn.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kChunk = 256;       // positions per chunk
constexpr int kRows = 32;         // (query, q head) rows per chunk CTA
constexpr int kScoreWarps = 8;    // warps of the score and value tiles
constexpr int kAttnThreads = 32 * (kScoreWarps + 1);   // + one warp for the weight sums l
constexpr int kMergeBatch = 16;   // chunk values a merge thread has in flight at once

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
    for (int k = 5; k >= 0; --k) p = __fmaf_rn(p, f, e.c[k]);
    return __fmul_rn(p, __int_as_float((n + 127) << 23));    // 2^n, n in [-126, 0]
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Two fp32 lanes in one 64-bit register (low half first) and the packed
// fused multiply-add: each lane is one correctly rounded fma, as a scalar fma.
__device__ __forceinline__ unsigned long long pk(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void upk(unsigned long long x, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Two 64-bit words (four fp32) from shared memory.
__device__ __forceinline__ void lds2x64(const void *p, unsigned long long &a, unsigned long long &b)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(s));
}

// Shared-memory plan of the chunk kernel for head size D.  K rows are padded
// by 16 bytes so that 32 lanes reading 16 bytes of 32 different rows hit
// distinct banks; q is kept as fp32 [d][row] so that a row pair is one 64-bit
// word; the weights P are [position][row], padded by 4 floats per position.
// Broadcast reads (q in the scores, P in the values) cost the SM about 8
// bytes a cycle, so the tiles are sized to keep them under the fma time.
template <int D>
struct ChunkSmem {
    static constexpr int kRow = 2 * D + 16;           // bytes per K row
    static constexpr int kPRow = kRows + 4;           // floats per P row
    static constexpr int kK = 0;
    static constexpr int kV = kK + kChunk * kRow;
    static constexpr int kQ = kV + kChunk * 2 * D;
    static constexpr int kP = kQ + kRows * D * 4;
    static constexpr int kRed = kP + kChunk * kPRow * 4;
    static constexpr int kL = kRed + 2 * kRows * 4;
    static constexpr int kBytes = kL + kRows * 4;
};

// Positions of chunk c that query m sees (0 .. 256; 0 when the chunk is past it).
__device__ __forceinline__ int chunk_positions(int T0, int m, int c)
{
    return max(0, min(kChunk, T0 + m + 1 - kChunk * c));
}

// One CTA per (chunk c, kv head hk, block of 32 rows).  The rows of a kv head
// are its (query m, q head g) pairs, r = m * G + g, G = Hq / Hkv.  The chunk's
// K and V rows are staged once in shared memory and shared by all the rows.
// Sums run as packed pairs of independent fmas (fma.rn.f32x2), each lane the
// same correctly rounded step as a scalar fma.
//   scores: warp w < 8 holds rows 8 (w >> 1) .. +7 (as 4 row pairs) at
//           positions 128 (w & 1) + lane + 32 j (j < 4); sum over d in order.
//   values: warp w < 8 holds rows 4 w .. +3 at d = (D / 32) lane .. (pairs
//           of adjacent d); sum over positions in order.
//   l:      warp 8 sums the weights of row lane in position order meanwhile.
// A row whose query sees one chunk writes o; otherwise (mx, l, a) go to ws.
template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_chunk_kernel(AttnArgs a)
{
    using L = ChunkSmem<D>;
    constexpr int DP = D / 32;                         // d-values per lane in the value sums (2 or 4)
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *Ks = smem + L::kK;
    unsigned char *Vs = smem + L::kV;
    float *Qs = reinterpret_cast<float *>(smem + L::kQ);
    float *Ps = reinterpret_cast<float *>(smem + L::kP);
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    float *ls = reinterpret_cast<float *>(smem + L::kL);

    const int c = blockIdx.x, hk = blockIdx.y, rb = blockIdx.z;
    const int G = a.Hq / a.Hkv;
    const int rows = a.M * G;                          // rows of this kv head
    const int r0 = kRows * rb;
    const int r_last = min(rows, r0 + kRows) - 1;
    const int n_max = chunk_positions(a.T0, r_last / G, c);
    if (n_max == 0) return;                            // no row of the block reaches this chunk
    pdl_launch_dependents();                           // the merge may launch; it waits for this grid to end
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = kChunk * c;
    const size_t kv_row = static_cast<size_t>(a.Hkv) * D;
    constexpr int kSeg = D / 8;                        // 16-byte pieces per row

    // q rows (loads issued first), then K; V is staged once K has landed, so
    // that K arrives at full bandwidth and V overlaps the scores
    constexpr int kQPer = (kRows * kSeg + kAttnThreads - 1) / kAttnThreads;
    uint4 qv[kQPer];                                   // piece i: row i % 32, 16-byte segment i / 32
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
        const int i = tid + k * kAttnThreads, rl = i % kRows, r = r0 + rl;
        qv[k] = make_uint4(0u, 0u, 0u, 0u);
        if (i < kRows * kSeg && r < rows) {
            const int m = r / G, h = hk * G + (r - m * G);
            qv[k] = __ldg(reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(m) * a.Hq + h) * D) + i / kRows);
        }
    }
    for (int i = tid; i < n_max * kSeg; i += kAttnThreads) {
        const int t = i / kSeg, sg = i - t * kSeg;
        cp_async16(Ks + t * L::kRow + 16 * sg, a.k + (t0 + t) * kv_row + hk * D + 8 * sg);
    }
    cp_async_commit();
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
        const int i = tid + k * kAttnThreads, rl = i % kRows, sg = i / kRows;
        if (i < kRows * kSeg) {
            float *dst = Qs + 8 * sg * kRows + rl;     // q as [d][row]: a warp's 32 rows hit 32 banks
            const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dst[(2 * e) * kRows] = __uint_as_float(w[e] << 16);
                dst[(2 * e + 1) * kRows] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
    }
    const ExpCoef ec = exp_coef();
    cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < n_max * kSeg; i += kAttnThreads) {
        const int t = i / kSeg, sg = i - t * kSeg;
        cp_async16(Vs + t * 2 * D + 16 * sg, a.v + (t0 + t) * kv_row + hk * D + 8 * sg);
    }
    cp_async_commit();

    // ---- scores of 8 rows x 4 positions per thread
    const bool scorer = warp < kScoreWarps;
    const int rg = (warp >> 1) & 3, pg = warp & 1;     // a row group's two warps sit on two partitions
    const int rs0 = r0 + 8 * rg;                       // first row of this warp's score tile
    float s[8][4];
    if (scorer && rs0 < rows) {
        unsigned long long sc[4][4];                   // rows 2 ip, 2 ip + 1 at position j
#pragma unroll
        for (int ip = 0; ip < 4; ++ip)
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[ip][j] = 0ull;
        const unsigned char *kb = Ks + (128 * pg + lane) * L::kRow;
        const float *qb = Qs + 8 * rg;
#pragma unroll 2
        for (int d0 = 0; d0 < D; d0 += 8) {
            uint4 kv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) kv[j] = *reinterpret_cast<const uint4 *>(kb + 32 * j * L::kRow + 2 * d0);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                unsigned long long q2[4];
                lds2x64(qb + (d0 + e) * kRows, q2[0], q2[1]);
                lds2x64(qb + (d0 + e) * kRows + 4, q2[2], q2[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w = (e >> 1) == 0 ? kv[j].x : (e >> 1) == 1 ? kv[j].y : (e >> 1) == 2 ? kv[j].z : kv[j].w;
                    const float kf = __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
                    const unsigned long long kd = pk(kf, kf);
#pragma unroll
                    for (int ip = 0; ip < 4; ++ip) sc[ip][j] = fma2(q2[ip], kd, sc[ip][j]);
                }
            }
        }
#pragma unroll
        for (int ip = 0; ip < 4; ++ip)
#pragma unroll
            for (int j = 0; j < 4; ++j) upk(sc[ip][j], s[2 * ip][j], s[2 * ip + 1][j]);
    }
    // scale, mask to the positions each row's query sees, row maxima
    float mxr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = rs0 + i;
        const int n = (scorer && r < rows) ? chunk_positions(a.T0, r / G, c) : 0;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = 128 * pg + lane + 32 * j;
            s[i][j] = t < n ? __fmul_rn(s[i][j], a.scale) : -INFINITY;
            mx = fmaxf(mx, s[i][j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mxr[i] = mx;
    }
    if (scorer && lane < 8) {
        float mv = mxr[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) mv = lane == i ? mxr[i] : mv;
        red[pg * kRows + 8 * rg + lane] = mv;
    }
    __syncthreads();                                   // maxima of both position halves in red
    // weights p = e(s - mx) into P[position][row]; masked positions weigh 0
    if (scorer) {
#pragma unroll
        for (int i = 0; i < 8; ++i) mxr[i] = fmaxf(red[8 * rg + i], red[kRows + 8 * rg + i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = 128 * pg + lane + 32 * j;
            float p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) p[i] = s[i][j] == -INFINITY ? 0.0f : attn_e(__fsub_rn(s[i][j], mxr[i]), ec);
            float4 *dst = reinterpret_cast<float4 *>(Ps + t * L::kPRow + 8 * rg);
            dst[0] = make_float4(p[0], p[1], p[2], p[3]);
            dst[1] = make_float4(p[4], p[5], p[6], p[7]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();                                   // P complete, V staged

    // ---- weighted values (warps 0..7) and weight sums (warp 8)
    const int rv0 = r0 + 4 * warp;                     // rows of this warp's value tile
    const int dl = DP * lane;                          // its first d
    int nr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) nr[i] = (warp < kScoreWarps && rv0 + i < rows) ? chunk_positions(a.T0, (rv0 + i) / G, c) : 0;
    unsigned long long acc2[4][DP / 2];                // row i at d = dl + 2 e, dl + 2 e + 1
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < DP / 2; ++e) acc2[i][e] = 0ull;
    if (warp == kScoreWarps) {
        if (r0 + lane < rows) {
            const int n = chunk_positions(a.T0, (r0 + lane) / G, c);
            float l = 0.0f;
#pragma unroll 8
            for (int t = 0; t < n; ++t) l = __fadd_rn(l, Ps[t * L::kPRow + lane]);
            ls[lane] = l;
        }
    } else {
        const int n_lo = nr[0];
        const int n_hi = max(max(nr[0], nr[1]), max(nr[2], nr[3]));
        const float *pb = Ps + 4 * warp;
        const unsigned char *vb = Vs + 2 * dl;
        auto vpairs = [&](int t, unsigned long long *v2) {
            if constexpr (DP == 4) {
                const uint2 u = *reinterpret_cast<const uint2 *>(vb + t * 2 * D);
                v2[0] = pk(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u));
                v2[1] = pk(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
            } else {
                const uint32_t u = *reinterpret_cast<const uint32_t *>(vb + t * 2 * D);
                v2[0] = pk(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
            }
        };
#pragma unroll 4
        for (int t = 0; t < n_lo; ++t) {
            const float4 pv = *reinterpret_cast<const float4 *>(pb + t * L::kPRow);
            const float p[4] = {pv.x, pv.y, pv.z, pv.w};
            unsigned long long v2[DP / 2];
            vpairs(t, v2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const unsigned long long pd = pk(p[i], p[i]);
#pragma unroll
                for (int e = 0; e < DP / 2; ++e) acc2[i][e] = fma2(pd, v2[e], acc2[i][e]);
            }
        }
#pragma unroll 1
        for (int t = n_lo; t < n_hi; ++t) {           // rows of later queries see a few more positions
            unsigned long long v2[DP / 2];
            vpairs(t, v2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (t < nr[i]) {
                    const float p = pb[t * L::kPRow + i];
                    const unsigned long long pd = pk(p, p);
#pragma unroll
                    for (int e = 0; e < DP / 2; ++e) acc2[i][e] = fma2(pd, v2[e], acc2[i][e]);
                }
            }
        }
    }
    __syncthreads();                                   // l of every row is in ls
    if (warp == kScoreWarps) return;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = rv0 + i;
        if (nr[i] == 0) continue;                      // past the rows or past this query's positions
        const int m = r / G, h = hk * G + (r - m * G);
        const float l = ls[4 * warp + i];
        float av[DP];
#pragma unroll
        for (int e = 0; e < DP / 2; ++e) upk(acc2[i][e], av[2 * e], av[2 * e + 1]);
        if (a.T0 + m + 1 <= kChunk) {                  // the query's only chunk: o = a / l
            uint32_t ob[DP / 2];
#pragma unroll
            for (int e = 0; e < DP / 2; ++e)
                ob[e] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(av[2 * e], l))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(av[2 * e + 1], l))))
                         << 16);
            uint16_t *dst = a.o + (static_cast<size_t>(m) * a.Hq + h) * D + dl;
            if constexpr (DP == 4)
                *reinterpret_cast<uint2 *>(dst) = make_uint2(ob[0], ob[1]);
            else
                *reinterpret_cast<uint32_t *>(dst) = ob[0];
        } else {
            float *part = a.ws + ((static_cast<size_t>(m) * a.Hq + h) * a.Cmax + c) * (D + 4);
            if (lane == 0) {
                const int rl = 4 * warp + i;
                part[0] = fmaxf(red[rl], red[kRows + rl]);
                part[1] = l;
            }
            if constexpr (DP == 4)
                *reinterpret_cast<float4 *>(part + 4 + dl) = make_float4(av[0], av[1], av[2], av[3]);
            else
                *reinterpret_cast<float2 *>(part + 4 + dl) = make_float2(av[0], av[1]);
        }
    }
}

// One CTA per (q head, query) whose query sees more than one chunk; thread d
// makes o_d from the chunk results in chunk order.  The chunk weights w_c and
// sums l_c are staged in shared memory first (their loads all in flight at
// once), so the in-order sums only wait on the a_cd loads, which are
// independent of one another.
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(AttnArgs a)
{
    extern __shared__ float wl[];                      // w [Cmax], l [Cmax]
    __shared__ float red[D / 32];
    const int h = blockIdx.x, m = blockIdx.y, d = threadIdx.x;
    const int T = a.T0 + m + 1;
    const int C = (T + kChunk - 1) / kChunk;
    if (C == 1) return;
    pdl_wait();                                        // the chunk grid has ended and its results are visible
    const float *part = a.ws + (static_cast<size_t>(m) * a.Hq + h) * a.Cmax * (D + 4);
    float a0[kMergeBatch];                             // the first chunks' values, loaded with the maxima
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) a0[k] = k < C ? part[static_cast<size_t>(k) * (D + 4) + 4 + d] : 0.0f;
    float mx = -INFINITY;
    for (int c = d; c < C; c += D) {
        const float mc = part[static_cast<size_t>(c) * (D + 4)];
        wl[c] = mc;
        wl[a.Cmax + c] = part[static_cast<size_t>(c) * (D + 4) + 1];
        mx = fmaxf(mx, mc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((d & 31) == 0) red[d >> 5] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w) mx = fmaxf(mx, red[w]);
    const ExpCoef ec = exp_coef();
    for (int c = d; c < C; c += D) wl[c] = attn_e(__fsub_rn(wl[c], mx), ec);
    __syncthreads();
    float L = 0.0f, num = 0.0f;
    const float *pa = part + 4 + d;
    for (int c0 = 0; c0 < C; c0 += kMergeBatch) {
        float av[kMergeBatch];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k)
            av[k] = c0 == 0 ? a0[k] : c0 + k < C ? pa[static_cast<size_t>(c0 + k) * (D + 4)] : 0.0f;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            if (c0 + k < C) {
                const float w = wl[c0 + k];
                L = __fmaf_rn(w, wl[a.Cmax + c0 + k], L);
                num = __fmaf_rn(w, av[k], num);
            }
        }
    }
    a.o[(static_cast<size_t>(m) * a.Hq + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(num, L)));
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t stream)
{
    constexpr int bytes = ChunkSmem<D>::kBytes;
    static bool configured = false;                    // one attribute call per process and head size
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int G = a.Hq / a.Hkv;
    const int blocks = (a.M * G + kRows - 1) / kRows;
    attn_chunk_kernel<D><<<dim3(static_cast<unsigned>(a.Cmax), static_cast<unsigned>(a.Hkv),
                                static_cast<unsigned>(blocks)),
                           kAttnThreads, bytes, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.Cmax == 1) return e;
    // the merge launches while the chunk grid runs (programmatic dependent
    // launch) and waits for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.Hq), static_cast<unsigned>(a.M));
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = 2 * a.Cmax * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel<D>, a);
}

}  // namespace

int attn_chunks(int T0, int M) { return (T0 + M + kChunk - 1) / kChunk; }

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t stream)
{
    return a.D == 64 ? launch_d<64>(a, stream) : launch_d<128>(a, stream);
}

}  // namespace bi
