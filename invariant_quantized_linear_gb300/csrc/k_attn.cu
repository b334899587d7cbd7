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

// The chunk kernel for a kv head with few rows (M * G <= R, R = 4 or 8: one
// or two verify queries of a Qwen3-8B-shaped layer).  The 32-row tile above
// would leave most of its lanes idle.  One CTA per (chunk, kv head), eight
// warps:
//   score warps 0-3: thread t holds positions t and t + 128 for all R rows
//           (each q row pair, broadcast from shared memory, serves both
//           positions).  Each warp stages the K rows of its own 64 positions
//           and starts as soon as they have landed.
//   staging warps 4-7: issue the V copies once the score warps' K has landed
//           (so that V does not slow K down in the memory system; the wait
//           is bounded and only orders the requests).
//   values, all warps: warp w holds d pairs 32 (w % n) + lane (n = D / 64)
//           of R n / 8 rows (at least one), one packed chain per row over
//           positions in order (the lanes are d, d + 1) and the row's weight
//           sum l beside it.  The weights are stored row by row, so that one
//           16-byte broadcast brings four positions of a row.
// Every sum is the same sequence of correctly rounded operations as in the
// 32-row kernel.
template <int D, int R>
struct SmallSmem {
    static constexpr int kRow = 2 * D + 16;            // bytes per K row (padded: conflict-free row reads)
    static constexpr int kK = 0;                       // K [256][kRow]
    static constexpr int kV = kK + kChunk * kRow;      // V [256][D] bf16
    static constexpr int kQ = kV + kChunk * 2 * D;     // q fp32 [D][R]
    static constexpr int kP = kQ + D * R * 4;          // weights fp32 [R][256]
    static constexpr int kRed = kP + kChunk * R * 4;   // score-warp maxima fp32 [R][4]
    static constexpr int kFlag = kRed + R * 4 * 4;     // score warps whose K has landed
    static constexpr int kBytes = kFlag + 16;
};

constexpr int kSmallThreads = 256;
constexpr int kScoreThreads = 128;                     // warps 0-3

__device__ __forceinline__ void bar_sync_scorers() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

constexpr int kKWaitLimit = 4096;                      // polls of the K-landed count before V is issued anyway

template <int D, int R>
__global__ void __launch_bounds__(kSmallThreads, 1) attn_chunk_small_kernel(AttnArgs a)
{
    using L = SmallSmem<D, R>;
    constexpr int kW = D / 8;                          // 16-byte pieces of a K, V or q row
    constexpr int kDG = D / 64;                        // 32-lane groups of d pairs (1 or 2)
    constexpr int kRPW = (R * kDG >= 8) ? R * kDG / 8 : 1;   // rows per value warp (1 or 2)
    constexpr int kQPer = (R * kW + kScoreThreads - 1) / kScoreThreads;
    static_assert((R == 4 || R == 8) && kSmallThreads == 256, "shape");
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *Ks = smem + L::kK;
    unsigned char *Vs = smem + L::kV;
    float *Qs = reinterpret_cast<float *>(smem + L::kQ);
    float *Ps = reinterpret_cast<float *>(smem + L::kP);
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    int *k_landed = reinterpret_cast<int *>(smem + L::kFlag);

    const int c = blockIdx.x, hk = blockIdx.y;
    const int G = a.Hq / a.Hkv;
    const int rows = a.M * G;                          // rows of this kv head, <= R
    const int n_max = chunk_positions(a.T0, a.M - 1, c);
    if (n_max == 0) return;
    pdl_launch_dependents();                           // the merge may launch; it waits for this grid to end
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = kChunk * c;
    const size_t kv_row = static_cast<size_t>(a.Hkv) * D;
    const bool scorer = tid < kScoreThreads;
    if (tid == 0) *k_landed = 0;
    __syncthreads();
    // positions of chunk c that row r's query sees (0 past the rows)
    auto row_n = [&](int r) { return r < rows ? chunk_positions(a.T0, r / G, c) : 0; };

    float s[2][R];                                     // scores of positions tid, tid + 128 (score warps)
    if (scorer) {
        // q pieces (row i % R, 16-byte piece i / R), then the K rows of this
        // warp's positions 32 w .. + 31 and 128 + 32 w .. + 31
        uint4 qv[kQPer];
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int i = tid + k * kScoreThreads, qr = i % R;
            qv[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < R * kW && qr < rows) {
                const int m = qr / G, h = hk * G + (qr - m * G);
                qv[k] = __ldg(reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(m) * a.Hq + h) * D) + i / R);
            }
        }
        for (int i = lane; i < 64 * kW; i += 32) {
            const int j = i / kW, sg = i - j * kW;
            const int t = (j < 32) ? 32 * warp + j : 128 + 32 * warp + (j - 32);
            if (t < n_max) cp_async16(Ks + t * L::kRow + 16 * sg, a.k + (t0 + t) * kv_row + hk * D + 8 * sg);
        }
        cp_async_commit();
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int i = tid + k * kScoreThreads, qr = i % R, qs = i / R;
            if (i < R * kW) {
                float *dst = Qs + 8 * qs * R + qr;     // q as [d][row]: a row pair is one 64-bit word
                const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dst[(2 * e) * R] = __uint_as_float(w[e] << 16);
                    dst[(2 * e + 1) * R] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
            }
        }
        bar_sync_scorers();                            // q staged
        cp_async_wait<0>();                            // this lane's K copies have landed
        __syncwarp();                                  // and the other lanes' of the warp
        if (lane == 0) atomicAdd(k_landed, 1);

        // scores: R / 2 packed chains over d for each of the two positions
        unsigned long long sc[2][R / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ip = 0; ip < R / 2; ++ip) sc[h][ip] = 0ull;
        const unsigned char *kb0 = Ks + tid * L::kRow;
        const unsigned char *kb1 = Ks + (tid + 128) * L::kRow;
        // fully unrolled with 4 rows of 128 (measured faster); otherwise by
        // two pieces (a full unroll runs out of registers)
#pragma unroll (R == 4 && D == 128 ? kW : 2)
        for (int j = 0; j < kW; ++j) {
            const uint4 k0 = *reinterpret_cast<const uint4 *>(kb0 + 16 * j);
            const uint4 k1 = *reinterpret_cast<const uint4 *>(kb1 + 16 * j);
            const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
            const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = 8 * j + e;
                unsigned long long q2[R / 2];
#pragma unroll
                for (int ip = 0; ip < R / 2; ip += 2) lds2x64(Qs + d * R + 2 * ip, q2[ip], q2[ip + 1]);
                const float kf0 = __uint_as_float((e & 1) ? (w0[e >> 1] & 0xFFFF0000u) : (w0[e >> 1] << 16));
                const float kf1 = __uint_as_float((e & 1) ? (w1[e >> 1] & 0xFFFF0000u) : (w1[e >> 1] << 16));
                const unsigned long long kd0 = pk(kf0, kf0), kd1 = pk(kf1, kf1);
#pragma unroll
                for (int ip = 0; ip < R / 2; ++ip) {
                    sc[0][ip] = fma2(q2[ip], kd0, sc[0][ip]);
                    sc[1][ip] = fma2(q2[ip], kd1, sc[1][ip]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ip = 0; ip < R / 2; ++ip) upk(sc[h][ip], s[h][2 * ip], s[h][2 * ip + 1]);
        // scale, mask to the positions each row's query sees, maxima over the warp's 64 positions
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = row_n(r);
            s[0][r] = tid < n ? __fmul_rn(s[0][r], a.scale) : -INFINITY;
            s[1][r] = tid + 128 < n ? __fmul_rn(s[1][r], a.scale) : -INFINITY;
            float mx = fmaxf(s[0][r], s[1][r]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[r * 4 + warp] = mx;
        }
    } else {
        if (lane == 0) {
            for (int it = 0; it < kKWaitLimit; ++it) {
                if (*static_cast<volatile int *>(k_landed) >= kScoreThreads / 32) break;
                __nanosleep(64);
            }
        }
        __syncwarp();
        for (int i = tid - kScoreThreads; i < n_max * kW; i += kSmallThreads - kScoreThreads) {
            const int t = i / kW, sg = i - t * kW;
            cp_async16(Vs + t * 2 * D + 16 * sg, a.v + (t0 + t) * kv_row + hk * D + 8 * sg);
        }
        cp_async_commit();
    }
    const ExpCoef ec = exp_coef();
    __syncthreads();                                   // maxima of every row in red
    if (scorer) {
        // weights p = e(s - mx) into P[row][position]; masked positions weigh 0
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 m4 = *reinterpret_cast<const float4 *>(red + r * 4);
            const float mx = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
#pragma unroll
            for (int h = 0; h < 2; ++h)
                Ps[r * kChunk + tid + 128 * h] = s[h][r] == -INFINITY ? 0.0f : attn_e(__fsub_rn(s[h][r], mx), ec);
        }
    } else {
        cp_async_wait<0>();                            // this thread's V copies have landed
    }
    __syncthreads();                                   // weights complete, V staged

    // ---- weighted values and weight sums, positions in order
    const int g = warp % kDG, rb = warp / kDG;         // d-pair group, row block
    const int dp = 32 * g + lane;
    const int r0 = kRPW * rb;                          // first row of this warp
    if (r0 >= R) return;                               // D = 64 with 4 rows: half the warps have none
    int nr[kRPW];
    int n_lo = kChunk, n_hi = 0;
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        nr[i] = row_n(r0 + i);
        if (nr[i] > 0) n_lo = min(n_lo, nr[i]);
        n_hi = max(n_hi, nr[i]);
    }
    if (n_hi == 0) n_lo = 0;
    unsigned long long acc[kRPW];                      // lanes d = 2 dp, 2 dp + 1 of row r0 + i
    float lsum[kRPW];
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        acc[i] = 0ull;
        lsum[i] = 0.0f;
    }
    const unsigned char *vb = Vs + 4 * dp;
    const float *pb = Ps + r0 * kChunk;
    // blocks of 4 positions: each row's 4 weights in one broadcast, the next
    // block's operands in flight; rows with no positions have zero weights
    // and are not written
    uint32_t vq[4];
    float4 pq[kRPW];
    auto load4 = [&](int t, uint32_t (&vv)[4], float4 (&pp)[kRPW]) {
        const int tt = min(t, kChunk - 4);             // past the chunk at the end: loaded, unused
#pragma unroll
        for (int k = 0; k < 4; ++k) vv[k] = *reinterpret_cast<const uint32_t *>(vb + (tt + k) * 2 * D);
#pragma unroll
        for (int i = 0; i < kRPW; ++i) pp[i] = *reinterpret_cast<const float4 *>(pb + i * kChunk + tt);
    };
    const int n_main = n_lo & ~3;
    if (n_main > 0) load4(0, vq, pq);
    for (int t = 0; t < n_main; t += 4) {
        uint32_t vn[4];
        float4 pn[kRPW];
        load4(t + 4, vn, pn);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const unsigned long long v2 = pk(__uint_as_float(vq[k] << 16), __uint_as_float(vq[k] & 0xFFFF0000u));
#pragma unroll
            for (int i = 0; i < kRPW; ++i) {
                const float p = k == 0 ? pq[i].x : k == 1 ? pq[i].y : k == 2 ? pq[i].z : pq[i].w;
                acc[i] = fma2(pk(p, p), v2, acc[i]);
                lsum[i] = __fadd_rn(lsum[i], p);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) vq[k] = vn[k];
#pragma unroll
        for (int i = 0; i < kRPW; ++i) pq[i] = pn[i];
    }
    // the last positions of the shortest row, then those only later queries see
#pragma unroll 1
    for (int t = n_main; t < n_hi; ++t) {
        const uint32_t vv = *reinterpret_cast<const uint32_t *>(vb + t * 2 * D);
        const unsigned long long v2 = pk(__uint_as_float(vv << 16), __uint_as_float(vv & 0xFFFF0000u));
#pragma unroll
        for (int i = 0; i < kRPW; ++i) {
            if (t < nr[i]) {
                const float p = pb[i * kChunk + t];
                acc[i] = fma2(pk(p, p), v2, acc[i]);
                lsum[i] = __fadd_rn(lsum[i], p);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        const int r = r0 + i;
        if (nr[i] == 0) continue;                      // past the rows or past this query's positions
        const int m = r / G, h = hk * G + (r - m * G);
        float a0, a1;
        upk(acc[i], a0, a1);
        const float l = lsum[i];
        if (a.T0 + m + 1 <= kChunk) {                  // the query's only chunk: o = a / l
            const uint32_t ob = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(a0, l))) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(a1, l))))
                                 << 16);
            *reinterpret_cast<uint32_t *>(a.o + (static_cast<size_t>(m) * a.Hq + h) * D + 2 * dp) = ob;
        } else {
            float *part = a.ws + ((static_cast<size_t>(m) * a.Hq + h) * a.Cmax + c) * (D + 4);
            if (dp == 0) {
                const float4 m4 = *reinterpret_cast<const float4 *>(red + r * 4);
                part[0] = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
                part[1] = l;
            }
            *reinterpret_cast<float2 *>(part + 4 + 2 * dp) = make_float2(a0, a1);
        }
    }
}

// ---- One or two queries with heads of 128: a cluster of four CTAs per (chunk,
// kv head).  CTA k of the cluster stages a quarter of the chunk's K (positions
// 64 k .. 64 k + 63) and a quarter of its V (d = 32 k .. 32 k + 31 of every
// position), so each SM waits for a quarter of the bytes.  Row maxima and the
// weights are exchanged through distributed shared memory:
//   scores: thread (p, g) of warps 0-3 holds position 64 k + p for row pair g
//           (two pairs with 8 rows), a packed chain over d in order;
//   maxima: each CTA's row maxima go to every CTA of the cluster; barrier;
//   weights: p = e(s - mx) of the CTA's 64 positions go to every CTA; barrier;
//   values: thread (r, j) sums p_t v_td for d = 32 k + 2 j, + 1 of row r over
//           all positions in order; warp 4 sums each row's weights l.
// Every CTA of a cluster passes the same three cluster barriers: the only
// early return comes before the first and is the same for the whole cluster
// (it depends on the chunk alone), and the last remote store precedes the last
// barrier.  The sums are the same correctly rounded steps as in the kernels
// above.
constexpr int kClusterCtas = 4;
constexpr int kClusterThreads = 160;

template <int R>
struct ClusterSmem {
    static constexpr int kD = 128;
    static constexpr int kRow = 2 * kD + 16;           // K row, padded
    static constexpr int kK = 0;                       // K [64][kRow]: this CTA's positions
    static constexpr int kV = kK + 64 * kRow;          // V [256][32] bf16: this CTA's d slice of every position
    static constexpr int kQ = kV + kChunk * 64;        // q fp32 [128][R]
    static constexpr int kP = kQ + kD * R * 4;         // weights fp32 [R][256] (every CTA's positions)
    static constexpr int kRed = kP + R * kChunk * 4;   // row maxima fp32 [R][4 CTAs]
    static constexpr int kWm = kRed + R * kClusterCtas * 4;   // warp maxima fp32 [4 warps][R]
    static constexpr int kL = kWm + 4 * R * 4;         // weight sums fp32 [R]
    static constexpr int kBytes = kL + R * 4;
};

template <int R>
__global__ void __launch_bounds__(kClusterThreads) attn_chunk_cluster_kernel(AttnArgs a)
{
    constexpr int D = 128;
    using L = ClusterSmem<R>;
    constexpr int kW = D / 8;                          // 16-byte pieces of a q or K row
    constexpr int kPairs = R / 2 / 2;                  // row pairs per score thread (1 or 2)
    static_assert(R == 4 || R == 8, "shape");
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *Ks = smem + L::kK;
    unsigned char *Vs = smem + L::kV;
    float *Qs = reinterpret_cast<float *>(smem + L::kQ);
    float *Ps = reinterpret_cast<float *>(smem + L::kP);
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    float *wm = reinterpret_cast<float *>(smem + L::kWm);
    float *ls = reinterpret_cast<float *>(smem + L::kL);

    const int k = blockIdx.x % kClusterCtas;          // rank in the cluster (clusters run along x)
    const int c = blockIdx.x / kClusterCtas, hk = blockIdx.y;
    const int G = a.Hq / a.Hkv;
    const int rows = a.M * G;                          // <= R
    const int n_max = chunk_positions(a.T0, a.M - 1, c);
    if (n_max == 0) return;                            // the whole cluster: it depends on the chunk only
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = kChunk * c, tk = 64 * k;           // first position of the chunk, of this CTA's quarter
    const size_t kv_row = static_cast<size_t>(a.Hkv) * D;
    auto row_n = [&](int r) { return r < rows ? chunk_positions(a.T0, r / G, c) : 0; };

    // ---- stage: q (all rows), K of this CTA's 64 positions, then V's d slice of all positions
    for (int i = tid; i < 64 * kW; i += kClusterThreads) {
        const int t = i / kW, sg = i - t * kW;
        if (tk + t < n_max) cp_async16(Ks + t * L::kRow + 16 * sg, a.k + (t0 + tk + t) * kv_row + hk * D + 8 * sg);
    }
    cp_async_commit();
    for (int i = tid; i < n_max * 4; i += kClusterThreads) {
        const int t = i >> 2, sg = i & 3;
        cp_async16(Vs + t * 64 + 16 * sg, a.v + (t0 + t) * kv_row + hk * D + 32 * k + 8 * sg);
    }
    cp_async_commit();
    for (int i = tid; i < R * kW; i += kClusterThreads) {
        const int qr = i % R, qs = i / R;
        uint4 qv = make_uint4(0u, 0u, 0u, 0u);
        if (qr < rows) {
            const int m = qr / G, h = hk * G + (qr - m * G);
            qv = __ldg(reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(m) * a.Hq + h) * D) + qs);
        }
        float *dst = Qs + 8 * qs * R + qr;
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            dst[(2 * e) * R] = __uint_as_float(w[e] << 16);
            dst[(2 * e + 1) * R] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
    const ExpCoef ec = exp_coef();
    cluster_sync_all();                                // 1: every CTA of the cluster is running
    cp_async_wait<1>();                                // this thread's K copies have landed
    __syncthreads();                                   // and everyone's; q staged

    // ---- scores: warps 0-3, position p = tid % 64 of this quarter, row pairs g * kPairs ..
    const bool scorer = tid < 128;
    const int p = tid & 63, g = (tid >> 6) & 1;
    float s[2 * kPairs];
    if (scorer) {
        unsigned long long sc[kPairs];
#pragma unroll
        for (int ip = 0; ip < kPairs; ++ip) sc[ip] = 0ull;
        const unsigned char *kb = Ks + p * L::kRow;
#pragma unroll 4
        for (int j = 0; j < kW; ++j) {
            const uint4 kj = *reinterpret_cast<const uint4 *>(kb + 16 * j);
            const uint32_t w[4] = {kj.x, kj.y, kj.z, kj.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = 8 * j + e;
                const float kf = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
                const unsigned long long kd = pk(kf, kf);
                if constexpr (kPairs == 2) {
                    unsigned long long q2[2];
                    lds2x64(Qs + d * R + 4 * g, q2[0], q2[1]);
                    sc[0] = fma2(q2[0], kd, sc[0]);
                    sc[1] = fma2(q2[1], kd, sc[1]);
                } else {
                    const unsigned long long q2 = *reinterpret_cast<const unsigned long long *>(Qs + d * R + 2 * g);
                    sc[0] = fma2(q2, kd, sc[0]);
                }
            }
        }
#pragma unroll
        for (int ip = 0; ip < kPairs; ++ip) upk(sc[ip], s[2 * ip], s[2 * ip + 1]);
        // scale, mask, maxima over this warp's 32 positions
#pragma unroll
        for (int x = 0; x < 2 * kPairs; ++x) {
            const int r = 2 * kPairs * g + x;
            s[x] = tk + p < row_n(r) ? __fmul_rn(s[x], a.scale) : -INFINITY;
            float mx = s[x];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) wm[warp * R + r] = mx;
        }
    }
    __syncthreads();
    // this CTA's maxima (over its 64 positions) to every CTA of the cluster
    if (tid < R) {
        const int r = tid, gw = r / (2 * kPairs);      // warps 2 gw, 2 gw + 1 hold row r
        const float mx = fmaxf(wm[(2 * gw) * R + r], wm[(2 * gw + 1) * R + r]);
        const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(red + r * kClusterCtas + k));
#pragma unroll
        for (int q = 0; q < kClusterCtas; ++q) st_cluster_f32(cluster_map(local, q), mx);
    }
    cluster_sync_all();                                // 2: every CTA has every quarter's maxima
    // ---- weights of this quarter's positions to every CTA
    if (scorer) {
#pragma unroll
        for (int x = 0; x < 2 * kPairs; ++x) {
            const int r = 2 * kPairs * g + x;
            const float4 m4 = *reinterpret_cast<const float4 *>(red + r * kClusterCtas);
            const float mx = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
            const float pv = s[x] == -INFINITY ? 0.0f : attn_e(__fsub_rn(s[x], mx), ec);
            const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(Ps + r * kChunk + tk + p));
#pragma unroll
            for (int q = 0; q < kClusterCtas; ++q) st_cluster_f32(cluster_map(local, q), pv);
        }
    }
    cp_async_wait<0>();                                // this thread's V copies have landed
    cluster_sync_all();                                // 3: all weights everywhere (the last remote stores)
    __syncthreads();                                   // V staged by every thread

    // ---- weight sums (warp 4) and weighted values (this CTA's d slice)
    if (warp == 4) {
        if (lane < R) {
            const int r = lane, n = row_n(r);
            const float *pr = Ps + r * kChunk;
            float l = 0.0f;
            int t = 0;
            for (; t + 4 <= n; t += 4) {
                const float4 p4 = *reinterpret_cast<const float4 *>(pr + t);
                l = __fadd_rn(l, p4.x);
                l = __fadd_rn(l, p4.y);
                l = __fadd_rn(l, p4.z);
                l = __fadd_rn(l, p4.w);
            }
            for (; t < n; ++t) l = __fadd_rn(l, pr[t]);
            ls[r] = l;
        }
    }
    const int r = tid >> 4, j = tid & 15;              // value unit: row r, d = 32 k + 2 j, + 1
    const bool valuer = tid < 16 * R;
    const int nr = valuer ? row_n(r) : 0;
    unsigned long long acc = 0ull;
    if (valuer && nr > 0) {
        const float *pr = Ps + r * kChunk;
        const unsigned char *vb = Vs + 4 * j;
        int t = 0;
        for (; t + 4 <= nr; t += 4) {
            const float4 p4 = *reinterpret_cast<const float4 *>(pr + t);
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint32_t vv = *reinterpret_cast<const uint32_t *>(vb + (t + x) * 64);
                acc = fma2(pk(pp[x], pp[x]), pk(__uint_as_float(vv << 16), __uint_as_float(vv & 0xFFFF0000u)), acc);
            }
        }
        for (; t < nr; ++t) {
            const float pv = pr[t];
            const uint32_t vv = *reinterpret_cast<const uint32_t *>(vb + t * 64);
            acc = fma2(pk(pv, pv), pk(__uint_as_float(vv << 16), __uint_as_float(vv & 0xFFFF0000u)), acc);
        }
    }
    __syncthreads();                                   // the weight sums in ls
    if (!valuer || nr == 0) return;
    const int m = r / G, h = hk * G + (r - m * G);
    float a0, a1;
    upk(acc, a0, a1);
    const float l = ls[r];
    const int dd = 32 * k + 2 * j;
    if (a.T0 + m + 1 <= kChunk) {                      // the query's only chunk: o = a / l
        const uint32_t ob = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(a0, l))) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(a1, l)))) << 16);
        *reinterpret_cast<uint32_t *>(a.o + (static_cast<size_t>(m) * a.Hq + h) * D + dd) = ob;
    } else {
        float *part = a.ws + ((static_cast<size_t>(m) * a.Hq + h) * a.Cmax + c) * (D + 4);
        if (k == 0 && j == 0) {
            const float4 m4 = *reinterpret_cast<const float4 *>(red + r * kClusterCtas);
            part[0] = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
            part[1] = l;
        }
        *reinterpret_cast<float2 *>(part + 4 + dd) = make_float2(a0, a1);
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

template <int D, int R>
cudaError_t launch_small(const AttnArgs &a, cudaStream_t stream)
{
    constexpr int bytes = SmallSmem<D, R>::kBytes;
    static bool configured = false;                    // one attribute call per process and shape
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(attn_chunk_small_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    attn_chunk_small_kernel<D, R>
        <<<dim3(static_cast<unsigned>(a.Cmax), static_cast<unsigned>(a.Hkv)), kSmallThreads, bytes, stream>>>(a);
    return cudaGetLastError();
}

template <int R>
cudaError_t launch_cluster(const AttnArgs &a, cudaStream_t stream)
{
    constexpr int bytes = ClusterSmem<R>::kBytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.Cmax * kClusterCtas), static_cast<unsigned>(a.Hkv));
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_chunk_cluster_kernel<R>, a);
}

template <int D>
cudaError_t launch_rows(const AttnArgs &a, cudaStream_t stream)
{
    const int G = a.Hq / a.Hkv;
    const int rows = a.M * G;
    // the four-CTA clusters while they need at most two CTAs per SM (measured
    // faster up to about 2048 cached positions at one and two queries); the
    // one-CTA kernel on larger grids, where four CTAs sharing an SM cost more
    // than the quarter-size staging saves
    if constexpr (D == 128) {
        const bool clusters = static_cast<long long>(a.Cmax) * a.Hkv * kClusterCtas <= 2LL * a.sms;
        if (clusters && rows <= 4) return launch_cluster<4>(a, stream);
        if (clusters && rows <= 8) return launch_cluster<8>(a, stream);
    }
    if (rows <= 4) return launch_small<D, 4>(a, stream);
    if (rows <= 8) return launch_small<D, 8>(a, stream);
    constexpr int bytes = ChunkSmem<D>::kBytes;
    static bool configured = false;                    // one attribute call per process and head size
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int blocks = (rows + kRows - 1) / kRows;
    attn_chunk_kernel<D><<<dim3(static_cast<unsigned>(a.Cmax), static_cast<unsigned>(a.Hkv),
                                static_cast<unsigned>(blocks)),
                           kAttnThreads, bytes, stream>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t stream)
{
    cudaError_t e = launch_rows<D>(a, stream);
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
