// Block-scaled variant of the verify-pass linear: the mat-vec of "why
// speculative decoding changed my output", "the mat-vec kernel".  q6-style
// weight blocks of 256 (16 sub-blocks of 16, 6-bit codes, int8 sub-scales,
// fp32 super-block scales), int8 activation blocks of 32 with fp32 scales;
// integer products inside a block, then an fp32 scale-and-add whose order
// depends on K only, so every token of every pass (M = 1 .. 16) gets the
// same adds:
//   isum_b = sc_j * sum(c * q) over the block's first 16 elements
//          + sc_(j+1) * sum over the next 16          (j = 2b; exact, < 2^24)
//   v_b    = ((float)isum_b * d_a[b]) * d[b / 8]
//   lane l of the row's warp: p = +0; p += v_l, v_(l+32), v_(l+64), ...
//   then p += shfl_xor(p, 16), 8, 4, 2, 1;  y = p (fp32).
// Stored layout (per row): ql [K/2] low 4 bits of c + 32 (element k in byte
// k/2, bits 4 (k & 1)); qh [K/4] high 2 bits (element k in byte k/4, bits
// 2 (k & 3)); sc [K/16]; d [K/256].
#include "blockq.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kQ6Threads = 256;
constexpr int kLinWarps = 8;                      // warps per CTA of the mat-vec

// clamp(rne(v), lo, hi) of an fp32 value (rne as the IEEE conversion does).
__device__ __forceinline__ int rne_clamp(float v, int lo, int hi)
{
    return max(lo, min(hi, __float2int_rn(v)));
}

// One thread per 16-weight sub-block; the 16 threads of a super-block are a
// half-warp, which finds the super-block's largest sub-block scale.
__global__ void __launch_bounds__(kQ6Threads) quantize_q6_kernel(const float *__restrict__ w, int64_t ldw, int K,
                                                                uint8_t *ql, uint8_t *qh, int8_t *sc, float *d)
{
    const int64_t n = blockIdx.x;
    const float *wr = w + n * ldw;
    const int nsub = K / 16;
    for (int j0 = 0; j0 < nsub; j0 += kQ6Threads) {
        const int j = j0 + static_cast<int>(threadIdx.x);   // nsub is a multiple of 16: half-warps stay whole
        const bool live = j < nsub;
        float v[16];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = live ? wr[16 * j + i] : 0.0f;
            amax = fmaxf(amax, fabsf(v[i]));
        }
        const float t = __fdiv_rn(amax, 31.0f);
        float tmax = t;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        if (!live) continue;
        const float ds = (tmax == 0.0f) ? 1.0f : __fdiv_rn(tmax, 127.0f);
        const int scj = rne_clamp(__fdiv_rn(t, ds), 0, 127);
        const float e = __fmul_rn(ds, static_cast<float>(scj));
        uint32_t lo[2] = {0u, 0u}, hi = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = (e != 0.0f) ? rne_clamp(__fdiv_rn(v[i], e), -32, 31) : 0;
            const uint32_t u = static_cast<uint32_t>(c + 32);
            lo[i >> 3] |= (u & 0xFu) << (4 * (i & 7));
            hi |= (u >> 4) << (2 * i);
        }
        *reinterpret_cast<uint2 *>(ql + n * (K / 2) + 8 * j) = make_uint2(lo[0], lo[1]);
        *reinterpret_cast<uint32_t *>(qh + n * (K / 4) + 4 * j) = hi;
        sc[n * nsub + j] = static_cast<int8_t>(scj);
        if ((j & 15) == 0) d[n * (K / 256) + j / 16] = ds;
    }
}

// One warp per activation block of 32: the per-token rule applied to the block.
__global__ void quantize_act_blocks_kernel(const uint16_t *__restrict__ x, int64_t ldx, int M, int K, int8_t *q,
                                           float *d_a)
{
    const int lane = threadIdx.x & 31;
    const long long blk = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int nb = K / 32;
    if (blk >= static_cast<long long>(M) * nb) return;
    const int m = static_cast<int>(blk / nb), b = static_cast<int>(blk % nb);
    const float v = __uint_as_float(static_cast<uint32_t>(x[m * ldx + 32 * b + lane]) << 16);
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
    q[static_cast<long long>(m) * K + 32 * b + lane] = static_cast<int8_t>(rne_clamp(__fdiv_rn(v, s), -127, 127));
    if (lane == 0) d_a[static_cast<long long>(m) * nb + b] = s;
}

// 32 codes of one 32-block as unsigned bytes u = c + 32 in [0, 63], in the
// order the stored bits give them cheaply: word 4q + j holds elements
// 16q + j, 16q + 4 + j, 16q + 8 + j, 16q + 12 + j (q = 0, 1; j = 0 .. 3).
// High bits: field j of every byte of qh word q, masked and moved to bits
// 4-5.  Low nibbles: of the ql words 2q and 2q + 1, bytes 0 and 2 hold those
// elements for j = 0, 1 (low, high nibble) and bytes 1 and 3 for j = 2, 3; one
// byte permute gathers each pair.  The activations are stored in the same
// order (act_natural_order), so the integer dot products are unchanged.
__device__ __forceinline__ void unpack32n(uint4 l, uint2 h, uint32_t (&u)[8])
{
    const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
    const uint32_t hw[2] = {h.x, h.y};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t w = hw[q];
        const uint32_t x0 = __byte_perm(lw[2 * q], lw[2 * q + 1], 0x6420);   // bytes 0, 2 of each
        const uint32_t x1 = __byte_perm(lw[2 * q], lw[2 * q + 1], 0x7531);   // bytes 1, 3 of each
        u[4 * q + 0] = (x0 & 0x0F0F0F0Fu) | ((w << 4) & 0x30303030u);
        u[4 * q + 1] = ((x0 >> 4) & 0x0F0F0F0Fu) | ((w << 2) & 0x30303030u);
        u[4 * q + 2] = (x1 & 0x0F0F0F0Fu) | (w & 0x30303030u);
        u[4 * q + 3] = ((x1 >> 4) & 0x0F0F0F0Fu) | ((w >> 2) & 0x30303030u);
    }
}

// 16 activation bytes (elements 4i + k in byte k of word i) in the order of
// unpack32n: word j = elements j, 4 + j, 8 + j, 12 + j (a 4 x 4 byte transpose).
__device__ __forceinline__ uint4 act_natural_order(uint4 a)
{
    const uint32_t t01l = __byte_perm(a.x, a.y, 0x5140), t23l = __byte_perm(a.z, a.w, 0x5140);
    const uint32_t t01h = __byte_perm(a.x, a.y, 0x7362), t23h = __byte_perm(a.z, a.w, 0x7362);
    return make_uint4(__byte_perm(t01l, t23l, 0x5410), __byte_perm(t01l, t23l, 0x7632),
                      __byte_perm(t01h, t23h, 0x5410), __byte_perm(t01h, t23h, 0x7632));
}

// sum over 4 byte pairs of (unsigned a byte) * (signed b byte), plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The stored weight data of one 32-block of one row.
struct BlockW {
    uint4 l;       // 16 bytes of ql: 32 low nibbles
    uint2 h;       // 8 bytes of qh: 32 high 2-bit fields
    char2 s;       // the two sub-block scales
    float d;       // the super-block scale
};

__device__ __forceinline__ BlockW load_block(const uint8_t *__restrict__ ql, const uint8_t *__restrict__ qh,
                                             const int8_t *__restrict__ sc, const float *__restrict__ d, int n, int K,
                                             int b)
{
    BlockW w;
    w.l = __ldg(reinterpret_cast<const uint4 *>(ql + static_cast<size_t>(n) * (K / 2)) + b);
    w.h = __ldg(reinterpret_cast<const uint2 *>(qh + static_cast<size_t>(n) * (K / 4)) + b);
    w.s = __ldg(reinterpret_cast<const char2 *>(sc + static_cast<size_t>(n) * (K / 16)) + b);
    w.d = __ldg(d + static_cast<size_t>(n) * (K / 256) + b / 8);
    return w;
}

__device__ __forceinline__ void q6_cp_async_16(void *smem, const void *gmem)
{
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void q6_cp_async_4(void *smem, const void *gmem)
{
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(gmem) : "memory");
}

// Shared-memory bytes of the staged activations of M tokens: per (token,
// block) the 32 codes, the two sub-block sums and the scale.
__host__ __device__ constexpr size_t q6_stage_bytes(int M, int K) { return static_cast<size_t>(M) * (K / 32) * 44; }

// y [M, N] fp32, M <= MT.  One warp per R rows; lane l takes 32-blocks
// l, l + 32, ... in that order (the next one's weights are loaded while the
// current one is computed), and each activation block is loaded once for the
// warp's R rows.  MT and R change the work per thread, not the adds.
// STAGED: the CTA first copies the activation codes and scales into shared
// memory, forms each block's two sub-block sums and puts its codes in the
// order of unpack32n once (instead of every warp loading them from L1 and
// doing so per block); the block's two 16-byte halves are stored swapped when
// bit 2 of its index is set, so that 8 lanes reading 8 consecutive blocks hit
// distinct banks.
template <int MT, int R, bool STAGED>
__device__ __forceinline__ void linear_q6_body(const int8_t *__restrict__ qa, const float *__restrict__ d_a, int M,
                                               int K, const uint8_t *__restrict__ ql, const uint8_t *__restrict__ qh,
                                               const int8_t *__restrict__ sc, const float *__restrict__ d, int N,
                                               float *y, int pdl)
{
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int lane = threadIdx.x & 31;
    const int n0 = (blockIdx.x * kLinWarps + (threadIdx.x >> 5)) * R;
    const int nb = K / 32;
    extern __shared__ __align__(16) unsigned char q6s[];
    unsigned char *sact = q6s;                                                             // [M][nb][32]
    int2 *ssum = reinterpret_cast<int2 *>(q6s + static_cast<size_t>(M) * nb * 32);         // [M][nb]
    float *sda = reinterpret_cast<float *>(q6s + static_cast<size_t>(M) * nb * 40);       // [M][nb]
    if constexpr (STAGED) {
        const int items = M * nb;
        for (int i = threadIdx.x; i < items; i += blockDim.x) {
            const int b = i % nb;
            const int8_t *src = qa + static_cast<size_t>(i / nb) * K + 32 * b;
            unsigned char *dst = sact + static_cast<size_t>(i) * 32;
            const int sw = (b >> 2) & 1;
            q6_cp_async_16(dst + 16 * sw, src);
            q6_cp_async_16(dst + 16 * (sw ^ 1), src + 16);
            q6_cp_async_4(sda + i, d_a + i);
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        for (int i = threadIdx.x; i < items; i += blockDim.x) {   // the items this thread copied
            const int sw = ((i % nb) >> 2) & 1;
            const uint4 h0 = *reinterpret_cast<const uint4 *>(sact + static_cast<size_t>(i) * 32 + 16 * sw);
            const uint4 h1 = *reinterpret_cast<const uint4 *>(sact + static_cast<size_t>(i) * 32 + 16 * (sw ^ 1));
            int s0 = 0, s1 = 0;
            s0 = __dp4a(0x01010101, static_cast<int>(h0.x), s0);
            s0 = __dp4a(0x01010101, static_cast<int>(h0.y), s0);
            s0 = __dp4a(0x01010101, static_cast<int>(h0.z), s0);
            s0 = __dp4a(0x01010101, static_cast<int>(h0.w), s0);
            s1 = __dp4a(0x01010101, static_cast<int>(h1.x), s1);
            s1 = __dp4a(0x01010101, static_cast<int>(h1.y), s1);
            s1 = __dp4a(0x01010101, static_cast<int>(h1.z), s1);
            s1 = __dp4a(0x01010101, static_cast<int>(h1.w), s1);
            ssum[i] = make_int2(-32 * s0, -32 * s1);   // each sub-block's dp4a chain starts here
            *reinterpret_cast<uint4 *>(sact + static_cast<size_t>(i) * 32 + 16 * sw) = act_natural_order(h0);
            *reinterpret_cast<uint4 *>(sact + static_cast<size_t>(i) * 32 + 16 * (sw ^ 1)) = act_natural_order(h1);
        }
        __syncthreads();
    }
    if (n0 >= N) return;
    float p[MT][R];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) p[m][r] = 0.0f;
    BlockW cur[R], nxt[R];
    if (lane < nb) {
#pragma unroll
        for (int r = 0; r < R; ++r) cur[r] = load_block(ql, qh, sc, d, min(n0 + r, N - 1), K, lane);
    }
    for (int b = lane; b < nb; b += 32) {
        if (b + 32 < nb) {
#pragma unroll
            for (int r = 0; r < R; ++r) nxt[r] = load_block(ql, qh, sc, d, min(n0 + r, N - 1), K, b + 32);
        }
        uint32_t u[R][8];                              // codes + 32, unsigned
#pragma unroll
        for (int r = 0; r < R; ++r) unpack32n(cur[r].l, cur[r].h, u[r]);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m >= M) break;
            uint4 a0, a1;
            float da;
            int as0 = 0, as1 = 0;                      // sum(c a) = sum(u a) - 32 sum(a) per sub-block of 16:
                                                       // the dp4a chains start at -32 sum(a)
            if constexpr (STAGED) {
                const size_t it = static_cast<size_t>(m) * nb + b;
                const int sw = (b >> 2) & 1;
                a0 = *reinterpret_cast<const uint4 *>(sact + it * 32 + 16 * sw);
                a1 = *reinterpret_cast<const uint4 *>(sact + it * 32 + 16 * (sw ^ 1));
                da = sda[it];
                const int2 as = ssum[it];
                as0 = as.x;
                as1 = as.y;
            } else {
                a0 = __ldg(reinterpret_cast<const uint4 *>(qa + static_cast<size_t>(m) * K) + 2 * b);
                a1 = __ldg(reinterpret_cast<const uint4 *>(qa + static_cast<size_t>(m) * K) + 2 * b + 1);
                da = __ldg(d_a + static_cast<size_t>(m) * nb + b);
                as0 = __dp4a(0x01010101, static_cast<int>(a0.x), as0);
                as0 = __dp4a(0x01010101, static_cast<int>(a0.y), as0);
                as0 = __dp4a(0x01010101, static_cast<int>(a0.z), as0);
                as0 = __dp4a(0x01010101, static_cast<int>(a0.w), as0);
                as1 = __dp4a(0x01010101, static_cast<int>(a1.x), as1);
                as1 = __dp4a(0x01010101, static_cast<int>(a1.y), as1);
                as1 = __dp4a(0x01010101, static_cast<int>(a1.z), as1);
                as1 = __dp4a(0x01010101, static_cast<int>(a1.w), as1);
                as0 *= -32;
                as1 *= -32;
                a0 = act_natural_order(a0);
                a1 = act_natural_order(a1);
            }
            const int a[8] = {static_cast<int>(a0.x), static_cast<int>(a0.y), static_cast<int>(a0.z),
                              static_cast<int>(a0.w), static_cast<int>(a1.x), static_cast<int>(a1.y),
                              static_cast<int>(a1.z), static_cast<int>(a1.w)};
#pragma unroll
            for (int r = 0; r < R; ++r) {
                int s0 = as0, s1 = as1;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    s0 = dp4a_us(u[r][k], a[k], s0);
                    s1 = dp4a_us(u[r][4 + k], a[4 + k], s1);
                }
                const int isum = cur[r].s.x * s0 + cur[r].s.y * s1;
                const float v = __fmul_rn(__fmul_rn(__int2float_rn(isum), da), cur[r].d);
                p[m][r] = __fadd_rn(p[m][r], v);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) cur[r] = nxt[r];
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float v = p[m][r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0 && n0 + r < N) y[static_cast<size_t>(m) * N + n0 + r] = v;
        }
    }
}

template <int MT, int R, bool STAGED>
__global__ void __launch_bounds__(kLinWarps * 32) linear_q6_kernel(const int8_t *__restrict__ qa,
                                                                   const float *__restrict__ d_a, int M, int K,
                                                                   const uint8_t *__restrict__ ql,
                                                                   const uint8_t *__restrict__ qh,
                                                                   const int8_t *__restrict__ sc,
                                                                   const float *__restrict__ d, int N, float *y,
                                                                   int pdl)
{
    linear_q6_body<MT, R, STAGED>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl);
}

// One token: fewer live registers, so more warps per SM keep weight loads in flight.
__global__ void __launch_bounds__(kLinWarps * 32, 5) linear_q6_kernel_m1(const int8_t *__restrict__ qa,
                                                                         const float *__restrict__ d_a, int M, int K,
                                                                         const uint8_t *__restrict__ ql,
                                                                         const uint8_t *__restrict__ qh,
                                                                         const int8_t *__restrict__ sc,
                                                                         const float *__restrict__ d, int N, float *y,
                                                                         int pdl)
{
    linear_q6_body<1, 1, false>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl);
}

constexpr size_t kQ6StageMax = 96 * 1024;

template <int MT, int R>
cudaError_t launch_q6(const int8_t *qa, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                      const int8_t *sc, const float *d, int N, float *y, bool pdl, cudaStream_t stream)
{
    const int rows_per_cta = kLinWarps * R;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + rows_per_cta - 1) / rows_per_cta));
    cfg.blockDim = dim3(kLinWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if constexpr (MT == 1) {
        return cudaLaunchKernelEx(&cfg, linear_q6_kernel_m1, qa, d_a, M, K, ql, qh, sc, d, N, y, pdl ? 1 : 0);
    } else {
        // the activations staged in shared memory while they fit beside a
        // second CTA on the SM; otherwise loaded per warp
        const size_t bytes = q6_stage_bytes(M, K);
        if (bytes > kQ6StageMax)
            return cudaLaunchKernelEx(&cfg, linear_q6_kernel<MT, R, false>, qa, d_a, M, K, ql, qh, sc, d, N, y,
                                      pdl ? 1 : 0);
        static bool configured = false;                // one attribute call per process and shape
        if (!configured) {
            const cudaError_t e = cudaFuncSetAttribute(linear_q6_kernel<MT, R, true>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kQ6StageMax));
            if (e != cudaSuccess) return e;
            configured = true;
        }
        cfg.dynamicSmemBytes = bytes;
        return cudaLaunchKernelEx(&cfg, linear_q6_kernel<MT, R, true>, qa, d_a, M, K, ql, qh, sc, d, N, y,
                                  pdl ? 1 : 0);
    }
}

}  // namespace

cudaError_t launch_quantize_q6(const float *w, int64_t ldw, int N, int K, uint8_t *ql, uint8_t *qh, int8_t *sc,
                               float *d, cudaStream_t stream)
{
    quantize_q6_kernel<<<static_cast<unsigned>(N), kQ6Threads, 0, stream>>>(w, ldw, K, ql, qh, sc, d);
    return cudaGetLastError();
}

cudaError_t launch_quantize_act_blocks(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *d_a,
                                       cudaStream_t stream)
{
    const long long blocks = static_cast<long long>(M) * (K / 32);
    const unsigned grid = static_cast<unsigned>((blocks + 7) / 8);
    quantize_act_blocks_kernel<<<grid, 256, 0, stream>>>(x, ldx, M, K, q, d_a);
    return cudaGetLastError();
}

cudaError_t launch_linear_q6(const int8_t *qa, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                             const int8_t *sc, const float *d, int N, float *y, bool pdl, cudaStream_t stream)
{
    // one row per warp at M <= 4; two above, where each activation load then
    // serves two rows (measured best of one, two and four rows per warp)
    if (M == 1) return launch_q6<1, 1>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl, stream);
    if (M <= 4) return launch_q6<4, 1>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl, stream);
    if (M <= 8) return launch_q6<8, 2>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl, stream);
    return launch_q6<16, 2>(qa, d_a, M, K, ql, qh, sc, d, N, y, pdl, stream);
}

}  // namespace bi
