// Tiled W8A8 kernel for prefill-sized batches (M > 16): a dense int8
// contraction with exact int32 accumulation and the same per-element
// epilogue as the weight-streaming kernel, so every row matches it bitwise.
//
// sm_103a has no int8 kind for tcgen05.mma, and its warp-level int8 MMA runs
// at a fraction of the f16 rate, so the contraction runs on f16 tensor-core
// MMAs (m16n8k16, fp32 accumulate) over int8 values converted exactly to f16;
// fp32 partials are moved into int32 totals while they are integers far below
// 2^24, so the sum is the exact integer dot product.  Tiles are moved by TMA
// into a ring of 128-byte-swizzled shared-memory stages by one producer warp;
// eight consumer warps each own a 32-token x 64-row tile.
// CTA tile: 128 tokens x 128 weight rows, 128 bytes of K per stage.
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kWarpsM = 4, kWarpsN = 2;
constexpr int kConsumers = kWarpsM * kWarpsN;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kTileM = 128, kTileN = 128, kTileK = 128;
constexpr int kStageQ = kTileM * kTileK;   // 16 KB
constexpr int kStageW = kTileN * kTileK;   // 16 KB
constexpr int kStages = 4;
constexpr int kSmemBytes = kStages * (kStageQ + kStageW) + 1024 + 256;

struct Params {
    const float *s_a;
    const float *s_w;
    uint16_t *y;
    int M, N, K;
    int kt;  // K tiles
    Workspace ws;
    int pdl;
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_q, Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;                                  // [stages][128 tokens][128 B]
    uint8_t *sW = smem + kStages * kStageQ;              // [stages][128 rows][128 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(sW + kStages * kStageW);
    uint64_t *empty = full + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileN;
    const int m0 = blockIdx.y * kTileM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (p.pdl) pdl_launch_dependents();

    if (warp == kConsumers) {
        if (lane == 0) {
            prefetch_tensormap(&map_w);
            prefetch_tensormap(&map_q);
            const uint64_t pol = policy_evict_last();  // both operands are re-read by other CTAs
            if (p.pdl) pdl_wait();
            int issued = 0;
            for (int j = 0; j < p.kt; ++j) {
                const int s = j % kStages;
                if (j >= kStages && !mbar_wait_bounded(&empty[s], ((j / kStages) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    atomicExch(p.ws.status, DEV_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kStageQ + kStageW);
                tma_load_2d(sQ + s * kStageQ, &map_q, &full[s], j * kTileK, m0, pol);
                tma_load_2d(sW + s * kStageW, &map_w, &full[s], j * kTileK, n0, pol);
                issued = j + 1;
            }
            if (*abort_flag) {
                volatile int never = 0;
                const int first = issued > kStages ? issued - kStages : 0;
                for (int j = first; j < issued; ++j) mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, &never);
            }
        }
        return;
    }

    if (p.pdl) pdl_wait();
    const int wm = warp % kWarpsM, wn = warp / kWarpsM;   // warp tile: tokens wm*32.., rows wn*64..
    const int g = lane >> 2, tq = lane & 3;
    const int mat = lane >> 3, r8 = lane & 7;
    // A operand (tokens): x4 = (tok 0-7, X), (tok 8-15, X), (tok 0-7, Y), (tok 8-15, Y)
    const uint32_t a_tok = wm * 32 + ((mat & 1) ? 8 : 0) + r8;
    const int a_hi = (mat >> 1) & 1;
    // B operand (weight rows): x4 = (rows 0-7, X), (rows 0-7, Y), (rows 8-15, X), (rows 8-15, Y)
    const uint32_t b_row = wn * 64 + ((mat & 2) ? 8 : 0) + r8;
    const int b_hi = mat & 1;

    // int32 totals; fp32 tensor-core partials are moved into them every two
    // stages (256 bytes of K: |partial| <= 256 * 127^2 < 2^22, exact in fp32)
    int32_t acc[2][8][4];
    float facc[2][8][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int jn = 0; jn < 8; ++jn)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[i][jn][e] = 0;
                facc[i][jn][e] = 0.0f;
            }

    for (int j = 0; j < p.kt; ++j) {
        const int s = j % kStages;
        if (*abort_flag || !mbar_wait_bounded(&full[s], (j / kStages) & 1, abort_flag)) {
            if (!*abort_flag) {
                *abort_flag = 1;
                atomicExch(p.ws.status, DEV_TIMEOUT);
            }
            break;
        }
        const uint32_t qb = smem_u32(sQ + s * kStageQ);
        const uint32_t wb = smem_u32(sW + s * kStageW);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            // int8 fragments of 32 bytes of K (chunks X and Y)
            uint32_t a8[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                ldmatrix_x4(qb + swz128(a_tok + 16 * i, 2 * ks + a_hi), a8[i][0], a8[i][1], a8[i][2], a8[i][3]);
            uint32_t b8[4][4];
#pragma unroll
            for (int jp = 0; jp < 4; ++jp)
                ldmatrix_x4(wb + swz128(b_row + 16 * jp, 2 * ks + b_hi), b8[jp][0], b8[jp][1], b8[jp][2], b8[jp][3]);
#pragma unroll
            for (int xy = 0; xy < 2; ++xy) {
                uint32_t a[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    i8x4_to_f16x2x2(a8[i][2 * xy], a[i][0], a[i][2]);      // token g
                    i8x4_to_f16x2x2(a8[i][2 * xy + 1], a[i][1], a[i][3]);  // token g + 8
                }
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    uint32_t b0, b1, b2, b3;
                    i8x4_to_f16x2x2(b8[jp][xy], b0, b1);       // rows 0-7 of the pair
                    i8x4_to_f16x2x2(b8[jp][2 + xy], b2, b3);   // rows 8-15
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        mma_f16_16816(facc[i][2 * jp], a[i][0], a[i][1], a[i][2], a[i][3], b0, b1);
                        mma_f16_16816(facc[i][2 * jp + 1], a[i][0], a[i][1], a[i][2], a[i][3], b2, b3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if ((j & 1) || j + 1 == p.kt) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int jn = 0; jn < 8; ++jn)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[i][jn][e] += f2i_exact(facc[i][jn][e]);
                        facc[i][jn][e] = 0.0f;
                    }
        }
    }
    if (*abort_flag) return;

    // epilogue: acc[i][jn] = (token wm*32 + 16i + g (+8), row wn*64 + 8jn + 2tq (+1))
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int tok = m0 + wm * 32 + 16 * i + g + 8 * h;
            if (tok >= p.M) continue;
            const float sa = p.s_a[tok];
            uint16_t *yr = p.y + static_cast<size_t>(tok) * p.N;
#pragma unroll
            for (int jn = 0; jn < 8; ++jn) {
                const int n = n0 + wn * 64 + 8 * jn + 2 * tq;
                uint16_t b[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int nn = n + e;
                    float f = __int2float_rn(acc[i][jn][2 * h + e]);
                    f = __fmul_rn(f, sa);
                    f = __fmul_rn(f, nn < p.N ? p.s_w[nn] : 0.0f);
                    b[e] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                }
                if (n + 1 < p.N && ((reinterpret_cast<uintptr_t>(yr + n) & 3u) == 0)) {
                    *reinterpret_cast<uint32_t *>(yr + n) = static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[1]) << 16);
                } else {
                    if (n < p.N) yr[n] = b[0];
                    if (n + 1 < p.N) yr[n + 1] = b[1];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.y = a.y;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.kt = (a.K + kTileK - 1) / kTileK;
    p.ws = a.ws;
    p.pdl = a.pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.N + kTileN - 1) / kTileN), static_cast<unsigned>((a.M + kTileM - 1) / kTileM));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_kernel, a.map_w, a.map_q, p);
}

}  // namespace bi
