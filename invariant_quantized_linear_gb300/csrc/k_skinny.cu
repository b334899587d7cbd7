// Weight-streaming W8A8 kernel for M <= 16 tokens (decode / speculative
// verify), plain linear or LM head with a fused greedy argmax.
//
// The weight read is the whole cost of such a pass ("why speculative decoding
// changed my output", Fig. 1; "My speculative decoder got slower", "The
// physics"), so the kernel is built to stream W at HBM speed:
//  * persistent grid, one CTA per SM; the flattened sequence of units
//    (64 weight rows x 256 bytes of K) is cut into equal contiguous ranges,
//    one per CTA, so every SM reads the same number of bytes;
//  * a producer warp moves each unit's weight tile and the matching slice of
//    the int8 activations into a ring of shared-memory stages with TMA
//    (128-byte swizzle, evict-first L2 policy for the weights);
//  * four consumer warps own 16 weight rows each and run int8 tensor-core
//    MMAs (m16n8k32: weight rows as the 16-row operand, tokens as the 8
//    columns) into int32 accumulators;
//  * a row block whose K range straddles two CTAs is finished through int32
//    atomics in the workspace; the CTA that completes the count applies the
//    epilogue.  Integer sums are exact, so the split, the MMA order and the
//    atomic order cannot change a bit ("The Integer Alibi", abstract), and
//    none of them depends on M.
// Epilogue, per element: bf16_rne(fmul_rn(fmul_rn(i2f_rn(acc), s_a), s_w))
// ("Deterministic LLM Inference Across GPU Kernels ...", Table II, the
// complement of faults F1-F5).
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kNch = 2;                    // 128-byte chunks of K per unit
constexpr int kUnitK = kNch * 128;         // bytes of K per unit
constexpr int kWChunkBytes = kBM * 128;    // 8 KB: 64 rows x 128 B

template <int MT>
struct Cfg {
    static constexpr int kTok = 8 * MT;                         // token rows staged
    static constexpr int kAChunkBytes = kTok * 128;             // 1 or 2 KB
    static constexpr int kWStage = kNch * kWChunkBytes;         // 16 KB
    static constexpr int kAStage = kNch * kAChunkBytes;         // 2 or 4 KB
    static constexpr int kStages = (MT == 1) ? 6 : 5;           // <= ~110 KB of shared memory
    static constexpr int kSmemBytes = kStages * (kWStage + kAStage) + 1024 /*align*/ + 1024 /*barriers, flags*/;
};

struct Params {
    const float *s_a;
    const float *s_w;
    uint16_t *y;
    int32_t *argmax;
    int M, N, K;
    int upr;          // units per row block
    long long units;  // total units
    Workspace ws;
    int pdl;
};

__device__ __forceinline__ long long range_start(long long i, long long units, int G)
{
    return (i * units) / G;
}

// CTA whose range holds unit u: the largest i with range_start(i) <= u.
__device__ __forceinline__ int unit_owner(long long u, long long units, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / units);
}

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
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

template <int MT, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_q, Params p)
{
    using C = Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;                                   // [stages][kNch][64 rows][128 B]
    uint8_t *sA = smem + C::kStages * C::kWStage;         // [stages][kNch][kTok rows][128 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(sA + C::kStages * C::kAStage);
    uint64_t *empty = full + C::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::kStages);
    volatile int *last_flag = abort_flag + 1;
    unsigned long long *sbest = reinterpret_cast<unsigned long long *>(empty + C::kStages + 2);  // [4][16]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long u_begin = range_start(blockIdx.x, p.units, G);
    const long long u_end = range_start(blockIdx.x + 1, p.units, G);
    const int n_units = static_cast<int>(u_end - u_begin);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (p.pdl) pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_units > 0) {
            prefetch_tensormap(&map_w);
            prefetch_tensormap(&map_q);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const uint32_t stage_bytes = C::kWStage + C::kAStage;
            auto issue_w = [&](int j) {
                const int s = j % C::kStages;
                const long long u = u_begin + j;
                const int rb = static_cast<int>(u / p.upr), c = static_cast<int>(u % p.upr);
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sW + s * C::kWStage + ch * kWChunkBytes, &map_w, &full[s], c * kUnitK + ch * 128,
                                rb * kBM, pol_w);
            };
            auto issue_a = [&](int j) {
                const int s = j % C::kStages;
                const long long u = u_begin + j;
                const int c = static_cast<int>(u % p.upr);
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sA + s * C::kAStage + ch * C::kAChunkBytes, &map_q, &full[s], c * kUnitK + ch * 128,
                                0, pol_a);
            };
            // The weights do not depend on the preceding kernel: start them
            // before waiting for it; the activations only after.
            const int n_pre = n_units < C::kStages ? n_units : C::kStages;
            for (int j = 0; j < n_pre; ++j) {
                mbar_arrive_expect_tx(&full[j], stage_bytes);
                issue_w(j);
            }
            if (p.pdl) pdl_wait();
            for (int j = 0; j < n_pre; ++j) issue_a(j);
            int issued = n_pre;
            for (int j = n_pre; j < n_units; ++j) {
                const int s = j % C::kStages;
                if (!mbar_wait_bounded(&empty[s], ((j / C::kStages) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    atomicExch(p.ws.status, DEV_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                issue_w(j);
                issue_a(j);
                issued = j + 1;
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits
                volatile int never = 0;
                const int first = issued > C::kStages ? issued - C::kStages : 0;
                for (int j = first; j < issued; ++j)
                    mbar_wait_bounded(&full[j % C::kStages], (j / C::kStages) & 1, &never);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    if (p.pdl) pdl_wait();
    const int g = lane >> 2, tq = lane & 3;
    const int mat = lane >> 3, r8 = lane & 7;
    // ldmatrix row addresses: weight rows for the A operand, token rows for B
    const uint32_t a_row = warp * 16 + ((mat & 1) ? 8 : 0) + r8;
    const int a_hi = (mat & 2) ? 1 : 0;                    // chunk X or Y
    const uint32_t b_tok = (MT == 2 && (lane >> 4)) ? 8 + r8 : r8;
    const int b_hi = (lane >> 3) & 1;

    unsigned long long best[MT][2];
#pragma unroll
    for (int t = 0; t < MT; ++t) best[t][0] = best[t][1] = 0ull;

    int j = 0;
    long long u = u_begin;
    while (u < u_end) {
        const int rb = static_cast<int>(u / p.upr);
        const int c0 = static_cast<int>(u % p.upr);
        const long long left = u_end - u;
        const int nch = (p.upr - c0) < left ? (p.upr - c0) : static_cast<int>(left);
        int32_t acc[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0;

        for (int it = 0; it < nch; ++it, ++j) {
            const int s = j % C::kStages;
            if (*abort_flag || !mbar_wait_bounded(&full[s], (j / C::kStages) & 1, abort_flag)) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicExch(p.ws.status, DEV_TIMEOUT);
                }
                continue;
            }
            const uint32_t wbase = smem_u32(sW + s * C::kWStage);
            const uint32_t abase = smem_u32(sA + s * C::kAStage);
#pragma unroll
            for (int ch = 0; ch < kNch; ++ch) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(wbase + ch * kWChunkBytes + swz128(a_row, 2 * ks + a_hi), a0, a1, a2, a3);
                    if constexpr (MT == 1) {
                        uint32_t b0, b1;
                        ldmatrix_x2(abase + ch * C::kAChunkBytes + swz128(b_tok, 2 * ks + b_hi), b0, b1);
                        mma_s8_16832(acc[0], a0, a1, a2, a3, b0, b1);
                    } else {
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(abase + ch * C::kAChunkBytes + swz128(b_tok, 2 * ks + b_hi), b0, b1, b2, b3);
                        mma_s8_16832(acc[0], a0, a1, a2, a3, b0, b1);
                        mma_s8_16832(acc[1], a0, a1, a2, a3, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---------------------------------------------------- row-block flush
        bool finish = (c0 == 0 && nch == p.upr);
        if (!finish) {
            const int slot = unit_owner(static_cast<long long>(rb) * p.upr, p.units, G);
            int32_t *part = p.ws.partial + static_cast<size_t>(slot) * (kBM * kMaxTok);
            if (!*abort_flag) {
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = warp * 16 + g + ((i & 2) ? 8 : 0);
                        const int tok = 8 * t + 2 * tq + (i & 1);
                        if (acc[t][i] != 0) atomicAdd(&part[r * kMaxTok + tok], acc[t][i]);
                    }
                __threadfence();
            }
            consumer_bar();
            if (threadIdx.x == 0) {
                int last = 0;
                if (!*abort_flag) {
                    __threadfence();
                    const int old = atomicAdd(&p.ws.rb_counter[slot], nch);
                    last = (old + nch == p.upr);
                    if (last) atomicExch(&p.ws.rb_counter[slot], 0);
                }
                *last_flag = last;
            }
            consumer_bar();
            finish = *last_flag != 0;
            if (finish) {
                __threadfence();
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = warp * 16 + g + ((i & 2) ? 8 : 0);
                        const int tok = 8 * t + 2 * tq + (i & 1);
                        acc[t][i] = atomicExch(&part[r * kMaxTok + tok], 0);
                    }
            }
        }
        if (finish && !*abort_flag) {
            const int n0 = rb * kBM + warp * 16 + g;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = n0 + ((i & 2) ? 8 : 0);
                if (n >= p.N) continue;
                const float sw = p.s_w[n];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const int tok = 8 * t + 2 * tq + (i & 1);
                    if (tok >= p.M) continue;
                    float f = __int2float_rn(acc[t][i]);
                    f = __fmul_rn(f, p.s_a[tok]);
                    f = __fmul_rn(f, sw);
                    const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                    if (p.y) p.y[static_cast<size_t>(tok) * p.N + n] = b;
                    if constexpr (ARGMAX) {
                        const unsigned long long key = argmax_key(b, n);
                        if (key > best[t][i & 1]) best[t][i & 1] = key;
                    }
                }
            }
        }
        u += nch;
    }

    if constexpr (ARGMAX) {
        // per warp: reduce over the 8 lanes that share tq (lane bits 2..4)
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                unsigned long long v = best[t][h];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
                    v = w > v ? w : v;
                }
                if (g == 0) sbest[warp * kMaxTok + 8 * t + 2 * tq + h] = v;
            }
        if (MT == 1 && lane < 8) sbest[warp * kMaxTok + 8 + lane] = 0ull;
        consumer_bar();
        if (warp == 0) {
            if (lane < kMaxTok) {
                unsigned long long v = 0ull;
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const unsigned long long x = sbest[w * kMaxTok + lane];
                    v = x > v ? x : v;
                }
                p.ws.best[blockIdx.x * kMaxTok + lane] = v;
                __threadfence();
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence();
                last = (atomicAdd(p.ws.ticket, 1) == G - 1);
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                if (lane < p.M) {
                    unsigned long long v = 0ull;
                    for (int b = 0; b < G; ++b) {
                        const unsigned long long x = __ldcg(&p.ws.best[b * kMaxTok + lane]);
                        v = x > v ? x : v;
                    }
                    p.argmax[lane] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(v & 0xFFFFFFFFull));
                }
                if (lane == 0) atomicExch(p.ws.ticket, 0);
            }
        }
    }
}

template <int MT, bool ARGMAX>
cudaError_t launch_t(const SkinnyArgs &a, cudaStream_t stream)
{
    using C = Cfg<MT>;
    auto kern = skinny_kernel<MT, ARGMAX>;
    static bool attr_set = false;  // per process; the attribute applies to every device
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.y = a.y;
    p.argmax = a.argmax;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.upr = (a.K + kUnitK - 1) / kUnitK;
    p.units = static_cast<long long>((a.N + kBM - 1) / kBM) * p.upr;
    p.ws = a.ws;
    p.pdl = a.pdl ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a.map_w, a.map_q, p);
}

}  // namespace

cudaError_t launch_skinny(const SkinnyArgs &a, cudaStream_t stream)
{
    const bool two = a.M > 8;
    if (a.argmax) return two ? launch_t<2, true>(a, stream) : launch_t<1, true>(a, stream);
    return two ? launch_t<2, false>(a, stream) : launch_t<1, false>(a, stream);
}

}  // namespace bi
