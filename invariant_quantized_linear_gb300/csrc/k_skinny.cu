// Weight-streaming W8A8 kernel for M <= 16 tokens (decode / speculative
// verify), plain linear or LM head with a fused greedy argmax.
//
// The weight read is the whole cost of such a pass ("why speculative decoding
// changed my output", Fig. 1; "My speculative decoder got slower", "The
// physics"), so the kernel is built to stream W at HBM speed:
//  * persistent grid, two CTAs per SM for a large matrix, one for a small
//    one (the caller's choice, by measured speed); the flattened sequence of units
//    (64 weight rows x 256 bytes of K) is cut into equal contiguous ranges,
//    one per CTA, so every CTA reads the same number of bytes;
//  * a producer warp moves each unit's weight tile and the matching slice of
//    the int8 activations into a ring of shared-memory stages with TMA
//    (128-byte swizzle, evict-first L2 policy for the weights);
//  * eight consumer warps: four 16-row groups, each row group's 256 bytes
//    of K per stage split between two warps.  Half of the 32-byte K groups
//    (a quarter with 9..16 tokens) run on the int8 tensor-core MMA
//    (m16n8k32, int32 accumulate); the rest are converted exactly to f16 and
//    run on the f16 MMA (m16n8k16, fp32 accumulate), whose partials (integers
//    below 2^20) are moved into the int32 accumulators every stage.  On
//    sm_103a the int8 MMA alone runs at a fraction of the f16 rate and the
//    f16 MMA alone costs an int8 -> f16 conversion per operand; the split
//    keeps both pipes and the ALU clear of the weight stream's pace;
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
#include "stream_mma.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

using namespace stream;
using Gs = Geo<2>;   // eight consumer warps: two CTAs fit on one SM
constexpr int kKSplit = Gs::kKSplit;
constexpr int kConsumerWarps = Gs::kConsumerWarps;
constexpr int kThreads = Gs::kThreads;

template <int MT>
struct Cfg {
    static constexpr int kTok = 8 * MT;                         // token rows staged
    static constexpr int kAChunkBytes = kTok * 128;             // 1 or 2 KB
    static constexpr int kWStage = kNch * kWChunkBytes;         // 16 KB
    static constexpr int kAStage = kNch * kAChunkBytes;         // 2 or 4 KB
    static constexpr int kStages = (MT == 1) ? 5 : 4;           // two CTAs per SM fit
    static constexpr int kRedBytes = (kKSplit - 1) * kBM * kMaxTok * 4;  // cross-warp K reduction
    static constexpr int kCtlBytes = 2 * kStages * 8 + 16 + kConsumerWarps * kMaxTok * 8;  // barriers, flags, keys
    static constexpr int kSmemBytes = kStages * (kWStage + kAStage) + kRedBytes + 1024 /*align*/ + kCtlBytes;
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
__global__ void __launch_bounds__(kThreads, 2)
    skinny_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_q, Params p)
{
    using C = Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;                                   // [stages][kNch][64 rows][128 B]
    uint8_t *sA = smem + C::kStages * C::kWStage;         // [stages][kNch][kTok rows][128 B]
    int32_t *sred = reinterpret_cast<int32_t *>(sA + C::kStages * C::kAStage);   // [kKSplit-1][64][16]
    uint64_t *full = reinterpret_cast<uint64_t *>(sA + C::kStages * C::kAStage + C::kRedBytes);
    uint64_t *empty = full + C::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::kStages);
    volatile int *last_flag = abort_flag + 1;  // [2]
    unsigned long long *sbest = reinterpret_cast<unsigned long long *>(empty + C::kStages + 2);  // [warps][16]
    static_assert(sizeof(uint64_t) * 2 >= 3 * sizeof(int), "flags fit before sbest");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long u_begin = range_start(blockIdx.x, p.units, G);
    const long long u_end = range_start(blockIdx.x + 1, p.units, G);
    const int n_units = static_cast<int>(u_end - u_begin);

    // The producer thread sets up the barriers and starts the first weight
    // copies before the CTA-wide barrier, so DRAM is busy as early as possible.
    const bool producer = (threadIdx.x == kConsumerWarps * 32);
    const uint32_t stage_bytes = C::kWStage + C::kAStage;
    const int n_pre = n_units < C::kStages ? n_units : C::kStages;
    uint64_t pol_w = 0, pol_a = 0;
    int w_rb = 0, w_c = 0, a_c = 0;   // next weight / activation unit to issue
    if (producer) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        last_flag[0] = last_flag[1] = 0;
        fence_mbarrier_init();
        if (n_units > 0) {
            pol_w = policy_evict_first();
            pol_a = policy_evict_last();
            // unit j of this CTA is (row block, K unit) = (rb0, c0) advanced j
            // times along K, wrapping to the next row block
            w_rb = static_cast<int>(u_begin / p.upr);
            w_c = static_cast<int>(u_begin % p.upr);
            a_c = w_c;
            for (int j = 0; j < n_pre; ++j) {
                mbar_arrive_expect_tx(&full[j], stage_bytes);
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sW + j * C::kWStage + ch * kWChunkBytes, &map_w, &full[j], w_c * kUnitK + ch * 128,
                                w_rb * kBM, pol_w);
                if (++w_c == p.upr) {
                    w_c = 0;
                    ++w_rb;
                }
            }
        }
    }
    __syncthreads();
    if (p.pdl) pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_units > 0) {
            auto issue_w = [&](int j) {
                const int s = j % C::kStages;
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sW + s * C::kWStage + ch * kWChunkBytes, &map_w, &full[s], w_c * kUnitK + ch * 128,
                                w_rb * kBM, pol_w);
                if (++w_c == p.upr) {
                    w_c = 0;
                    ++w_rb;
                }
            };
            auto issue_a = [&](int j) {
                const int s = j % C::kStages;
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sA + s * C::kAStage + ch * C::kAChunkBytes, &map_q, &full[s], a_c * kUnitK + ch * 128,
                                0, pol_a);
                if (++a_c == p.upr) a_c = 0;
            };
            // The weights do not depend on the preceding kernel and were
            // started above; the activations only after waiting for it.
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
    const Lane L = lane_setup<MT, kKSplit>(warp, lane);
    const int g = L.g, tq = L.tq, rg = L.rg, kq = L.kq;

    unsigned long long best[MT][2];
#pragma unroll
    for (int t = 0; t < MT; ++t) best[t][0] = best[t][1] = 0ull;

    // activation scales of the tokens this thread's accumulators hold
    float sa_reg[MT][2];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tok = 8 * t + 2 * tq + e;
            sa_reg[t][e] = tok < p.M ? p.s_a[tok] : 0.0f;
        }
    // weight scales of rows g and g + 8 of this warp's row group
    auto load_sw = [&](int rb, float (&sw)[2]) {
        const int n0 = rb * kBM + rg * 16 + g;
        sw[0] = n0 < p.N ? p.s_w[n0] : 0.0f;
        sw[1] = n0 + 8 < p.N ? p.s_w[n0 + 8] : 0.0f;
    };

    // Epilogue of one finished 16-row x (8 * MT)-token tile of this warp.
    auto epilogue = [&](int rb, const int32_t (&v)[MT][4], const float (&sw)[2]) {
        const int n0 = rb * kBM + rg * 16 + g;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = n0 + ((i & 2) ? 8 : 0);
            if (n >= p.N) continue;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int tok = 8 * t + 2 * tq + (i & 1);
                if (tok >= p.M) continue;
                float f = __int2float_rn(v[t][i]);
                f = __fmul_rn(f, sa_reg[t][i & 1]);
                f = __fmul_rn(f, sw[(i & 2) ? 1 : 0]);
                const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                if (p.y) p.y[static_cast<size_t>(tok) * p.N + n] = b;
                if constexpr (ARGMAX) {
                    const unsigned long long key = argmax_key(b, n);
                    if (key > best[t][i & 1]) best[t][i & 1] = key;
                }
            }
        }
    };

    // Row blocks this CTA covers only in part: their partial sums go to the
    // workspace now (fire-and-forget atomics) and are settled after the loop,
    // so the stream of weights never waits on a global round trip.
    int pend_rb[2] = {0, 0}, pend_n[2] = {0, 0};
    int npend = 0;

    int j = 0;
    long long u = u_begin;
    while (u < u_end) {
        const int rb = static_cast<int>(u / p.upr);
        const int c0 = static_cast<int>(u % p.upr);
        const long long left = u_end - u;
        const int nch = (p.upr - c0) < left ? (p.upr - c0) : static_cast<int>(left);
        int32_t v[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t) v[t][0] = v[t][1] = v[t][2] = v[t][3] = 0;
        float sw[2];
        load_sw(rb, sw);   // in flight while the row block's stages stream

        for (int it = 0; it < nch; ++it, ++j) {
            const int s = j % C::kStages;
            if (*abort_flag || !mbar_wait_bounded(&full[s], (j / C::kStages) & 1, abort_flag)) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicExch(p.ws.status, DEV_TIMEOUT);
                }
                continue;
            }
            consume_stage<MT, kKSplit>(smem_u32(sW + s * C::kWStage), smem_u32(sA + s * C::kAStage), C::kAChunkBytes, L, v);
            // every fragment has been consumed by an issued MMA, so the
            // stage's shared memory has been read: hand it back
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // the kKSplit warps of a row group hold partial sums of the same
        // outputs: fold them into the kq == 0 warp through shared memory
        if constexpr (kKSplit > 1) {
            if (kq > 0) {
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        sred[((kq - 1) * kBM + rg * 16 + g + ((i & 2) ? 8 : 0)) * kMaxTok + 8 * t + 2 * tq + (i & 1)] =
                            v[t][i];
            }
            consumer_bar();
            if (kq == 0) {
#pragma unroll
                for (int o = 1; o < kKSplit; ++o)
#pragma unroll
                    for (int t = 0; t < MT; ++t)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            v[t][i] += sred[((o - 1) * kBM + rg * 16 + g + ((i & 2) ? 8 : 0)) * kMaxTok + 8 * t +
                                            2 * tq + (i & 1)];
            }
            consumer_bar();
        }
        if (c0 == 0 && nch == p.upr) {
            if (!*abort_flag && kq == 0) epilogue(rb, v, sw);
        } else {
            if (!*abort_flag && kq == 0) {
                const int slot = unit_owner(static_cast<long long>(rb) * p.upr, p.units, G);
                int32_t *part = p.ws.partial + static_cast<size_t>(slot) * (kBM * kMaxTok);
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = rg * 16 + g + ((i & 2) ? 8 : 0);
                        const int tok = 8 * t + 2 * tq + (i & 1);
                        if (v[t][i] != 0) atomicAdd(&part[r * kMaxTok + tok], v[t][i]);
                    }
            }
            pend_rb[npend] = rb;
            pend_n[npend] = nch;
            ++npend;
        }
        u += nch;
    }

    // ------------------------------------------------ settle split row blocks
    if (npend > 0) {
        consumer_bar();
        if (threadIdx.x == 0) {
            for (int i = 0; i < npend; ++i) {
                int last = 0;
                if (!*abort_flag) {
                    const int slot = unit_owner(static_cast<long long>(pend_rb[i]) * p.upr, p.units, G);
                    const int old = atom_add_acq_rel_gpu(&p.ws.rb_counter[slot], pend_n[i]);
                    last = (old + pend_n[i] == p.upr);
                    if (last) atomicExch(&p.ws.rb_counter[slot], 0);
                }
                last_flag[i] = last;
            }
        }
        consumer_bar();
        for (int i = 0; i < npend; ++i) {
            if (!last_flag[i] || kq != 0) continue;
            const int slot = unit_owner(static_cast<long long>(pend_rb[i]) * p.upr, p.units, G);
            int32_t *part = p.ws.partial + static_cast<size_t>(slot) * (kBM * kMaxTok);
            int32_t v[MT][4];
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = rg * 16 + g + ((k & 2) ? 8 : 0);
                    const int tok = 8 * t + 2 * tq + (k & 1);
                    v[t][k] = atomicExch(&part[r * kMaxTok + tok], 0);
                }
            float swp[2];
            load_sw(pend_rb[i], swp);
            epilogue(pend_rb[i], v, swp);
        }
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
