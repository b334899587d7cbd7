// Tiled W8A8 kernel for prefill-sized batches (M > 16) with both operands fed
// by TMA: the same exact int32 contraction and per-element epilogue as the
// weight-streaming kernel, so every row matches it bitwise.
//
// sm_103a's tcgen05.mma has no int8 kind.  A first pass (expand_f16_kernel)
// writes exact f16 copies of the int8 codes and weights into the workspace;
// the tensor cores then multiply them with kind::f16 MMAs into fp32
// accumulators in tensor memory (TMEM).  Every product is an integer of
// magnitude <= 127^2, so the fp32 sum of a 1024-wide K chunk (<= 2^24) is
// exact; it is moved into an int32 total before it could grow past that.
//
// Compared with converting the codes inside the tile loop (k_prefill.cu), no
// thread stores operands into shared memory: TMA writes them and the tensor
// core reads them, and the SM's load/store pipe stays free.
//
// CTA tile: 128 tokens (MMA M = TMEM lanes) x 256 weight rows (MMA N), 64 K
// per stage, one CTA per SM, persistent.  Two fp32 accumulators of 256 TMEM
// columns alternate from one 1024-K chunk to the next, so the tensor core
// starts a chunk while the previous one is moved out.  Roles:
//   warp 0     lane 0 issues the TMA loads of both operands into a 4-stage
//              ring;
//   warp 1     allocates TMEM; lane 0 issues the MMAs and commits them;
//   warps 2-9  (TMEM lane quarter = warp % 4, column half = (warp - 2) / 4)
//              one token row and 128 of the tile's 256 weight columns per
//              thread: add each chunk's sums into int32 totals held in
//              registers, then the epilogue bf16_rne((float(acc) * s_a) *
//              s_w).
// The work of a CTA is a list of items: whole tiles (b, b + G, ...; tiles are
// numbered token tile fastest, so the CTAs running together share weight
// tiles in L2), then, when the last wave would be at most half full, one K
// half of one of its tiles.  The kernel is then launched in clusters of two
// CTAs (as many pairs as fit at once), the two halves of a tile run on the
// two CTAs of a pair, and their int32 sums meet in distributed shared memory:
// each CTA owns every other group of 8 columns, receives its partner's sums of
// those groups, adds them to its own and applies the epilogue.  Integer sums
// are exact in any order, so the bits do not depend on the split.  (Partial
// sums exchanged through global memory instead made the kernel's completion
// markedly slower on this GPU.)
// Every mbarrier wait is bounded: on a timeout the kernel writes DEV_TIMEOUT
// to the workspace status word and every role returns.  The two cluster
// barriers of a pair are then still reached by every thread of both CTAs (no
// role returns early), so a timeout cannot leave a partner waiting.
#include "kernels.cuh"
#include "ptx.cuh"
#include "tc.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kTileM = 128;                       // tokens per tile: MMA M, TMEM lanes
constexpr int kTileN = 256;                       // weight rows per tile: MMA N
constexpr int kStepK = 64;                        // K per stage: one 128-byte f16 row
constexpr int kStages = 4;
constexpr int kChunkSteps = 16;                   // 1024 K per exact fp32 chunk
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;   // 320
constexpr int kCols = kTileN / 2;                 // weight columns per epilogue thread
constexpr int kStageA = kTileM * 128;             // 16 KB of f16 tokens
constexpr int kStageB = kTileN * 128;             // 32 KB of f16 weights
constexpr int kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 512;               // two fp32 accumulators of 256 columns
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 256;

static_assert(kChunkSteps * kStepK * 127 * 127 <= (1 << 24), "chunk sums must stay exact in fp32");

struct Params {
    const float *s_a;
    const float *s_w;
    uint16_t *y;         // [M, N] bf16
    int M, N;
    int kt;              // K steps
    int vec_y;           // y rows allow 16-byte stores
    int tiles_m;         // token tiles (tile t: token tile t % tiles_m, weight tile t / tiles_m)
    int whole;           // tiles 0 .. whole - 1 run whole
    int tail_items;      // 2 * (tiles - whole): K halves, one per CTA 0 .. tail_items - 1 (clusters of 2)
    Workspace ws;
};

// One item of a CTA's list: a tile and its range of K steps.
struct Item {
    int tile;
    int kb, nsteps;
};

// Items of CTA b out of G: whole tiles b, b + G, ... below p.whole, then at
// most one K half of a later tile (tile whole + b / 2, half b % 2 = the CTA's
// rank in its cluster).
__device__ __forceinline__ int item_count(const Params &p, int b, int G)
{
    const int n_whole = b < p.whole ? (p.whole - 1 - b) / G + 1 : 0;
    return n_whole + (b < p.tail_items ? 1 : 0);
}

__device__ __forceinline__ Item item_at(const Params &p, int b, int G, int i)
{
    Item it;
    const int n_whole = b < p.whole ? (p.whole - 1 - b) / G + 1 : 0;
    if (i < n_whole) {
        it.tile = b + i * G;
        it.kb = 0;
        it.nsteps = p.kt;
    } else {
        it.tile = p.whole + (b >> 1);
        it.kb = (b & 1) ? p.kt / 2 : 0;
        it.nsteps = (b & 1) ? p.kt - p.kt / 2 : p.kt / 2;
    }
    return it;
}

// int8 -> f16 copies of q [M, K] and w [N, K] (same layout, exact values).
// A warp converts 512 codes per iteration: lane l loads 8 bytes at 8 l and at
// 256 + 8 l and stores their 16 f16 values as two 16-byte chunks, so every
// load covers 256 contiguous bytes and every store 512.  Each thread keeps
// kExpandAhead iterations' loads in flight; the grid is one wave.
constexpr int kExpandThreads = 256;
constexpr int kExpandAhead = 4;

// 16-byte store with an L2 evict-last policy: the copies are read by the
// GEMM right after, so they should stay in L2.
__device__ __forceinline__ void st_keep_l2(void *p, uint4 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ uint4 i8x8_to_f16x8(uint2 v)
{
    uint4 r;
    i8x4_to_f16x2x2(v.x, r.x, r.y);
    i8x4_to_f16x2x2(v.y, r.z, r.w);
    return r;
}

__global__ void __launch_bounds__(kExpandThreads) expand_f16_kernel(const int8_t *__restrict__ q,
                                                                    uint16_t *__restrict__ qf, long long nq,
                                                                    const int8_t *__restrict__ w,
                                                                    uint16_t *__restrict__ wf, long long nw, int pdl)
{
    if (pdl) pdl_wait();
    const int lane = threadIdx.x & 31;
    const uint64_t keep = policy_evict_last();
    const long long total = nq + nw;   // 512-code blocks: of q, then of w
    const long long nwarps = static_cast<long long>(gridDim.x) * (kExpandThreads / 32);
    long long blk = static_cast<long long>(blockIdx.x) * (kExpandThreads / 32) + (threadIdx.x >> 5);
    for (; blk < total; blk += kExpandAhead * nwarps) {
        uint2 v[kExpandAhead][2];
#pragma unroll
        for (int u = 0; u < kExpandAhead; ++u) {
            const long long c = blk + u * nwarps;
            if (c < total) {
                const int8_t *src = (c < nq ? q + 512 * c : w + 512 * (c - nq)) + 8 * lane;
                v[u][0] = __ldcs(reinterpret_cast<const uint2 *>(src));
                v[u][1] = __ldcs(reinterpret_cast<const uint2 *>(src + 256));
            }
        }
#pragma unroll
        for (int u = 0; u < kExpandAhead; ++u) {
            const long long c = blk + u * nwarps;
            if (c >= total) break;
            uint16_t *dst = (c < nq ? qf + 512 * c : wf + 512 * (c - nq)) + 8 * lane;
            st_keep_l2(dst, i8x8_to_f16x8(v[u][0]), keep);
            st_keep_l2(dst + 256, i8x8_to_f16x8(v[u][1]), keep);
        }
    }
    pdl_launch_dependents();
}

// The codes after the last whole 512-code block of q (block 0) and of w
// (block 1): fewer than 512, a multiple of 16.
__global__ void __launch_bounds__(32) expand_tail_kernel(const int8_t *q, uint16_t *qf, int nq, const int8_t *w,
                                                         uint16_t *wf, int nw)
{
    pdl_wait();
    const int8_t *src = blockIdx.x == 0 ? q : w;
    uint16_t *dst = blockIdx.x == 0 ? qf : wf;
    const int n = blockIdx.x == 0 ? nq : nw;
    for (int i = 16 * threadIdx.x; i < n; i += 16 * 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src + i);
        *reinterpret_cast<uint4 *>(dst + i) = i8x8_to_f16x8(make_uint2(v.x, v.y));
        *reinterpret_cast<uint4 *>(dst + i + 8) = i8x8_to_f16x8(make_uint2(v.z, v.w));
    }
    pdl_launch_dependents();
}

// bf16_rne((float(acc) * s_a) * s_w) of 8 columns of a token row, stored at
// y[n .. n + 7] (ragged at the end of the row).  Eight at a time keeps the
// temporaries small beside the 128 int32 totals each thread holds.
__device__ __forceinline__ void store_y8(uint16_t *yr, int n, int N, bool vec, float sa, const float *s_w,
                                         const int32_t *acc)
{
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        uint32_t b2 = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float sw = (n + e + h < N) ? __ldg(s_w + n + e + h) : 0.0f;
            float f = __int2float_rn(acc[e + h]);
            f = __fmul_rn(f, sa);
            f = __fmul_rn(f, sw);
            b2 |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f))) << (16 * h);
        }
        o[e >> 1] = b2;
    }
    if (vec && n + 8 <= N) {
        *reinterpret_cast<uint4 *>(yr + n) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (n + e < N) yr[n + e] = static_cast<uint16_t>(o[e >> 1] >> (16 * (e & 1)));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tma_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);   // TMA landed
    uint64_t *empty = full + kStages;                                             // MMA done reading
    uint64_t *acc_full = empty + kStages;                                         // [2] chunk sum ready
    uint64_t *acc_empty = acc_full + 2;                                           // [2] chunk sum moved out
    uint64_t *drain = acc_empty + 2;                                              // all MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int nitems = item_count(p, b, G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);                // producer's expect_tx arrival + bytes
            mbar_init(&empty[s], 1);               // MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);            // MMA commit
            mbar_init(&acc_empty[a], kEpiWarps);   // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            atomicExch(p.ws.status, DEV_TIMEOUT);
        }
    };

    // a CTA with a K half (clusters of two): both CTAs of the pair meet in two
    // cluster barriers after their roles, every thread of each (see below)
    const bool pair = b < p.tail_items;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&map_a);
            prefetch_tensormap(&map_b);
            const uint64_t pol_a = policy_evict_last();    // token tile: reused by every weight tile
            const uint64_t pol_b = policy_evict_first();   // weight tile: read by the CTAs running together
            pdl_wait();   // the f16 copies come from the preceding expand pass
            long long j = 0;
            bool ok = true;
            for (int i = 0; ok && i < nitems; ++i) {
                const Item it = item_at(p, b, G, i);
                const int m0 = (it.tile % p.tiles_m) * kTileM;
                const int n0 = (it.tile / p.tiles_m) * kTileN;
                for (int st = 0; st < it.nsteps; ++st, ++j) {
                    const int s = static_cast<int>(j % kStages);
                    if (j >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / kStages) - 1) & 1u,
                                                           abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    const int k = (it.kb + st) * kStepK;
                    tma_load_2d(sa, &map_a, &full[s], k, m0, pol_a);
                    tma_load_2d(sa + kStageA, &map_b, &full[s], k, n0, pol_b);
                }
            }
            // let every issued copy land before the CTA can exit
            volatile int never = 0;
            for (long long jj = j > kStages ? j - kStages : 0; jj < j; ++jj)
                mbar_wait_bounded(&full[jj % kStages], static_cast<uint32_t>(jj / kStages) & 1u, &never);
        }
        __syncwarp();
        if (pair) {
            cluster_sync_all();
            cluster_sync_all();
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        long long j = 0, c = 0;
        bool ok = true;
        for (int i = 0; ok && i < nitems; ++i) {
            const Item it = item_at(p, b, G, i);
            const uint32_t idesc = tc::idesc_f16_f32(kTileM, kTileN);
            const int nch = (it.nsteps + kChunkSteps - 1) / kChunkSteps;
            for (int ch = 0; ok && ch < nch; ++ch, ++c) {
                const int acc = static_cast<int>(c & 1);
                if (c >= 2) {
                    // the chunk before last left this accumulator (all epilogue warps)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[acc],
                                                                   static_cast<uint32_t>((c >> 1) - 1) & 1u, abort_flag));
                    if (!ok) break;
                    tc::fence_after();
                }
                const int s0 = ch * kChunkSteps, s1 = min(it.nsteps, s0 + kChunkSteps);
                for (int st = s0; st < s1; ++st, ++j) {
                    const int s = static_cast<int>(j % kStages);
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait_bounded(&full[s], static_cast<uint32_t>(j / kStages) & 1u, abort_flag));
                    if (!ok) break;
                    tc::fence_after();
                    if (lane == 0) {
                        const uint32_t a0 = smem_u32(smem + s * kStageBytes);
                        const uint32_t b0 = a0 + kStageA;
#pragma unroll
                        for (int k = 0; k < kStepK / 16; ++k)
                            tc::mma_f16_ss(tmem + acc * kTileN, tc::sdesc_kmajor_sw128(a0 + 32 * k),
                                           tc::sdesc_kmajor_sw128(b0 + 32 * k), idesc, (st > s0 || k > 0) ? 1u : 0u);
                        tc::commit(&empty[s]);
                        if (st == s1 - 1) tc::commit(&acc_full[acc]);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok) fail();
        // nothing may still read shared memory or write TMEM when the CTA
        // frees them
        tc::fence_before();
        if (lane == 0) tc::commit(drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait_bounded(drain, 0, &never);
        __syncwarp();
        if (pair) {
            cluster_sync_all();
            cluster_sync_all();
        }
    } else {
        // ------------------------------------------------ chunk moves and epilogue
        // one token row and the column half `half` (128 columns) per thread
        const int qd = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int row = 32 * qd + lane;
        int32_t tot[kCols];
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16) + half * kCols;
        long long c = 0;
        pdl_wait();   // scales and outputs follow the kernels before
        for (int i = 0; i < nitems; ++i) {
            const Item it = item_at(p, b, G, i);
            const int m0 = (it.tile % p.tiles_m) * kTileM;
            const int n0 = (it.tile / p.tiles_m) * kTileN + half * kCols;
            const int nch = (it.nsteps + kChunkSteps - 1) / kChunkSteps;
            bool ok = true;
            for (int ch = 0; ch < nch; ++ch, ++c) {
                const int acc = static_cast<int>(c & 1);
                // warp-uniform: the TMEM loads below are warp-collective
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&acc_full[acc], static_cast<uint32_t>(c >> 1) & 1u, abort_flag))) {
                    fail();
                    ok = false;
                    break;
                }
                tc::fence_after();
#pragma unroll
                for (int g = 0; g < kCols / 16; ++g) {
                    uint32_t d[16];
                    tc::ld16(lane_addr + acc * kTileN + 16 * g, d);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int32_t v = f2i_exact(__uint_as_float(d[e]));
                        tot[16 * g + e] = ch > 0 ? tot[16 * g + e] + v : v;
                    }
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[acc]);
            }
            if (!ok) break;
            if (it.nsteps < p.kt) break;   // a K half: finished below, with the partner's sums
            const int tok = m0 + row;
            if (tok < p.M) {
                const float sa = p.s_a[tok];
                uint16_t *yr = p.y + static_cast<size_t>(tok) * p.N;
#pragma unroll
                for (int g = 0; g < kCols / 8; ++g)
                    store_y8(yr, n0 + 8 * g, p.N, p.vec_y != 0, sa, p.s_w, tot + 8 * g);
            }
        }
        if (pair) {
        // The two K halves of a tile meet in distributed shared memory (both
        // CTAs of the pair take this branch).  Column group g (8 columns)
        // belongs to rank g % 2.  The ring is free once both CTAs have passed
        // the first barrier (their copies landed, their MMAs drained); each
        // then writes the groups it does not own into its partner's ring, and
        // after the second barrier each adds them to its own and stores.
        const int r = b & 1;
        const uint32_t recv = smem_u32(smem);              // [16 groups][128 rows][8] int32
        __syncwarp();
        cluster_sync_all();
        {
#pragma unroll
            for (int j = 0; j < kCols / 8; ++j) {
                const int g = half * (kCols / 8) + j;
                if ((g & 1) == r) continue;
                const uint32_t dst = cluster_map(recv + static_cast<uint32_t>(((g >> 1) * kTileM + row) * 32), r ^ 1);
                st_cluster_v4(dst, tot[8 * j], tot[8 * j + 1], tot[8 * j + 2], tot[8 * j + 3]);
                st_cluster_v4(dst + 16, tot[8 * j + 4], tot[8 * j + 5], tot[8 * j + 6], tot[8 * j + 7]);
            }
        }
        cluster_sync_all();
        if (!*abort_flag) {
            const Item it = item_at(p, b, G, nitems - 1);
            const int tok = (it.tile % p.tiles_m) * kTileM + row;
            const int n0 = (it.tile / p.tiles_m) * kTileN + half * kCols;
            if (tok < p.M) {
                const float sa = p.s_a[tok];
                uint16_t *yr = p.y + static_cast<size_t>(tok) * p.N;
#pragma unroll
                for (int j = 0; j < kCols / 8; ++j) {
                    const int g = half * (kCols / 8) + j;
                    if ((g & 1) != r) continue;
                    const int4 *src = reinterpret_cast<const int4 *>(smem + ((g >> 1) * kTileM + row) * 32);
                    const int4 x0 = src[0], x1 = src[1];
                    int32_t v[8] = {tot[8 * j] + x0.x,     tot[8 * j + 1] + x0.y, tot[8 * j + 2] + x0.z,
                                    tot[8 * j + 3] + x0.w, tot[8 * j + 4] + x1.x, tot[8 * j + 5] + x1.y,
                                    tot[8 * j + 6] + x1.z, tot[8 * j + 7] + x1.w};
                    store_y8(yr, n0 + 8 * j, p.N, p.vec_y != 0, sa, p.s_w, v);
                }
            }
        }
    }
    }
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_tma(const PrefillTmaArgs &a, cudaStream_t stream)
{
    static bool attr_set = false;
    static int sms = 0;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    // the f16 copies: 512-code blocks of q, then of w (sizes are multiples of
    // 16 codes; a ragged last block is copied by the tail launch below)
    {
        const long long cq = static_cast<long long>(a.M) * a.K, cw = static_cast<long long>(a.N) * a.K;
        cudaLaunchConfig_t cfg = {};
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, expand_f16_kernel, kExpandThreads, 0);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(static_cast<unsigned>(sms * (per_sm > 0 ? per_sm : 1)));
        cfg.blockDim = dim3(kExpandThreads);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = a.pdl ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, expand_f16_kernel, a.q, a.qf, cq / 512, a.w_q, a.wf, cw / 512, a.pdl ? 1 : 0);
        if (e != cudaSuccess) return e;
        if ((cq | cw) % 512 != 0) {
            // the last partial blocks, 16 codes per thread
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(32);
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, expand_tail_kernel, a.q + cq / 512 * 512, a.qf + cq / 512 * 512,
                                   static_cast<int>(cq % 512), a.w_q + cw / 512 * 512, a.wf + cw / 512 * 512,
                                   static_cast<int>(cw % 512));
            if (e != cudaSuccess) return e;
        }
    }

    Params p;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.y = a.y;
    p.M = a.M;
    p.N = a.N;
    p.kt = (a.K + kStepK - 1) / kStepK;
    p.vec_y = ((a.N % 8) == 0 && (reinterpret_cast<uintptr_t>(a.y) & 15u) == 0) ? 1 : 0;
    p.ws = a.ws;
    p.tiles_m = (a.M + kTileM - 1) / kTileM;
    const int tiles = p.tiles_m * ((a.N + kTileN - 1) / kTileN);
    p.whole = tiles;
    p.tail_items = 0;
    // One CTA per SM, all tiles whole; or, when the last wave would be at
    // most half full, clusters of two CTAs (as many pairs as fit on the GPU at
    // once) with the last wave's tiles split into K halves, one per CTA.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute lattr[2];
    lattr[0] = attr[0];   // a programmatic dependent of the expand pass (its TMA waits for it)
    lattr[1].id = cudaLaunchAttributeClusterDimension;
    lattr[1].val.clusterDim.x = 2;
    lattr[1].val.clusterDim.y = 1;
    lattr[1].val.clusterDim.z = 1;
    cfg.attrs = lattr;
    int grid = tiles < sms ? tiles : sms;
    if (tiles % sms != 0 && p.kt >= 16) {
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(static_cast<unsigned>(sms));
        int pairs = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&pairs, prefill_tma_kernel, &cfg);
        if (e != cudaSuccess) return e;
        const int g2 = 2 * pairs;
        const int rem = g2 > 0 ? tiles % g2 : 0;
        if (g2 > 0 && rem > 0 && 2 * rem <= g2) {
            p.whole = tiles - rem;
            p.tail_items = 2 * rem;
            grid = p.whole > 0 ? g2 : p.tail_items;
        }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.numAttrs = p.tail_items > 0 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, prefill_tma_kernel, a.map_a, a.map_b, p);
}

}  // namespace bi
