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
//              one token row and half of the item's weight columns (at
//              most 128) per thread: add each chunk's sums into int32
//              totals held in registers, then the epilogue
//              bf16_rne((float(acc) * s_a) * s_w).
// The work of a CTA is a list of items: whole tiles (b, b + G, ...; tiles are
// numbered token tile fastest, so the CTAs running together share weight
// tiles in L2), then, when the last wave would be at most half full, one
// slice of its tiles: the tile's 256 weight rows cut into slices of `tail_w`
// rows (a multiple of 32), each run over the whole K by its own CTA with an
// MMA of N = its width.  A slice needs no partial sums from other CTAs: on
// this GPU, split-K partials exchanged through global memory made the
// kernel's completion markedly slower (its written bytes are flushed at the
// end).
// Every wait is bounded: on a timeout the kernel writes DEV_TIMEOUT to the
// workspace status word and every role returns.
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
    int tail_w;          // later tiles run as slices of tail_w weight rows (multiple of 32)
    int slices;          // ceil(256 / tail_w)
    int tail_items;      // (tiles - whole) * slices: one per CTA 0 .. tail_items - 1
    Workspace ws;
};

// One item of a CTA's list: a tile and the slice of its 256 weight rows.
struct Item {
    int tile;
    int c0, cw;          // weight rows c0 .. c0 + cw - 1 of the tile (cw a multiple of 32)
};

// Items of CTA b out of G: whole tiles b, b + G, ... below p.whole, then at
// most one slice of a later tile (slice b of the (tiles - whole) * slices).
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
        it.c0 = 0;
        it.cw = kTileN;
    } else {
        it.tile = p.whole + b / p.slices;
        it.c0 = (b % p.slices) * p.tail_w;
        it.cw = min(p.tail_w, kTileN - it.c0);
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
            *reinterpret_cast<uint4 *>(dst) = i8x8_to_f16x8(v[u][0]);
            *reinterpret_cast<uint4 *>(dst + 256) = i8x8_to_f16x8(v[u][1]);
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
    prefill_tma_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_bs, Params p)
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&map_a);
            prefetch_tensormap(&map_b);
            if (p.tail_items > 0) prefetch_tensormap(&map_bs);
            const uint64_t pol_a = policy_evict_last();    // token tile: reused by every weight tile
            const uint64_t pol_b = policy_evict_first();   // weight tile: read by the CTAs running together
            pdl_wait();   // the f16 copies come from the preceding expand pass
            long long j = 0;
            bool ok = true;
            for (int i = 0; ok && i < nitems; ++i) {
                const Item it = item_at(p, b, G, i);
                const int m0 = (it.tile % p.tiles_m) * kTileM;
                const int n0 = (it.tile / p.tiles_m) * kTileN + it.c0;
                for (int st = 0; st < p.kt; ++st, ++j) {
                    const int s = static_cast<int>(j % kStages);
                    if (j >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((j / kStages) - 1) & 1u,
                                                           abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], kStageA + it.cw * 128);
                    const int k = st * kStepK;
                    tma_load_2d(sa, &map_a, &full[s], k, m0, pol_a);
                    if (it.cw == kTileN) {
                        tma_load_2d(sa + kStageA, &map_b, &full[s], k, n0, pol_b);
                    } else {
                        for (int r = 0; r < it.cw; r += 32)   // a slice: boxes of 32 weight rows
                            tma_load_2d(sa + kStageA + r * 128, &map_bs, &full[s], k, n0 + r, pol_b);
                    }
                }
            }
            // let every issued copy land before the CTA can exit
            volatile int never = 0;
            for (long long jj = j > kStages ? j - kStages : 0; jj < j; ++jj)
                mbar_wait_bounded(&full[jj % kStages], static_cast<uint32_t>(jj / kStages) & 1u, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        long long j = 0, c = 0;
        bool ok = true;
        for (int i = 0; ok && i < nitems; ++i) {
            const Item it = item_at(p, b, G, i);
            const uint32_t idesc = tc::idesc_f16_f32(kTileM, it.cw);
            const int nch = (p.kt + kChunkSteps - 1) / kChunkSteps;
            for (int ch = 0; ok && ch < nch; ++ch, ++c) {
                const int acc = static_cast<int>(c & 1);
                if (c >= 2) {
                    // the chunk before last left this accumulator (all epilogue warps)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[acc],
                                                                   static_cast<uint32_t>((c >> 1) - 1) & 1u, abort_flag));
                    if (!ok) break;
                    tc::fence_after();
                }
                const int s0 = ch * kChunkSteps, s1 = min(p.kt, s0 + kChunkSteps);
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
    } else {
        // ------------------------------------------------ chunk moves and epilogue
        // thread: token row `row` of the tile, the item's weight rows
        // c0 + half * cw / 2 .. + cw / 2 - 1 (at most 128: kCols)
        const int qd = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int row = 32 * qd + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        const int nch = (p.kt + kChunkSteps - 1) / kChunkSteps;
        long long c = 0;
        int32_t tot[kCols];
        pdl_wait();   // scales and outputs follow the kernels before
        for (int i = 0; i < nitems; ++i) {
            const Item it = item_at(p, b, G, i);
            const int m0 = (it.tile % p.tiles_m) * kTileM;
            const int hw = it.cw >> 1;                    // columns per half: a multiple of 16
            const int col = half * hw;                    // first accumulator column of this thread
            const int n0 = (it.tile / p.tiles_m) * kTileN + it.c0 + col;
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
                    if (16 * g < hw) {
                        uint32_t d[16];
                        tc::ld16(lane_addr + acc * kTileN + col + 16 * g, d);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int32_t v = f2i_exact(__uint_as_float(d[e]));
                            tot[16 * g + e] = ch > 0 ? tot[16 * g + e] + v : v;
                        }
                    }
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[acc]);
            }
            if (!ok) break;
            const int tok = m0 + row;
            if (tok < p.M) {
                const float sa = p.s_a[tok];
                uint16_t *yr = p.y + static_cast<size_t>(tok) * p.N;
#pragma unroll
                for (int g = 0; g < kCols / 8; ++g)
                    if (8 * g < hw) store_y8(yr, n0 + 8 * g, p.N, p.vec_y != 0, sa, p.s_w, tot + 8 * g);
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
    p.tail_w = kTileN;
    p.slices = 1;
    p.tail_items = 0;
    // One CTA per SM.  Tiles that fill whole waves run whole; when the last
    // wave would be at most half full, its tiles run as slices of the
    // narrowest width (a multiple of 32 rows) whose slices all fit in it.
    int grid = tiles < sms ? tiles : sms;
    const int rem = tiles % sms;
    if (rem > 0 && rem <= sms / 2) {
        int w = 32;
        while (w < kTileN && rem * ((kTileN + w - 1) / w) > sms) w += 32;
        if (w < kTileN) {
            p.whole = tiles - rem;
            p.tail_w = w;
            p.slices = (kTileN + w - 1) / w;
            p.tail_items = rem * p.slices;
            grid = p.whole > 0 ? sms : p.tail_items;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;   // a programmatic dependent of the expand pass (its TMA waits for it)
    return cudaLaunchKernelEx(&cfg, prefill_tma_kernel, a.map_a, a.map_b, a.map_bs, p);
}

}  // namespace bi
