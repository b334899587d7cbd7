// Tiled W8A8 kernel for prefill-sized batches (M > 16) on the tcgen05 tensor
// cores: a dense int8 contraction with exact int32 results and the same
// per-element epilogue as the weight-streaming kernel, so every row matches
// it bitwise.
//
// sm_103a's tcgen05.mma has no int8 kind, so the int8 codes are converted
// exactly to f16 and multiplied by kind::f16 MMAs into fp32 accumulators in
// tensor memory (TMEM).  Every product is an integer of magnitude <= 128^2,
// so an fp32 sum of at most 1024 of them (<= 2^24) is exact; the fp32 sum of
// each 1024-wide K chunk is moved into an int32 total, kept in the other half
// of TMEM, before the next chunk starts.
//
// CTA tile: 128 tokens (MMA M = TMEM lanes) x 256 weight rows (MMA N = TMEM
// columns), 64 K per stage, one CTA per SM.  Roles:
//   warps 0-7   load the tile's int8 rows from global memory four stages
//               ahead (two in split tiles) into registers, convert them to
//               f16, store them into a ring of K-major, 128-byte-swizzled
//               stages and arrive on the stage's barrier (one arrival per
//               warp);
//   warps 8-11  TMEM lane quarters 0-3: move chunk sums into the int32
//               totals, then the epilogue, one token row per thread; warp 8
//               also allocates TMEM, and its lane 0 issues the MMAs and
//               commits them (the MMAs of a chunk wait for the previous
//               chunk's move in any case).
// Loading through registers rather than TMA keeps the int8 bytes out of
// shared memory, whose bandwidth the MMA operands and the f16 stores share.
//
// Tiles that fill whole waves run whole (prefill_kernel<false>).  When the
// last wave would be at most half full, its tiles run in a second launch
// (prefill_kernel<true>), each split along K into ranges whose int32 sums
// meet in workspace slots; the range that arrives last adds them and applies
// the epilogue.  Integer sums are exact in any order, so the bits do not
// depend on the split.
// Every wait is bounded: on a timeout the kernel writes DEV_TIMEOUT to the
// workspace status word and every role returns.
#include "kernels.cuh"
#include "ptx.cuh"
#include "tc.cuh"

#include <cuda_bf16.h>

namespace bi {

namespace {

constexpr int kTileM = 128;                       // tokens per tile: MMA M, TMEM lanes
constexpr int kTileN = 256;                       // weight rows per tile: MMA N, TMEM columns
constexpr int kStepK = 64;                        // K per stage: one 128-byte f16 row
constexpr int kStages = 4;
constexpr int kChunkSteps = 16;                   // 1024 K per exact fp32 chunk
constexpr int kConvWarps = 8;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiWarp0 = kConvWarps;             // warps 8 .. 11 (warp % 4 = lane quarter)
constexpr int kThreads = (kEpiWarp0 + 4) * 32;    // 384: three warps per scheduler
constexpr int kStageA = kTileM * 128;             // 16 KB of f16 tokens
constexpr int kStageB = kTileN * 128;             // 32 KB of f16 weights
constexpr int kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 512;               // [0, 256) fp32 chunk sums, [256, 512) int32 totals
constexpr uint32_t kTotCol = 256;
constexpr int kChunksA = kTileM * 4 / kConvThreads;   // 16-byte int8 chunks per thread and stage: 2
constexpr int kChunksB = kTileN * 4 / kConvThreads;   // 4
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kTileN * 4 + 256;

static_assert(kTileM * 4 % kConvThreads == 0 && kTileN * 4 % kConvThreads == 0, "converter split");
static_assert(kChunkSteps * kStepK * 128 * 128 <= (1 << 24), "chunk sums must stay exact in fp32");

struct Params {
    const int8_t *q;     // [M, K]
    const int8_t *w;     // [N, K]
    const float *s_a;
    const float *s_w;
    uint16_t *y;         // [M, N] bf16
    int M, N, K;
    int kt;              // K steps
    int vec_y;           // y rows allow 16-byte stores
    int tiles_m;         // token tiles (tile t: token tile t % tiles_m, weight tile t / tiles_m)
    int full_tiles;      // tiles 0 .. full_tiles - 1 run whole, one per CTA
    int parts;           // every later tile runs as `parts` K ranges, one per CTA
    int32_t *tail_acc;   // per split tile: parts - 1 slots of int32 [256 columns][128 rows] (scratch)
    int *tail_cnt;       // per split tile: arrivals and K ranges stored, zero between calls
    Workspace ws;
    int pdl;
};

// 16 int8 values -> 16 f16 values, stored as two 16-byte chunks (2c, 2c + 1)
// of a 128-byte swizzled row.
__device__ __forceinline__ void store_f16_row(uint8_t *row_base, int row, int c, uint4 v)
{
    uint32_t h[8];
    i8x4_to_f16x2x2(v.x, h[0], h[1]);
    i8x4_to_f16x2x2(v.y, h[2], h[3]);
    i8x4_to_f16x2x2(v.z, h[4], h[5]);
    i8x4_to_f16x2x2(v.w, h[6], h[7]);
    const int sw = row & 7;
    *reinterpret_cast<uint4 *>(row_base + (((2 * c) ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(row_base + (((2 * c + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
}

// kSplit = false: tiles 0 .. full_tiles - 1, whole.  kSplit = true: the
// later tiles, each as `parts` K ranges (one CTA per range), launched after.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sw_tile = reinterpret_cast<float *>(smem + kStages * kStageBytes);     // [kTileN]
    uint64_t *full = reinterpret_cast<uint64_t *>(sw_tile + kTileN);             // converters -> MMA
    uint64_t *empty = full + kStages;                                             // MMA done reading
    uint64_t *acc_full = empty + kStages;                                         // chunk sum ready
    uint64_t *acc_empty = acc_full + 1;                                           // chunk sum moved
    uint64_t *drain = acc_empty + 1;                                              // all MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_part = abort_flag + 1;                                     // split tile: arrival ticket

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's tile and K range: whole tiles first, then the split tiles'
    // ranges (tiles are numbered token tile fastest, so the CTAs resident
    // together share weight tiles in L2)
    int tile = static_cast<int>(blockIdx.x), part = 0, parts = 1;
    if constexpr (kSplit) {
        tile = p.full_tiles + static_cast<int>(blockIdx.x) / p.parts;
        part = static_cast<int>(blockIdx.x) % p.parts;
        parts = p.parts;
    }
    const int m0 = (tile % p.tiles_m) * kTileM;
    const int n0 = (tile / p.tiles_m) * kTileN;
    const int kb = static_cast<int>(static_cast<long long>(p.kt) * part / parts);   // first K step
    const int nsteps = static_cast<int>(static_cast<long long>(p.kt) * (part + 1) / parts) - kb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kConvWarps);       // one arrival per converter warp
            mbar_init(&empty[s], 1);               // MMA commit
        }
        mbar_init(acc_full, 1);                    // MMA commit
        mbar_init(acc_empty, 4);                   // the four epilogue warps
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kEpiWarp0) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    if (p.pdl) pdl_launch_dependents();

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            atomicExch(p.ws.status, DEV_TIMEOUT);
        }
    };

    if (warp < kConvWarps) {
        // ------------------------------------------------ int8 -> f16 stages
        // (the split tiles' epilogue needs registers: fewer loads in flight)
        constexpr int kAhead = kSplit ? 2 : 4;
        const int t = threadIdx.x;
        const int c = t & 3;        // 16-byte chunk of the 64-byte int8 row slice
        const int r0 = t >> 2;      // rows r0 + 64 i
        if (p.pdl) pdl_wait();
        auto load = [&](int j, uint4 (&ra)[kChunksA], uint4 (&rb)[kChunksB]) {
            const int k = (kb + j) * kStepK + 16 * c;
            const bool kin = k < p.K;
#pragma unroll
            for (int i = 0; i < kChunksA; ++i) {
                const int tok = m0 + r0 + 64 * i;
                ra[i] = (kin && tok < p.M)
                            ? __ldg(reinterpret_cast<const uint4 *>(p.q + static_cast<size_t>(tok) * p.K + k))
                            : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < kChunksB; ++i) {
                const int n = n0 + r0 + 64 * i;
                rb[i] = (kin && n < p.N)
                            ? __ldg(reinterpret_cast<const uint4 *>(p.w + static_cast<size_t>(n) * p.K + k))
                            : make_uint4(0, 0, 0, 0);
            }
        };
        auto step = [&](int j, uint4 (&ra)[kChunksA], uint4 (&rb)[kChunksB]) -> bool {
            const int s = j % kStages;
            if (j >= kStages && !mbar_wait_bounded(&empty[s], ((j / kStages) - 1) & 1, abort_flag)) {
                fail();
                return false;
            }
            uint8_t *sa = smem + s * kStageBytes;
            uint8_t *sb = sa + kStageA;
#pragma unroll
            for (int i = 0; i < kChunksA; ++i) store_f16_row(sa + (r0 + 64 * i) * 128, r0 + 64 * i, c, ra[i]);
#pragma unroll
            for (int i = 0; i < kChunksB; ++i) store_f16_row(sb + (r0 + 64 * i) * 128, r0 + 64 * i, c, rb[i]);
            fence_proxy_async_smem();   // the tensor core reads the stage through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
            if (j + kAhead < nsteps) load(j + kAhead, ra, rb);
            return true;
        };
        // kAhead register sets: the loads of step j + kAhead are issued when
        // step j is stored, which covers the L2 latency under load
        uint4 ra0[kChunksA], rb0[kChunksB], ra1[kChunksA], rb1[kChunksB];
        load(0, ra0, rb0);
        if (nsteps > 1) load(1, ra1, rb1);
        if constexpr (kAhead == 4) {
            uint4 ra2[kChunksA], rb2[kChunksB], ra3[kChunksA], rb3[kChunksB];
            if (nsteps > 2) load(2, ra2, rb2);
            if (nsteps > 3) load(3, ra3, rb3);
            for (int j = 0; j < nsteps; j += 4) {
                if (!step(j, ra0, rb0)) break;
                if (j + 1 < nsteps && !step(j + 1, ra1, rb1)) break;
                if (j + 2 < nsteps && !step(j + 2, ra2, rb2)) break;
                if (j + 3 < nsteps && !step(j + 3, ra3, rb3)) break;
            }
        } else {
            for (int j = 0; j < nsteps; j += 2) {
                if (!step(j, ra0, rb0)) break;
                if (j + 1 < nsteps && !step(j + 1, ra1, rb1)) break;
            }
        }
    } else {
        // ------------------------------------------------ MMA issue, chunk moves, epilogue
        // warp 8 + qd reads TMEM lanes 32 qd .. 32 qd + 31 (token rows of
        // the tile); warp 8 also issues each chunk's MMAs (lane 0)
        const int qd = warp - kEpiWarp0;
        const int et = threadIdx.x - kEpiWarp0 * 32;
        const bool issuer = (qd == 0);
        if (p.pdl) pdl_wait();
        for (int i = et; i < kTileN; i += 128) sw_tile[i] = (n0 + i < p.N) ? p.s_w[n0 + i] : 0.0f;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int tok = m0 + 32 * qd + lane;
        const float sa = tok < p.M ? p.s_a[tok] : 0.0f;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        uint16_t *yr = p.y + static_cast<size_t>(tok < p.M ? tok : 0) * p.N;
        // bf16_rne((float(acc) * s_a) * s_w) of 32 columns of this thread's
        // token row, stored to y
        auto store_y = [&](int col, const uint32_t (&tot)[32]) {
            if (tok >= p.M) return;
            uint32_t o[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                uint32_t b2 = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float f = __int2float_rn(static_cast<int32_t>(tot[e + h]));
                    f = __fmul_rn(f, sa);
                    f = __fmul_rn(f, sw_tile[col + e + h]);
                    b2 |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f))) << (16 * h);
                }
                o[e >> 1] = b2;
            }
            const int n = n0 + col;
            if (p.vec_y && n + 32 <= p.N) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4 *>(yr + n + 8 * v) = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (n + e < p.N) yr[n + e] = static_cast<uint16_t>(o[e >> 1] >> (16 * (e & 1)));
            }
        };
        const int nch = (nsteps + kChunkSteps - 1) / kChunkSteps;
        constexpr uint32_t idesc = tc::idesc_f16_f32(kTileM, kTileN);
        int j = 0;
        for (int ch = 0; ch < nch; ++ch) {
            if (issuer) {
                bool ok = true;
                if (ch > 0) {
                    // the previous chunk's sum must have left D (all four warps)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(acc_empty, (ch - 1) & 1, abort_flag));
                    tc::fence_after();
                }
                const int jend = min(nsteps, (ch + 1) * kChunkSteps);
                for (; ok && j < jend; ++j) {
                    const int s = j % kStages;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (j / kStages) & 1, abort_flag));
                    if (!ok) break;
                    tc::fence_after();
                    if (lane == 0) {
                        const uint32_t a0 = smem_u32(smem + s * kStageBytes);
                        const uint32_t b0 = a0 + kStageA;
                        const int kc = j % kChunkSteps;
#pragma unroll
                        for (int k = 0; k < kStepK / 16; ++k)
                            tc::mma_f16_ss(tmem, tc::sdesc_kmajor_sw128(a0 + 32 * k),
                                           tc::sdesc_kmajor_sw128(b0 + 32 * k), idesc, (kc | k) != 0 ? 1u : 0u);
                        tc::commit(&empty[s]);
                        if (j == jend - 1) tc::commit(acc_full);
                    }
                    __syncwarp();
                }
                if (!ok) {
                    fail();
                    break;
                }
            }
            // warp-uniform: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(acc_full, ch & 1, abort_flag))) {
                fail();
                break;
            }
            tc::fence_after();
            if (ch + 1 < nch) {
#pragma unroll 1
                for (int col = 0; col < kTileN; col += 32) {
                    uint32_t d[32], tot[32];
                    tc::ld32(lane_addr + col, d);
                    if (ch > 0) tc::ld32(lane_addr + kTotCol + col, tot);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int32_t v = f2i_exact(__uint_as_float(d[e]));
                        tot[e] = ch > 0 ? static_cast<uint32_t>(static_cast<int32_t>(tot[e]) + v) : static_cast<uint32_t>(v);
                    }
                    tc::st32(lane_addr + kTotCol + col, tot);
                }
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            } else if constexpr (!kSplit) {
#pragma unroll 1
                for (int col = 0; col < kTileN; col += 32) {
                    uint32_t d[32], tot[32];
                    __syncwarp();   // reconverge after the ragged stores of the previous columns
                    tc::ld32(lane_addr + col, d);
                    if (ch > 0) tc::ld32(lane_addr + kTotCol + col, tot);
                    tc::wait_ld();
                    if (tok >= p.M) continue;
                    uint32_t o[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        uint32_t b2 = 0;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            int32_t acc = f2i_exact(__uint_as_float(d[e + h]));
                            if (ch > 0) acc += static_cast<int32_t>(tot[e + h]);
                            float f = __int2float_rn(acc);
                            f = __fmul_rn(f, sa);
                            f = __fmul_rn(f, sw_tile[col + e + h]);
                            b2 |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f))) << (16 * h);
                        }
                        o[e >> 1] = b2;
                    }
                    const int n = n0 + col;
                    if (p.vec_y && n + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            *reinterpret_cast<uint4 *>(yr + n + 8 * v) =
                                make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (n + e < p.N) yr[n + e] = static_cast<uint16_t>(o[e >> 1] >> (16 * (e & 1)));
                    }
                }
            } else {
                // A split tile.  Each K range takes an arrival ticket.  The
                // first parts - 1 arrivals store their sums into the tile's
                // slots (one per ticket, column-major so that a warp's stores
                // cover contiguous rows) and count themselves done; the last
                // arrival keeps its own sums in TMEM, waits until the others
                // are done (they are running: they arrived first), adds their
                // slots and applies the epilogue.  Integer adds in any order
                // give the same exact sum.
                const int ti = tile - p.full_tiles;
                int *arrive = p.tail_cnt + 2 * ti, *done = arrive + 1;
                const size_t slot0 = static_cast<size_t>(ti) * (parts - 1);
                const int row = 32 * qd + lane;
                if (et == 0) *last_part = atomicAdd(arrive, 1);
                asm volatile("bar.sync 1, 128;" ::: "memory");
                const int ticket = *last_part;
                if (ticket < parts - 1) {
                    int32_t *dst = p.tail_acc + (slot0 + ticket) * (kTileN * kTileM) + row;
#pragma unroll 1
                    for (int col = 0; col < kTileN; col += 32) {
                        uint32_t d[32], tot[32];
                        tc::ld32(lane_addr + col, d);
                        if (ch > 0) tc::ld32(lane_addr + kTotCol + col, tot);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            int32_t v = f2i_exact(__uint_as_float(d[e]));
                            if (ch > 0) v += static_cast<int32_t>(tot[e]);
                            __stcg(dst + (col + e) * kTileM, v);
                        }
                    }
                    __threadfence();
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (et == 0) red_release_gpu_add(done, 1);
                } else {
                    if (et == 0) {
                        const unsigned long long t0 = global_timer_ns();
                        int spins = 0;
                        while (ld_acquire_gpu(done) < parts - 1) {
                            __nanosleep(64);
                            if ((++spins & 63) == 0 && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                                fail();
                                break;
                            }
                        }
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (!*abort_flag) {
                        const int32_t *src = p.tail_acc + slot0 * (kTileN * kTileM) + row;
#pragma unroll 1
                        for (int col = 0; col < kTileN; col += 32) {
                            uint32_t d[32], tot[32];
                            __syncwarp();   // reconverge after the ragged stores of the previous columns
                            tc::ld32(lane_addr + col, d);
                            if (ch > 0) tc::ld32(lane_addr + kTotCol + col, tot);
                            tc::wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int32_t v = f2i_exact(__uint_as_float(d[e]));
                                tot[e] = ch > 0 ? static_cast<uint32_t>(static_cast<int32_t>(tot[e]) + v)
                                                : static_cast<uint32_t>(v);
                            }
                            // two slots per round trip: 64 loads in flight
                            const int32_t *sc = src + col * kTileM;
                            int o = 0;
#pragma unroll 1
                            for (; o + 1 < parts - 1; o += 2) {
                                int32_t l0[32], l1[32];
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    l0[e] = __ldcg(sc + static_cast<size_t>(o) * (kTileN * kTileM) + e * kTileM);
                                    l1[e] = __ldcg(sc + static_cast<size_t>(o + 1) * (kTileN * kTileM) + e * kTileM);
                                }
#pragma unroll
                                for (int e = 0; e < 32; ++e) tot[e] += static_cast<uint32_t>(l0[e] + l1[e]);
                            }
                            if (o < parts - 1) {
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    tot[e] += static_cast<uint32_t>(
                                        __ldcg(sc + static_cast<size_t>(o) * (kTileN * kTileM) + e * kTileM));
                            }
                            store_y(col, tot);
                        }
                        if (et == 0) {
                            *arrive = 0;
                            *done = 0;
                        }
                    }
                }
            }
        }
        __syncwarp();
        tc::fence_before();
        if (issuer) {
            // nothing may still read shared memory or write TMEM when the CTA
            // frees them
            if (lane == 0) tc::commit(drain);
            volatile int never = 0;
            mbar_wait_bounded(drain, 0, &never);
        }
    }
    __syncwarp();
    tc::fence_before();
    __syncthreads();
    if (warp == kEpiWarp0) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream)
{
    static bool attr_set = false;
    static int sms = 0;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Params p;
    p.q = a.q;
    p.w = a.w_q;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.y = a.y;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.kt = (a.K + kStepK - 1) / kStepK;
    p.vec_y = ((a.N % 8) == 0 && (reinterpret_cast<uintptr_t>(a.y) & 15u) == 0) ? 1 : 0;
    p.ws = a.ws;
    p.pdl = a.pdl ? 1 : 0;
    // One CTA per SM.  Tiles that fill whole waves run whole; when the last
    // wave would be at most half full, its tiles are split along K into as
    // many ranges (of at least 8 steps) as fill it, within the scratch slots.
    p.tiles_m = (a.M + kTileM - 1) / kTileM;
    const int tiles = p.tiles_m * ((a.N + kTileN - 1) / kTileN);
    p.full_tiles = tiles;
    p.parts = 1;
    p.tail_acc = a.tail_acc;
    p.tail_cnt = a.tail_cnt;
    const int rem = sms > 0 ? tiles % sms : 0;
    if (a.tail_acc && rem > 0 && rem <= sms / 2 && rem <= kMaxTailTiles) {
        // ranges of at least 8 steps; rem * (parts - 1) slots of scratch
        const int parts = min(min(sms / rem, p.kt / 8), 1 + kMaxTailSlots / rem);
        if (parts >= 2) {
            p.full_tiles = tiles - rem;
            p.parts = parts;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (p.full_tiles > 0) {
        cfg.gridDim = dim3(static_cast<unsigned>(p.full_tiles));
        cfg.numAttrs = a.pdl ? 1 : 0;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_kernel<false>, p);
        if (e != cudaSuccess || p.full_tiles == tiles) return e;
    }
    // The split tiles, after the whole ones: a programmatic dependent whose
    // CTAs wait (griddepcontrol.wait) for everything before them, so they
    // take the SMs as the whole tiles finish.
    cfg.gridDim = dim3(static_cast<unsigned>((tiles - p.full_tiles) * p.parts));
    cfg.numAttrs = (a.pdl || p.full_tiles > 0) ? 1 : 0;
    p.pdl = cfg.numAttrs;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<true>, p);
}

}  // namespace bi
