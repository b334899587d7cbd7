// Verify-pass executor: a program of W8A8 ops (activation quantisation,
// linear layers, the LM-head argmax) run by one persistent kernel.
//
// A decode or verify pass is a chain of small dependent steps whose cost is
// the weight read ("why speculative decoding changed my output", Fig. 1;
// "My speculative decoder got slower", "The physics").  Launched one by one,
// every step pays a launch, a ramp to full HBM bandwidth and a tail; for the
// 4 MB k/v projections those cost more than the read itself.  Here one CTA
// per SM runs every op in order.  Between ops the CTAs meet at a grid-wide
// barrier (ops may read what earlier ops wrote), but the producer warp of
// each CTA keeps streaming weight tiles of the ops ahead, because weights
// never depend on earlier ops; only the activation tiles wait for the
// barrier.  A deep shared-memory ring (11 stages of 18 KB) carries the weight
// stream across the barriers and the quantisation steps.
//
// Results are bit-identical to issuing the same calls one by one: the
// arithmetic of each op is that of bi_quantize_act / bi_linear_w8a8 /
// bi_lmhead_argmax (exact int32 sums, fixed per-element epilogue).
#include "bi.h"
#include "kernels.cuh"
#include "ptx.cuh"
#include "row_ops.cuh"
#include "stream_mma.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

namespace bi {

namespace {

using namespace stream;
using Gp = Geo<2>;   // eight consumer warps per CTA, two CTAs per SM (measured best)

constexpr int kKSplit = Gp::kKSplit;
constexpr int kConsumerWarps = Gp::kConsumerWarps;
constexpr int kThreads = Gp::kThreads;

struct alignas(128) DevOp {
    int kind;            // BI_OP_*
    int M, N, K;
    int upr;             // units per row block (linear ops)
    int bar;             // grid barrier to pass before the op (0: none)
    int qwait;           // or: rows quantised so far (whole run) to wait for (0: none)
    long long units;     // total units (linear ops)
    const uint16_t *x;   // quantise: input rows
    long long ldx;
    int8_t *q;           // quantise: output codes; linear: input codes
    float *s_a;          // quantise: output scales; linear: input scales
    const float *s_w;
    uint16_t *y;         // linear: output; head: logits or null
    int32_t *argmax;     // head: output
    int map_w, map_q;    // indices of the TMA descriptors
    int row_shift;       // quantise: row m is done by CTA (m + row_shift) % G
};

struct alignas(128) ProgHeader {
    int n_ops;
    int n_maps;
    int mt;              // token tiles: 1 (M <= 8) or 2 (M <= 16)
    int magic;
    // greedy verification after the run, for the last LM-head op that asks for
    // it (verify_M = 0: none): its argmax, drafted tokens and result
    int verify_M;
    const int32_t *verify_argmax;
    const int32_t *verify_draft;
    int32_t *verify_accept;
};

constexpr int kProgMagic = 0x42495031;  // "BIP1"

size_t ops_offset() { return sizeof(ProgHeader); }
size_t maps_offset(int n_ops) { return sizeof(ProgHeader) + sizeof(DevOp) * static_cast<size_t>(n_ops); }

template <int MT>
struct PCfg {
    static constexpr int kTok = 8 * MT;
    static constexpr int kAChunkBytes = kTok * 128;
    static constexpr int kWStage = kNch * kWChunkBytes;                 // 16 KB
    static constexpr int kAStage = kNch * kAChunkBytes;                 // 2 or 4 KB
    static constexpr int kStages = (MT == 1) ? 5 : 4;                   // two CTAs per SM
    static constexpr int kRedBytes = (kKSplit - 1) * kBM * kMaxTok * 4;
    // a deferred run's slot values after its adds: [4 row groups x 32 lanes][MT * 4] uint64
    static constexpr int kDeferBytes = 4 * 32 * MT * 4 * 8;
    // full, empty, pend_map (8 B each per stage), sbest, pend_bar/qw/c (4 B each per stage), flags, sq
    static constexpr int kCtlBytes =
        3 * kStages * 8 + kConsumerWarps * kMaxTok * 8 + 3 * kStages * 4 + 16 * 4 + kConsumerWarps * 4;
    static constexpr int kSmemBytes = kStages * (kWStage + kAStage) + kRedBytes + kDeferBytes + 1024 + kCtlBytes;
};

// Order this thread's earlier generic-proxy global writes (or, on the reading
// side, its acquire) with async-proxy (TMA) accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Workspace of a program run (its own layout: up to kProgMaxGrid CTAs):
//   [0, 256)  status, argmax ticket, barrier arrivals, exit ticket, rows quantised
//   best [kProgMaxGrid][16] uint64, partial [kProgMaxGrid][64][16] uint64
// A partial slot holds, per element of a row block shared by several CTAs,
// (K units summed so far) * 2^40 + (their int32 partial sum), as one 64-bit
// integer, so one atomic add both accumulates a contribution and tells its
// issuer whether it completed the element.
constexpr int kProgMaxGrid = 512;
constexpr size_t kPwBestOff = 256;
constexpr size_t kPwPartialOff = kPwBestOff + sizeof(unsigned long long) * kProgMaxGrid * kMaxTok;
constexpr size_t kPwBytes = kPwPartialOff + sizeof(unsigned long long) * kProgMaxGrid * kBM * kMaxTok;

struct ProgWs {
    int *status;
    int *ticket;
    int *bar;            // grid barrier arrivals (G per barrier)
    int *exit_ticket;
    int *qdone;          // activation rows quantised so far in this run
    unsigned long long *best;
    unsigned long long *partial;
};

template <int MT>
__global__ void __launch_bounds__(kThreads, 2) program_kernel(const ProgHeader *__restrict__ prog, ProgWs ws)
{
    using C = PCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    uint8_t *sA = smem + C::kStages * C::kWStage;
    int32_t *sred = reinterpret_cast<int32_t *>(sA + C::kStages * C::kAStage);
    unsigned long long *sdefer = reinterpret_cast<unsigned long long *>(sA + C::kStages * C::kAStage + C::kRedBytes);
    // control area: 8-byte fields first, then 4-byte ones, so every field is
    // naturally aligned whatever the stage count
    uint64_t *full =
        reinterpret_cast<uint64_t *>(sA + C::kStages * C::kAStage + C::kRedBytes + C::kDeferBytes);
    uint64_t *empty = full + C::kStages;
    // per ring stage, for a use whose activation tile is not yet requested:
    const CUtensorMap **pend_map = reinterpret_cast<const CUtensorMap **>(empty + C::kStages);  // its q descriptor
    unsigned long long *sbest = reinterpret_cast<unsigned long long *>(pend_map + C::kStages);   // [warps][16]
    int *pend_bar = reinterpret_cast<int *>(sbest + kConsumerWarps * kMaxTok);               // barrier to pass
    int *pend_qw = pend_bar + C::kStages;                                                    // or rows to await
    int *pend_c = pend_qw + C::kStages;                                                      // its K unit
    volatile int *flags = reinterpret_cast<volatile int *>(pend_c + C::kStages);  // abort
    volatile int *abort_flag = flags;
    float *sq = reinterpret_cast<float *>(const_cast<int *>(flags) + 16);        // [kConsumerWarps] quant reduce

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const DevOp *ops = reinterpret_cast<const DevOp *>(reinterpret_cast<const char *>(prog) + sizeof(ProgHeader));
    const CUtensorMap *maps =
        reinterpret_cast<const CUtensorMap *>(reinterpret_cast<const char *>(ops) + sizeof(DevOp) * prog->n_ops);
    const int n_ops = prog->n_ops;
    const uint32_t stage_bytes = C::kWStage + C::kAStage;

    if (threadIdx.x == kConsumerWarps * 32) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    // a program built for the other token-tile count would overrun the stages
    if (prog->magic != kProgMagic || prog->mt != MT) {
        if (threadIdx.x == 0) atomicExch(ws.status, DEV_BAD_PROGRAM);
        return;
    }

    if (warp == kConsumerWarps) {
        // -------------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_a = policy_evict_last();
        int seen = 0;        // last value read from the barrier counter
        int ja = 0;          // next ring use whose activation tile is not yet requested
        int j = 0;           // next ring use
        // Walks this CTA's weight units of all linear ops in program order;
        // the fields of the current op are kept in registers.
        struct Cursor {
            int op;
            long long u, ue;
            int rb, c, upr, bar, qwait;
            const CUtensorMap *mw, *mq;
        };
        auto seek = [&](Cursor &k, int from) {   // first unit of the first linear op >= from
            for (k.op = from; k.op < n_ops; ++k.op) {
                const DevOp o = ops[k.op];
                if (o.kind != BI_OP_LINEAR && o.kind != BI_OP_LMHEAD) continue;
                k.u = range_start(blockIdx.x, o.units, G);
                k.ue = range_start(blockIdx.x + 1, o.units, G);
                if (k.u < k.ue) {
                    k.upr = o.upr;
                    k.bar = o.bar;
                    k.qwait = o.qwait;
                    k.rb = static_cast<int>(k.u / o.upr);
                    k.c = static_cast<int>(k.u % o.upr);
                    k.mw = &maps[o.map_w];
                    k.mq = &maps[o.map_q];
                    return;
                }
            }
        };
        auto advance = [&](Cursor &k) {
            if (++k.u == k.ue) {
                seek(k, k.op + 1);
            } else if (++k.c == k.upr) {
                k.c = 0;
                ++k.rb;
            }
        };
        Cursor wc;           // next unit to load into the ring
        seek(wc, 0);

        // request activation tiles of every use whose op's barrier has passed
        int seen_q = 0;      // last value read from the rows-quantised counter
        auto issue_ready_a = [&](bool refresh) {
            bool refreshed = false;
            while (ja < j) {
                const int s = ja % C::kStages;
                const int b = pend_bar[s], qw = pend_qw[s];
                if ((b > 0 && seen < b * G) || (qw > 0 && seen_q < qw)) {
                    if (!refresh || refreshed) return;
                    if (b > 0) seen = ld_acquire_gpu(ws.bar);
                    if (qw > 0) seen_q = ld_acquire_gpu(ws.qdone);
                    fence_proxy_async_global();
                    refreshed = true;
                    if ((b > 0 && seen < b * G) || (qw > 0 && seen_q < qw)) {
                        __nanosleep(128);   // back off: every CTA polls the same counters
                        return;
                    }
                }
#pragma unroll
                for (int ch = 0; ch < kNch; ++ch)
                    tma_load_2d(sA + s * C::kAStage + ch * C::kAChunkBytes, pend_map[s], &full[s],
                                pend_c[s] * kUnitK + ch * 128, 0, pol_a);
                ++ja;
            }
        };
        unsigned long long t0 = global_timer_ns();
        while (wc.op < n_ops && !*abort_flag) {
            const int s = j % C::kStages;
            if (j >= C::kStages) {
                const uint32_t par = ((j / C::kStages) - 1) & 1;
                int spins = 0;
                // poll without sleeping: a freed stage or a passed barrier must
                // turn into requests at once
                while (!mbar_test_wait(&empty[s], par)) {
                    issue_ready_a(true);
                    if ((++spins & 63) == 0 && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                        *abort_flag = 1;
                        atomicExch(ws.status, DEV_TIMEOUT);
                        break;
                    }
                }
                if (*abort_flag) break;
            }
            mbar_arrive_expect_tx(&full[s], stage_bytes);
#pragma unroll
            for (int ch = 0; ch < kNch; ++ch)
                tma_load_2d(sW + s * C::kWStage + ch * kWChunkBytes, wc.mw, &full[s], wc.c * kUnitK + ch * 128,
                            wc.rb * kBM, pol_w);
            pend_map[s] = wc.mq;
            pend_bar[s] = wc.bar;
            pend_qw[s] = wc.qwait;
            pend_c[s] = wc.c;
            ++j;
            advance(wc);
            issue_ready_a(false);
            t0 = global_timer_ns();
        }
        // remaining activation tiles once their barriers pass
        t0 = global_timer_ns();
        while (ja < j && !*abort_flag) {
            issue_ready_a(true);
            if (ja < j && global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicExch(ws.status, DEV_TIMEOUT);
            }
        }
        if (*abort_flag) {
            // let every copy still in flight land before the CTA exits
            volatile int never = 0;
            const int first = ja > C::kStages ? ja - C::kStages : 0;
            for (int k = first; k < ja; ++k) mbar_wait_bounded(&full[k % C::kStages], (k / C::kStages) & 1, &never);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const Lane L = lane_setup<MT, kKSplit>(warp, lane);
    const int g = L.g, tq = L.tq, rg = L.rg, kq = L.kq;
    const int ctid = threadIdx.x;   // 0 .. 32 * kConsumerWarps - 1
    int j = 0;

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            atomicExch(ws.status, DEV_TIMEOUT);
        }
    };
    // all CTAs have finished every op before barrier b
    auto grid_sync = [&](int b) {
        consumer_bar();
        if (ctid == 0) {
            red_release_gpu_add(ws.bar, 1);
            const unsigned long long t0 = global_timer_ns();
            int spins = 0;
            while (ld_acquire_gpu(ws.bar) < b * G) {
                __nanosleep(64);
                if ((++spins & 63) == 0 && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                    fail();
                    break;
                }
            }
        }
        consumer_bar();
    };

    for (int i = 0; i < n_ops; ++i) {
        const DevOp op = ops[i];   // by value: the loops below store to global memory
        if (op.bar > 0) grid_sync(op.bar);
        if (op.qwait > 0) {          // the quantisation this op reads has finished everywhere
            if (ctid == 0) {
                const unsigned long long t0 = global_timer_ns();
                int spins = 0;
                while (ld_acquire_gpu(ws.qdone) < op.qwait) {
                    __nanosleep(64);
                    if ((++spins & 63) == 0 && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                        fail();
                        break;
                    }
                }
            }
            consumer_bar();
        }

        if (op.kind != BI_OP_LINEAR && op.kind != BI_OP_LMHEAD) {
            // ------------------------------------------ quantise rows (three kinds)
            // rows (m + row_shift) % G == this CTA; 256 threads per row.  The
            // row's input: x (plain), bf16(h + x) rescaled (residual, h = op.y
            // updated in place), or bf16(relu(x[:, :K]) * x[:, K:2K]).
            const int kind = op.kind;
            int rows_here = 0;
            for (int m = (static_cast<int>(blockIdx.x) - op.row_shift % G + G) % G; m < op.M; m += G) {
                ++rows_here;
                constexpr int kT = kConsumerWarps * 32;
                constexpr int kRegChunks = 8;   // rows up to 8 * kT * 8 = 16384 values stay in registers
                const uint16_t *xr = op.x + static_cast<long long>(m) * op.ldx;
                uint16_t *hr = op.y ? op.y + static_cast<long long>(m) * op.K : nullptr;
                const int nchunk = op.K / 8;
                const bool in_regs = nchunk <= kRegChunks * kT;
                auto load_in = [&](int ci) -> uint4 {
                    const uint4 a = *reinterpret_cast<const uint4 *>(xr + ci * 8);
                    if (kind == BI_OP_RESIDUAL_QUANT)
                        return residual8(*reinterpret_cast<const uint4 *>(hr + ci * 8), a);
                    if (kind == BI_OP_RELU_MUL_QUANT)
                        return relu_mul8(a, *reinterpret_cast<const uint4 *>(xr + op.K + ci * 8));
                    return a;
                };
                float amax = 0.0f;
                uint4 v[kRegChunks];
#pragma unroll
                for (int c = 0; c < kRegChunks; ++c) {
                    const int ci = c * kT + ctid;
                    v[c] = (in_regs && ci < nchunk) ? load_in(ci) : make_uint4(0, 0, 0, 0);
                }
                if (in_regs) {
#pragma unroll
                    for (int c = 0; c < kRegChunks; ++c) amax = absmax8(v[c], amax);
                } else {
                    for (int ci = ctid; ci < nchunk; ci += kT) amax = absmax8(load_in(ci), amax);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                if (lane == 0) sq[warp] = amax;
                consumer_bar();
                amax = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) amax = fmaxf(amax, sq[w]);
                consumer_bar();
                int p2 = 0;
                if (kind == BI_OP_RESIDUAL_QUANT) {
                    p2 = rescale_shift(amax);
                    amax = scale_pow2(amax, p2);   // exact: the rescaled row's largest magnitude
                }
                const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
                const float r = __frcp_rn(s);
                // each thread writes only chunks it read itself (in-place h is safe)
                auto emit = [&](uint4 t, int ci, bool fast) {
                    if (kind == BI_OP_RESIDUAL_QUANT) {
                        t = rescale8(t, p2);
                        *reinterpret_cast<uint4 *>(hr + ci * 8) = t;
                    } else if (kind == BI_OP_RELU_MUL_QUANT && hr) {
                        *reinterpret_cast<uint4 *>(hr + ci * 8) = t;
                    }
                    *reinterpret_cast<uint2 *>(op.q + static_cast<long long>(m) * op.K + ci * 8) =
                        fast ? quant8(t, s, r) : quant8_div(t, s);
                };
                if (in_regs && s >= kQuotientMinScale) {
#pragma unroll
                    for (int c = 0; c < kRegChunks; ++c) {
                        const int ci = c * kT + ctid;
                        if (ci < nchunk) emit(v[c], ci, true);
                    }
                } else {
                    // rows too long for registers, or with a tiny scale
                    const bool fast = s >= kQuotientMinScale;
#pragma unroll 1
                    for (int ci = ctid; ci < nchunk; ci += kT) emit(load_in(ci), ci, fast);
                }
                if (ctid == 0) op.s_a[m] = s;
                fence_proxy_async_global();   // the codes are read by other CTAs' TMA
            }
            if (rows_here > 0) {
                consumer_bar();
                if (ctid == 0) red_release_gpu_add(ws.qdone, rows_here);
            }
            continue;
        }

        // -------------------------------------------------------- linear / head
        const bool head = (op.kind == BI_OP_LMHEAD);
        const long long u_begin = range_start(blockIdx.x, op.units, G);
        const long long u_end = range_start(blockIdx.x + 1, op.units, G);
        float sa_reg[MT][2];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = 8 * t + 2 * tq + e;
                sa_reg[t][e] = tok < op.M ? op.s_a[tok] : 0.0f;
            }
        unsigned long long best[MT][2];
#pragma unroll
        for (int t = 0; t < MT; ++t) best[t][0] = best[t][1] = 0ull;

        auto load_sw = [&](int rb, float (&sw)[2]) {
            const int n0 = rb * kBM + rg * 16 + g;
            sw[0] = n0 < op.N ? op.s_w[n0] : 0.0f;
            sw[1] = n0 + 8 < op.N ? op.s_w[n0 + 8] : 0.0f;
        };
        // y[tok, n] (and the argmax key) of one accumulator element
        auto emit1 = [&](int rb, int t, int e, int32_t acc, const float (&sw)[2]) {
            const int n = rb * kBM + rg * 16 + g + ((e & 2) ? 8 : 0);
            const int tok = 8 * t + 2 * tq + (e & 1);
            if (n >= op.N || tok >= op.M) return;
            float f = __int2float_rn(acc);
            f = __fmul_rn(f, sa_reg[t][e & 1]);
            f = __fmul_rn(f, sw[(e & 2) ? 1 : 0]);
            const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
            if (op.y) op.y[static_cast<size_t>(tok) * op.N + n] = b;
            if (head) {
                const unsigned long long key = argmax_key(b, n);
                if (key > best[t][e & 1]) best[t][e & 1] = key;
            }
        };
        auto slot_of = [&](int rb) {
            const int slot = unit_owner(static_cast<long long>(rb) * op.upr, op.units, G);
            return ws.partial + static_cast<size_t>(slot) * (kBM * kMaxTok);
        };
        auto elem = [&](int t, int e) { return (rg * 16 + g + ((e & 2) ? 8 : 0)) * kMaxTok + 8 * t + 2 * tq + (e & 1); };
        // Add a run's partial sums (nch of the row block's upr K units) to the
        // row block's slot; old[] receives the values before the add.
        auto push = [&](int rb, int nch, const int32_t (&v)[MT][4], unsigned long long (&old)[MT][4]) {
            unsigned long long *part = slot_of(rb);
            const unsigned long long tag = static_cast<unsigned long long>(nch) << 40;
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    old[t][e] = atomicAdd(&part[elem(t, e)],
                                          tag + static_cast<unsigned long long>(static_cast<long long>(v[t][e])));
        };
        // The add that brought an element's unit count to upr completed it:
        // its issuer, seeing the slot's value just after its own add, holds
        // the whole sum; it writes the output and clears the slot.
        auto finish1 = [&](int rb, int t, int e, unsigned long long after, const float (&sw)[2]) {
            const long long a = static_cast<long long>(after);
            const long long units = (a + (1LL << 39)) >> 40;
            if (units == op.upr) {
                slot_of(rb)[elem(t, e)] = 0ull;
                emit1(rb, t, e, static_cast<int32_t>(a - (units << 40)), sw);
            }
        };
        auto after_add = [&](int nch, int32_t v, unsigned long long old) {
            return old + (static_cast<unsigned long long>(nch) << 40) +
                   static_cast<unsigned long long>(static_cast<long long>(v));
        };

        // The first run of the range, if it shares its row block with earlier
        // CTAs, is completed only after the last run is pushed, so that the
        // two atomic round trips overlap.
        bool first_deferred = false;
        int f_rb = 0;
        float f_sw[2] = {0.0f, 0.0f};
        unsigned long long *my_defer = sdefer + (rg * 32 + lane) * (MT * 4);
        long long u = u_begin;
        while (u < u_end) {
            const int rb = static_cast<int>(u / op.upr);
            const int c0 = static_cast<int>(u % op.upr);
            const long long left = u_end - u;
            const int nch = (op.upr - c0) < left ? (op.upr - c0) : static_cast<int>(left);
            int32_t v[MT][4];
#pragma unroll
            for (int t = 0; t < MT; ++t) v[t][0] = v[t][1] = v[t][2] = v[t][3] = 0;
            float sw[2];
            load_sw(rb, sw);
            for (int it = 0; it < nch; ++it, ++j) {
                const int s = j % C::kStages;
                if (*abort_flag || !mbar_wait_bounded(&full[s], (j / C::kStages) & 1, abort_flag)) {
                    fail();
                    continue;
                }
                consume_stage<MT, kKSplit>(smem_u32(sW + s * C::kWStage), smem_u32(sA + s * C::kAStage),
                                           C::kAChunkBytes, L, v);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // fold the two K halves of each row group (kq == 1 into kq == 0)
            if (kq > 0) {
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sred[((kq - 1) * kBM + rg * 16 + g + ((e & 2) ? 8 : 0)) * kMaxTok + 8 * t + 2 * tq + (e & 1)] =
                            v[t][e];
            }
            consumer_bar();
            if (kq == 0) {
#pragma unroll
                for (int o = 1; o < kKSplit; ++o)
#pragma unroll
                    for (int t = 0; t < MT; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[t][e] += sred[((o - 1) * kBM + rg * 16 + g + ((e & 2) ? 8 : 0)) * kMaxTok + 8 * t +
                                            2 * tq + (e & 1)];
            }
            consumer_bar();
            if (kq == 0 && !*abort_flag) {
                if (c0 == 0 && nch == op.upr) {
#pragma unroll
                    for (int t = 0; t < MT; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e) emit1(rb, t, e, v[t][e], sw);
                } else {
                    unsigned long long old[MT][4];
                    push(rb, nch, v, old);
                    if (u == u_begin && u + nch < u_end) {
                        first_deferred = true;
                        f_rb = rb;
                        f_sw[0] = sw[0];
                        f_sw[1] = sw[1];
#pragma unroll
                        for (int t = 0; t < MT; ++t)
#pragma unroll
                            for (int e = 0; e < 4; ++e) my_defer[t * 4 + e] = after_add(nch, v[t][e], old[t][e]);
                    } else {
#pragma unroll
                        for (int t = 0; t < MT; ++t)
#pragma unroll
                            for (int e = 0; e < 4; ++e) finish1(rb, t, e, after_add(nch, v[t][e], old[t][e]), sw);
                    }
                }
            }
            u += nch;
        }
        if (first_deferred && !*abort_flag) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) finish1(f_rb, t, e, my_defer[t * 4 + e], f_sw);
        }
        if (head) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    unsigned long long vv = best[t][h];
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        const unsigned long long w = __shfl_xor_sync(0xffffffffu, vv, o);
                        vv = w > vv ? w : vv;
                    }
                    if (g == 0) sbest[warp * kMaxTok + 8 * t + 2 * tq + h] = vv;
                }
            if (MT == 1 && lane < 8) sbest[warp * kMaxTok + 8 + lane] = 0ull;
            consumer_bar();
            if (warp == 0) {
                if (lane < kMaxTok) {
                    unsigned long long vv = 0ull;
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const unsigned long long x = sbest[w * kMaxTok + lane];
                        vv = x > vv ? x : vv;
                    }
                    ws.best[blockIdx.x * kMaxTok + lane] = vv;
                    __threadfence();
                }
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence();
                    last = (atomicAdd(ws.ticket, 1) == G - 1);
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    if (lane < op.M) {
                        unsigned long long vv = 0ull;
                        for (int b = 0; b < G; ++b) {
                            const unsigned long long x = __ldcg(&ws.best[b * kMaxTok + lane]);
                            vv = x > vv ? x : vv;
                        }
                        op.argmax[lane] =
                            static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(vv & 0xFFFFFFFFull));
                    }

                    if (lane == 0) atomicExch(ws.ticket, 0);
                }
            }
            consumer_bar();
        }
    }

    // the last CTA out resets the barrier counter for the next run
    consumer_bar();
    if (ctid == 0) {
        __threadfence();
        if (atomicAdd(ws.exit_ticket, 1) == G - 1) {
            atomicExch(ws.bar, 0);
            atomicExch(ws.qdone, 0);
            atomicExch(ws.exit_ticket, 0);
        }
    }
}

// Greedy verification after a program run (the same computation as
// bi_greedy_verify), one warp; nothing to do for a program without it.
__global__ void program_verify_kernel(const ProgHeader *__restrict__ prog)
{
    const int M = prog->verify_M;
    if (M < 1) return;
    const int32_t *argmax = prog->verify_argmax, *draft = prog->verify_draft;
    const int lane = threadIdx.x;
    int L = M - 1;
    for (int base = 0; base < M - 1; base += 32) {
        const int i = base + lane;
        const bool miss = i < M - 1 && argmax[i] != draft[i];
        const unsigned b = __ballot_sync(0xffffffffu, miss);
        if (b) {
            L = base + __ffs(b) - 1;
            break;
        }
    }
    if (lane == 0) {
        prog->verify_accept[0] = L;
        prog->verify_accept[1] = argmax[L];
    }
}

template <int MT>
cudaError_t launch_program(const void *prog, void *wsp, int grid, cudaStream_t stream)
{
    using C = PCfg<MT>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(program_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    char *b = static_cast<char *>(wsp);
    ProgWs ws;
    ws.status = reinterpret_cast<int *>(b);
    ws.ticket = reinterpret_cast<int *>(b + 4);
    ws.bar = reinterpret_cast<int *>(b + 8);
    ws.exit_ticket = reinterpret_cast<int *>(b + 12);
    ws.qdone = reinterpret_cast<int *>(b + 16);
    ws.best = reinterpret_cast<unsigned long long *>(b + kPwBestOff);
    ws.partial = reinterpret_cast<unsigned long long *>(b + kPwPartialOff);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, program_kernel<MT>, static_cast<const ProgHeader *>(prog), ws);
}

// ------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode(CUtensorMap *map, const void *base, long long rows, long long cols, int box_rows, bool once)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              once ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool is_quantising(int kind)
{
    return kind == BI_OP_QUANTIZE_ACT || kind == BI_OP_RESIDUAL_QUANT || kind == BI_OP_RELU_MUL_QUANT;
}

bool is_matmul(int kind) { return kind == BI_OP_LINEAR || kind == BI_OP_LMHEAD; }

// A byte range of device memory.
struct Range {
    const void *p;
    size_t n;
    bool meets(const Range &o) const
    {
        if (!p || !o.p || !n || !o.n) return false;
        const char *a = static_cast<const char *>(p), *b = static_cast<const char *>(o.p);
        return a < b + o.n && b < a + n;
    }
};

// What a quantising op reads: x (K or 2K columns per row) and, for the
// residual kind, the stream h it also writes.  Returns the number of ranges.
int quant_inputs(const bi_op &o, Range (&in)[2])
{
    if (!is_quantising(o.kind)) return 0;
    const size_t width = (o.kind == BI_OP_RELU_MUL_QUANT) ? 2 * static_cast<size_t>(o.K) : o.K;
    in[0] = {o.x, (static_cast<size_t>(o.M > 0 ? o.M : 1) - 1) * o.ldx * 2 + width * 2};
    if (o.kind == BI_OP_RESIDUAL_QUANT) {
        in[1] = {o.y, static_cast<size_t>(o.M) * o.K * 2};
        return 2;
    }
    return 1;
}

bool a16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool a4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace bi

extern "C" {

BI_API size_t bi_program_bytes(int n_ops)
{
    if (n_ops < 1) return 0;
    return bi::maps_offset(n_ops) + sizeof(CUtensorMap) * 2 * static_cast<size_t>(n_ops);
}

BI_API size_t bi_program_workspace_size(void)
{
    return bi::kPwBytes;
}

BI_API bi_status bi_program_build(const bi_op *ops, int n_ops, void *program, size_t program_bytes)
{
    using namespace bi;
    if (!ops || n_ops < 1 || !program) return BI_ERR_INVALID_ARG;
    if (program_bytes < bi_program_bytes(n_ops) || (reinterpret_cast<uintptr_t>(program) & 127u))
        return BI_ERR_INVALID_ARG;
    std::vector<char> host(bi_program_bytes(n_ops), 0);
    ProgHeader *h = reinterpret_cast<ProgHeader *>(host.data());
    DevOp *dops = reinterpret_cast<DevOp *>(host.data() + ops_offset());
    CUtensorMap *maps = reinterpret_cast<CUtensorMap *>(host.data() + maps_offset(n_ops));
    int n_maps = 0, mt = 1, n_bars = 0, rows_quantised = 0;
    for (int i = 0; i < n_ops; ++i) {
        const bi_op &o = ops[i];
        if (o.kind == BI_OP_LINEAR || o.kind == BI_OP_LMHEAD) mt = (o.M > 8) ? 2 : mt;
    }
    for (int i = 0; i < n_ops; ++i) {
        const bi_op &o = ops[i];
        DevOp &d = dops[i];
        d.kind = o.kind;
        d.M = o.M;
        d.N = o.N;
        d.K = o.K;
        // An op starts after every earlier op has completed: a grid barrier,
        // except that a linear or head op reading the codes the quantisation
        // just before it wrote waits only for that quantisation's rows.
        d.bar = 0;
        d.qwait = 0;
        if (i > 0) {
            const bi_op &p = ops[i - 1];
            const bool reads_prev_quant = is_matmul(o.kind) && is_quantising(p.kind) && p.q == o.q &&
                                          p.s_a == o.s_a && p.M == o.M && p.K == o.K;
            // the op's outputs must not be what the quantisation read (a write
            // could race with its reads)
            Range in[2];
            const int n_in = quant_inputs(p, in);
            const Range y = {o.y, o.y ? static_cast<size_t>(o.M) * o.N * 2 : 0};
            const Range am = {o.argmax, o.argmax ? static_cast<size_t>(o.M) * 4 : 0};
            bool overlap = false;
            for (int t = 0; t < n_in; ++t) overlap = overlap || in[t].meets(y) || in[t].meets(am);
            if (reads_prev_quant && !overlap) {
                d.qwait = rows_quantised;
            } else {
                d.bar = ++n_bars;
            }
        }
        if (o.M < 1 || o.K < 16 || (o.K % 16) != 0) return BI_ERR_INVALID_ARG;
        if (o.K > 133144) return BI_ERR_INT32_BOUND;
        if (is_quantising(o.kind)) {
            const long long width = (o.kind == BI_OP_RELU_MUL_QUANT) ? 2LL * o.K : o.K;
            if (!o.x || !o.q || !o.s_a || o.ldx < width || o.M > 65535) return BI_ERR_INVALID_ARG;
            if (o.kind == BI_OP_RESIDUAL_QUANT && !o.y) return BI_ERR_INVALID_ARG;
            if (!a16(o.x) || !a16(o.q) || !a4(o.s_a) || (o.ldx % 8) != 0 || (o.y && !a16(o.y)))
                return BI_ERR_ALIGNMENT;
            if (o.kind == BI_OP_QUANTIZE_ACT && o.y) return BI_ERR_INVALID_ARG;
            // h (or m) is written while x is read: they may not share memory
            Range in[2];
            quant_inputs(o, in);
            const Range out = {o.y, o.y ? static_cast<size_t>(o.M) * o.K * 2 : 0};
            if (out.meets(in[0])) return BI_ERR_INVALID_ARG;
            d.x = o.x;
            d.ldx = o.ldx;
            d.q = o.q;
            d.s_a = o.s_a;
            d.y = o.y;
            d.row_shift = (i * 37) & 1023;
            rows_quantised += o.M;
        } else if (o.kind == BI_OP_LINEAR || o.kind == BI_OP_LMHEAD) {
            if (!o.q || !o.s_a || !o.w_q || !o.s_w || o.N < 1 || o.M > 16) return BI_ERR_INVALID_ARG;
            if (o.kind == BI_OP_LINEAR && !o.y) return BI_ERR_INVALID_ARG;
            if (o.kind == BI_OP_LMHEAD && !o.argmax) return BI_ERR_INVALID_ARG;
            if (o.accept && (o.kind != BI_OP_LMHEAD || (o.M > 1 && !o.draft))) return BI_ERR_INVALID_ARG;
            if ((o.accept && !a4(o.accept)) || (o.draft && !a4(o.draft))) return BI_ERR_ALIGNMENT;
            if (o.accept) {
                h->verify_M = o.M;
                h->verify_argmax = o.argmax;
                h->verify_draft = o.draft;
                h->verify_accept = o.accept;
            }
            if (!a16(o.q) || !a16(o.w_q) || !a4(o.s_a) || !a4(o.s_w) || (o.argmax && !a4(o.argmax)))
                return BI_ERR_ALIGNMENT;
            d.q = o.q;
            d.s_a = o.s_a;
            d.s_w = o.s_w;
            d.y = o.y;
            d.argmax = o.argmax;
            d.upr = (o.K + kUnitK - 1) / kUnitK;
            d.units = static_cast<long long>((o.N + kBM - 1) / kBM) * d.upr;
            d.map_w = n_maps;
            if (!encode(&maps[n_maps++], o.w_q, o.N, o.K, kBM, true)) return BI_ERR_CUDA;
            d.map_q = n_maps;
            if (!encode(&maps[n_maps++], o.q, o.M, o.K, 8 * mt, false)) return BI_ERR_CUDA;
        } else {
            return BI_ERR_INVALID_ARG;
        }
    }
    h->n_ops = n_ops;
    h->n_maps = n_maps;
    h->mt = mt;
    h->magic = kProgMagic;
    if (cudaMemcpy(program, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess) return BI_ERR_CUDA;
    return BI_OK;
}

BI_API bi_status bi_program_run(const void *program, int max_tokens, void *ws, size_t ws_bytes, bi_stream_t stream)
{
    if (!program || (reinterpret_cast<uintptr_t>(program) & 127u)) return BI_ERR_INVALID_ARG;
    if (!ws || ws_bytes < bi::kPwBytes || (reinterpret_cast<uintptr_t>(ws) & 15u)) return BI_ERR_WORKSPACE;
    if (max_tokens < 1 || max_tokens > 16) return BI_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BI_ERR_UNSUPPORTED;
    if (major != 10 || minor != 3) return BI_ERR_UNSUPPORTED;
    const int grid = 2 * sms < bi::kProgMaxGrid ? 2 * sms : bi::kProgMaxGrid;   // two CTAs per SM
    cudaError_t e = max_tokens > 8 ? bi::launch_program<2>(program, ws, grid, stream)
                                   : bi::launch_program<1>(program, ws, grid, stream);
    if (e == cudaSuccess) {
        // the verification of the drafts, if the program asks for it
        bi::program_verify_kernel<<<1, 32, 0, stream>>>(static_cast<const bi::ProgHeader *>(program));
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // extern "C"
