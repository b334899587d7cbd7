// Internal launch interface between the C ABI (bi_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bi {

// ---------------------------------------------------------------- workspace
//
// One layout serves the skinny linear, the LM head and the prefill kernel
// (which uses only the status word):
//   [0, 256)          control words: status (int), argmax ticket (int)
//   rb_counter        kMaxGrid int32   split-K chunk counters, one per slot
//   best              kMaxGrid * 16 uint64   per-CTA argmax keys
//   partial           kMaxGrid * 64 * 16 int32   split-K partial sums
// A slot is owned by the CTA in whose range a split row block starts, so at
// most one split row block maps to a slot.  Counters and partials are reset
// by the kernel that consumes them, so a zero-filled workspace stays zeroed.
constexpr int kMaxGrid = 512;
constexpr int kBM = 64;        // weight rows per row block (4 warps x 16)
constexpr int kMaxTok = 16;    // token columns kept per partial row
constexpr size_t kWsCtrlBytes = 256;
constexpr size_t kWsCounterOff = kWsCtrlBytes;
constexpr size_t kWsBestOff = kWsCounterOff + sizeof(int32_t) * kMaxGrid;
constexpr size_t kWsPartialOff = kWsBestOff + sizeof(unsigned long long) * kMaxGrid * kMaxTok;
constexpr size_t kWsBytes = kWsPartialOff + sizeof(int32_t) * kMaxGrid * kBM * kMaxTok;

// Prefill (M > 16) workspaces append, after kWsBytes, the partial sums of
// tiles split along K (the leftover of the last wave): kMaxTailSlots slots of
// int32 [256][128] (scratch, overwritten before it is read), then two
// counters per split tile (zero between calls, like the rest).
constexpr int kMaxTailTiles = 96;
constexpr int kMaxTailSlots = 96;
constexpr size_t kWsTailAccOff = kWsBytes;
constexpr size_t kWsTailCntOff = kWsTailAccOff + sizeof(int32_t) * kMaxTailSlots * 256 * 128;
constexpr size_t kWsPrefillBytes = kWsTailCntOff + 256 * ((2 * sizeof(int32_t) * kMaxTailTiles + 255) / 256);

struct Workspace {
    int *status;                 // DEV_OK / DEV_TIMEOUT
    int *ticket;                 // CTAs finished (argmax)
    int32_t *rb_counter;         // [kMaxGrid]
    unsigned long long *best;    // [kMaxGrid][kMaxTok]
    int32_t *partial;            // [kMaxGrid][kBM][kMaxTok]
};

inline Workspace workspace_view(void *ws)
{
    char *b = static_cast<char *>(ws);
    Workspace w;
    w.status = reinterpret_cast<int *>(b);
    w.ticket = reinterpret_cast<int *>(b + 4);
    w.rb_counter = reinterpret_cast<int32_t *>(b + kWsCounterOff);
    w.best = reinterpret_cast<unsigned long long *>(b + kWsBestOff);
    w.partial = reinterpret_cast<int32_t *>(b + kWsPartialOff);
    return w;
}

// ---------------------------------------------------------------- launches

cudaError_t launch_quantize_act(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *s_a, bool pdl,
                                cudaStream_t stream);
cudaError_t launch_residual_quantize(uint16_t *h, const uint16_t *y, int64_t ldy, int M, int K, int8_t *q,
                                     float *s_a, bool pdl, cudaStream_t stream);
cudaError_t launch_relu_mul_quantize(const uint16_t *gu, int64_t ldgu, int M, int K, int8_t *q, float *s_a,
                                     uint16_t *m_out, bool pdl, cudaStream_t stream);
cudaError_t launch_wait_selftest(int *status, cudaStream_t stream);
cudaError_t launch_quotient_selftest(unsigned long long *out, cudaStream_t stream);
cudaError_t launch_greedy_verify(const int32_t *argmax, const int32_t *draft, int M, int32_t *out,
                                 cudaStream_t stream);
cudaError_t launch_quantize_weight(const float *w, int64_t ldw, int N, int K, int8_t *w_q, float *s_w,
                                   cudaStream_t stream);
cudaError_t launch_requant_pow2(const int8_t *w_q, const float *s_w, int N, int K, int8_t *w_q_out,
                                float *s_w_out, cudaStream_t stream);

struct SkinnyArgs {
    CUtensorMap map_w;         // W [N, K] int8, box 128 B x 64 rows, 128B swizzle
    CUtensorMap map_q;         // q [M, K] int8, box 128 B x (8 * token tiles) rows, 128B swizzle
    const float *s_a;
    const float *s_w;
    uint16_t *y;               // may be null for the LM head
    int32_t *argmax;           // null for the plain linear
    int M, N, K;
    Workspace ws;
    bool pdl;
    int grid;                  // CTAs (<= kMaxGrid)
};

// M <= 16 weight-streaming kernel (plain linear or LM head with argmax).
cudaError_t launch_skinny(const SkinnyArgs &a, cudaStream_t stream);

struct PrefillArgs {
    const int8_t *q;           // [M, K], rows 16-byte aligned
    const int8_t *w_q;         // [N, K], rows 16-byte aligned
    int32_t *tail_acc;         // split-tile sums (null: no tile is split)
    int *tail_cnt;             // split-tile counters
    const float *s_a;
    const float *s_w;
    uint16_t *y;
    int M, N, K;
    Workspace ws;
    bool pdl;
};

// M > 16 tiled kernel (tcgen05), converting the int8 operands in the tile loop.
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);

// Above kPrefillTmaMinM tokens, prefill workspaces also hold exact f16 copies
// of the operands after kWsPrefillBytes: q [M, K], then w [N, K], each
// 256-byte aligned (scratch: every call overwrites them before reading).  The
// copies cost a pass over the weights (about 3 bytes per weight) whatever M
// is; the TMA-fed kernel that reads them is faster than the converting one by
// more than that above about 256 tokens (measured with N = 12288, K = 4096).
constexpr int kPrefillTmaMinM = 256;
inline size_t prefill_f16_bytes(long long rows, long long K)
{
    return static_cast<size_t>((rows * K * 2 + 255) / 256 * 256);
}

struct PrefillTmaArgs {
    const int8_t *q;           // [M, K], rows 16-byte aligned
    const int8_t *w_q;         // [N, K]
    uint16_t *qf;              // [M, K] f16 copy (workspace)
    uint16_t *wf;              // [N, K] f16 copy (workspace)
    CUtensorMap map_a;         // qf: box 64 x 128, 128-byte swizzle
    CUtensorMap map_b;         // wf: box 64 x 256, 128-byte swizzle
    const float *s_a;
    const float *s_w;
    uint16_t *y;
    int M, N, K;
    Workspace ws;
    bool pdl;
};

// M > 16 tiled kernel (tcgen05) on f16 copies of the operands loaded by TMA,
// after the pass that writes those copies.
cudaError_t launch_prefill_tma(const PrefillTmaArgs &a, cudaStream_t stream);

}  // namespace bi
