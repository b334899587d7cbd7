// C ABI of the batch-invariant W8A8 library: argument validation, TMA
// descriptor encoding and kernel dispatch.  Declarations and the contract of
// every entry point are in include/bi.h.
#include "attn.cuh"
#include "bi.h"
#include "blockq.cuh"
#include "probe.cuh"
#include "host_common.h"
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

using bi::kMaxGrid;
using bi::host::aligned16;
using bi::host::aligned4;
using bi::host::check_k;
using bi::host::device_info;
using bi::host::encode_int8_2d;

constexpr int kMaxAttnQueries = 4096;         // queries of one attention call
constexpr int kMaxAttnPositions = 1 << 20;    // T0 + M: at most 4096 chunks (the merge stages 8 bytes a chunk)
constexpr long long kMaxAttnRows = 65535LL * 32; // M * Hq / Hkv: 32-row blocks on one grid axis

// [a, a + n) and [b, b + m) (bytes) share a byte
bool overlaps(const void *a, size_t n, const void *b, size_t m)
{
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + m && pb < pa + n;
}

bi_status from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

bi_status check_linear_args(const int8_t *q, const float *s_a, int M, int K, const int8_t *w_q, const float *s_w,
                            int N, void *ws, size_t ws_bytes)
{
    const bi_status s = bi::host::check_linear_operands(q, s_a, M, K, w_q, s_w, N);
    if (s != BI_OK) return s;
    if (!ws || ws_bytes < bi::kWsBytes || !aligned16(ws)) return BI_ERR_WORKSPACE;
    return BI_OK;
}

bi_status run_skinny(const int8_t *q, const float *s_a, int M, int K, const int8_t *w_q, const float *s_w, int N,
                     uint16_t *y, int32_t *argmax, void *ws, unsigned flags, cudaStream_t stream)
{
    int sms = 0;
    bi_status st = device_info(&sms);
    if (st != BI_OK) return st;
    bi::SkinnyArgs a;
    const int tok_rows = M > 8 ? 16 : 8;
    st = encode_int8_2d(&a.map_w, w_q, N, K, 128, bi::kBM, true);
    if (st != BI_OK) return st;
    st = encode_int8_2d(&a.map_q, q, M, K, 128, tok_rows, false);
    if (st != BI_OK) return st;
    a.s_a = s_a;
    a.s_w = s_w;
    a.y = y;
    a.argmax = argmax;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = bi::workspace_view(ws);
    a.pdl = (flags & BI_FLAG_PDL) != 0;
    a.grid = bi::host::skinny_grid(sms, N, K, bi::kMaxGrid);
    return from_cuda(bi::launch_skinny(a, stream));
}

}  // namespace

extern "C" {

const char *bi_status_string(bi_status s)
{
    switch (s) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG: null pointer or invalid shape";
    case BI_ERR_ALIGNMENT: return "BI_ERR_ALIGNMENT: pointer or row stride not 16-byte aligned";
    case BI_ERR_INT32_BOUND: return "BI_ERR_INT32_BOUND: K * 127^2 >= 2^31";
    case BI_ERR_WORKSPACE: return "BI_ERR_WORKSPACE: workspace missing or too small";
    case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED: no sm_103a device or missing driver feature";
    case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case BI_ERR_CUDA: return "BI_ERR_CUDA: a CUDA call failed";
    }
    return "unknown bi_status";
}

bi_status bi_quantize_act(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *s_a, unsigned flags,
                          bi_stream_t stream)
{
    if (!x || !q || !s_a) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > 65535 || ldx < K) return BI_ERR_INVALID_ARG;
    bi_status st = check_k(K);
    if (st != BI_OK) return st;
    if (!aligned16(x) || !aligned16(q) || !aligned4(s_a) || (ldx % 8) != 0) return BI_ERR_ALIGNMENT;
    st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_quantize_act(x, ldx, M, K, q, s_a, (flags & BI_FLAG_PDL) != 0, stream));
}

bi_status bi_residual_quantize(uint16_t *h, const uint16_t *y, int64_t ldy, int M, int K, int8_t *q, float *s_a,
                               unsigned flags, bi_stream_t stream)
{
    if (!h || !y || !q || !s_a) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > 65535 || ldy < K) return BI_ERR_INVALID_ARG;
    bi_status st = check_k(K);
    if (st != BI_OK) return st;
    if (!aligned16(h) || !aligned16(y) || !aligned16(q) || !aligned4(s_a) || (ldy % 8) != 0) return BI_ERR_ALIGNMENT;
    const size_t hb = static_cast<size_t>(M) * K * 2;
    const size_t yb = (static_cast<size_t>(M - 1) * ldy + K) * 2;
    if (overlaps(h, hb, y, yb) || overlaps(h, hb, q, static_cast<size_t>(M) * K) ||
        overlaps(h, hb, s_a, 4u * M))
        return BI_ERR_INVALID_ARG;
    st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_residual_quantize(h, y, ldy, M, K, q, s_a, (flags & BI_FLAG_PDL) != 0, stream));
}

bi_status bi_relu_mul_quantize(const uint16_t *gu, int64_t ldgu, int M, int K, int8_t *q, float *s_a,
                               uint16_t *m_out, unsigned flags, bi_stream_t stream)
{
    if (!gu || !q || !s_a) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > 65535 || ldgu < 2LL * K) return BI_ERR_INVALID_ARG;
    bi_status st = check_k(K);
    if (st != BI_OK) return st;
    if (!aligned16(gu) || !aligned16(q) || !aligned4(s_a) || (ldgu % 8) != 0 || (m_out && !aligned16(m_out)))
        return BI_ERR_ALIGNMENT;
    if (m_out && overlaps(m_out, static_cast<size_t>(M) * K * 2, gu, (static_cast<size_t>(M - 1) * ldgu + 2 * K) * 2))
        return BI_ERR_INVALID_ARG;
    st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(
        bi::launch_relu_mul_quantize(gu, ldgu, M, K, q, s_a, m_out, (flags & BI_FLAG_PDL) != 0, stream));
}

bi_status bi_quantize_weight(const float *w, int64_t ldw, int N, int K, int8_t *w_q, float *s_w, bi_stream_t stream)
{
    if (!w || !w_q || !s_w) return BI_ERR_INVALID_ARG;
    if (N < 1 || ldw < K) return BI_ERR_INVALID_ARG;
    bi_status st = check_k(K);
    if (st != BI_OK) return st;
    if (!aligned16(w) || !aligned16(w_q) || !aligned4(s_w) || (ldw % 4) != 0) return BI_ERR_ALIGNMENT;
    st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_quantize_weight(w, ldw, N, K, w_q, s_w, stream));
}

bi_status bi_requant_pow2(const int8_t *w_q, const float *s_w, int N, int K, int8_t *w_q_out, float *s_w_out,
                          bi_stream_t stream)
{
    if (!w_q || !s_w || !w_q_out || !s_w_out || N < 1) return BI_ERR_INVALID_ARG;
    bi_status st = check_k(K);
    if (st != BI_OK) return st;
    if (!aligned16(w_q) || !aligned16(w_q_out) || !aligned4(s_w) || !aligned4(s_w_out)) return BI_ERR_ALIGNMENT;
    // exact aliasing is allowed, partial overlap is not
    const size_t wbytes = static_cast<size_t>(N) * static_cast<size_t>(K);
    const char *a = reinterpret_cast<const char *>(w_q), *b = reinterpret_cast<const char *>(w_q_out);
    if (a != b && a < b + wbytes && b < a + wbytes) return BI_ERR_INVALID_ARG;
    const char *c = reinterpret_cast<const char *>(s_w), *d = reinterpret_cast<const char *>(s_w_out);
    const size_t sbytes = static_cast<size_t>(N) * sizeof(float);
    if (c != d && c < d + sbytes && d < c + sbytes) return BI_ERR_INVALID_ARG;
    st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_requant_pow2(w_q, s_w, N, K, w_q_out, s_w_out, stream));
}

size_t bi_linear_workspace_size(int M, int N, int K)
{
    if (M <= 16) return bi::kWsBytes;
    if (M <= bi::kPrefillTmaMinM || N < 1 || K < 1) return bi::kWsPrefillBytes;
    return bi::kWsPrefillBytes + bi::prefill_f16_bytes(M, K) + bi::prefill_f16_bytes(N, K);
}

size_t bi_lmhead_workspace_size(int M, int N, int K)
{
    (void)M;
    (void)N;
    (void)K;
    return bi::kWsBytes;
}

bi_status bi_linear_w8a8(const int8_t *q, const float *s_a, int M, int K, const int8_t *w_q, const float *s_w, int N,
                         uint16_t *y, void *ws, size_t ws_bytes, unsigned flags, bi_stream_t stream)
{
    bi_status st = check_linear_args(q, s_a, M, K, w_q, s_w, N, ws, ws_bytes);
    if (st != BI_OK) return st;
    if (!y) return BI_ERR_INVALID_ARG;
    if (M <= 16) return run_skinny(q, s_a, M, K, w_q, s_w, N, y, nullptr, ws, flags, stream);

    st = device_info(nullptr);
    if (st != BI_OK) return st;
    // a workspace sized for M <= 16 still works, without splitting tiles
    const bool tail = ws_bytes >= bi::kWsPrefillBytes;
    int32_t *tail_acc = tail ? reinterpret_cast<int32_t *>(static_cast<char *>(ws) + bi::kWsTailAccOff) : nullptr;
    int *tail_cnt = tail ? reinterpret_cast<int *>(static_cast<char *>(ws) + bi::kWsTailCntOff) : nullptr;
    if (M > bi::kPrefillTmaMinM && ws_bytes >= bi_linear_workspace_size(M, N, K)) {
        // room for f16 copies of the operands: the TMA-fed kernel
        bi::PrefillTmaArgs a;
        char *f16 = static_cast<char *>(ws) + bi::kWsPrefillBytes;
        a.q = q;
        a.w_q = w_q;
        a.qf = reinterpret_cast<uint16_t *>(f16);
        a.wf = reinterpret_cast<uint16_t *>(f16 + bi::prefill_f16_bytes(M, K));
        st = bi::host::encode_f16_2d(&a.map_a, a.qf, M, K, 64, 128);
        if (st != BI_OK) return st;
        st = bi::host::encode_f16_2d(&a.map_b, a.wf, N, K, 64, 256);
        if (st != BI_OK) return st;
        a.s_a = s_a;
        a.s_w = s_w;
        a.y = y;
        a.M = M;
        a.N = N;
        a.K = K;
        a.ws = bi::workspace_view(ws);
        a.pdl = (flags & BI_FLAG_PDL) != 0;
        return from_cuda(bi::launch_prefill_tma(a, stream));
    }
    bi::PrefillArgs a;
    a.q = q;
    a.w_q = w_q;
    a.tail_acc = tail_acc;
    a.tail_cnt = tail_cnt;
    a.s_a = s_a;
    a.s_w = s_w;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = bi::workspace_view(ws);
    a.pdl = (flags & BI_FLAG_PDL) != 0;
    return from_cuda(bi::launch_prefill(a, stream));
}

bi_status bi_lmhead_argmax(const int8_t *q, const float *s_a, int M, int K, const int8_t *w_q, const float *s_w,
                           int N, uint16_t *logits, int32_t *argmax, void *ws, size_t ws_bytes, unsigned flags,
                           bi_stream_t stream)
{
    bi_status st = check_linear_args(q, s_a, M, K, w_q, s_w, N, ws, ws_bytes);
    if (st != BI_OK) return st;
    if (!argmax || M > 16) return BI_ERR_INVALID_ARG;
    if (!aligned4(argmax)) return BI_ERR_ALIGNMENT;
    return run_skinny(q, s_a, M, K, w_q, s_w, N, logits, argmax, ws, flags, stream);
}

bi_status bi_greedy_verify(const int32_t *argmax, const int32_t *draft, int M, int32_t *out, bi_stream_t stream)
{
    if (!argmax || !out || M < 1 || M > 65535 || (M > 1 && !draft)) return BI_ERR_INVALID_ARG;
    if (!aligned4(argmax) || !aligned4(out) || (draft && !aligned4(draft))) return BI_ERR_ALIGNMENT;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_greedy_verify(argmax, draft, M, out, stream));
}

bi_status bi_selftest_wait_timeout(void *ws, size_t ws_bytes, bi_stream_t stream)
{
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    if (!ws) {
        // the no-alloc entry point's own scratch
        int *word = nullptr;
        const bi_status sw = bi::host::noalloc_status_word(&word);
        if (sw != BI_OK) return sw;
        return from_cuda(bi::launch_wait_selftest(word, stream));
    }
    if (ws_bytes < bi::kWsBytes || !aligned4(ws)) return BI_ERR_WORKSPACE;
    return from_cuda(bi::launch_wait_selftest(static_cast<int *>(ws), stream));
}

bi_status bi_quantize_weight_q6(const float *w, int64_t ldw, int N, int K, uint8_t *ql, uint8_t *qh, int8_t *sc,
                                float *d, bi_stream_t stream)
{
    if (!w || !ql || !qh || !sc || !d || N < 1 || K < 256 || (K % 256) != 0 || ldw < K) return BI_ERR_INVALID_ARG;
    if (!aligned16(w) || (ldw % 4) != 0 || !aligned16(ql) || !aligned16(qh) || !aligned16(sc) || !aligned4(d))
        return BI_ERR_ALIGNMENT;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_quantize_q6(w, ldw, N, K, ql, qh, sc, d, stream));
}

bi_status bi_quantize_act_blocks(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *d_a,
                                 bi_stream_t stream)
{
    if (!x || !q || !d_a || M < 1 || K < 32 || (K % 32) != 0 || ldx < K) return BI_ERR_INVALID_ARG;
    if (!aligned4(d_a)) return BI_ERR_ALIGNMENT;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_quantize_act_blocks(x, ldx, M, K, q, d_a, stream));
}

bi_status bi_linear_q6(const int8_t *q, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                       const int8_t *sc, const float *d, int N, float *y, unsigned flags, bi_stream_t stream)
{
    if (!q || !d_a || !ql || !qh || !sc || !d || !y) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > 16 || N < 1 || K < 256 || (K % 256) != 0) return BI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(ql) || !aligned16(qh) || !aligned16(sc) || !aligned4(d) || !aligned4(d_a) ||
        !aligned4(y))
        return BI_ERR_ALIGNMENT;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(
        bi::launch_linear_q6(q, d_a, M, K, ql, qh, sc, d, N, y, (flags & BI_FLAG_PDL) != 0, stream));
}

size_t bi_attention_workspace_size(int M, int Hq, int D, int T0)
{
    if (M < 1 || M > kMaxAttnQueries || Hq < 1 || Hq > 65535 || (D != 64 && D != 128) || T0 < 0 ||
        T0 > kMaxAttnPositions - M)
        return 0;
    const int C = bi::attn_chunks(T0, M);
    if (C == 1) return 0;
    return static_cast<size_t>(M) * Hq * C * (D + 4) * sizeof(float);
}

bi_status bi_attention_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v, int M, int Hq, int Hkv, int D,
                              int T0, int S, float scale, uint16_t *o, void *ws, size_t ws_bytes, bi_stream_t stream)
{
    if (!q || !k || !v || !o) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxAttnQueries || Hq < 1 || Hq > 65535 || Hkv < 1 || (Hq % Hkv) != 0 ||
        (D != 64 && D != 128) || T0 < 0 || S < 1 || T0 > S - M || T0 > kMaxAttnPositions - M ||
        static_cast<long long>(M) * (Hq / Hkv) > kMaxAttnRows || !(scale == scale) || scale == INFINITY ||
        scale == -INFINITY)
        return BI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BI_ERR_ALIGNMENT;
    const size_t need = bi_attention_workspace_size(M, Hq, D, T0);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return BI_ERR_WORKSPACE;
    int sms = 0;
    const bi_status st = device_info(&sms);
    if (st != BI_OK) return st;
    bi::AttnArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.ws = static_cast<float *>(ws);
    a.scale = scale;
    a.M = M;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.T0 = T0;
    a.Cmax = bi::attn_chunks(T0, M);
    a.sms = sms;
    return from_cuda(bi::launch_attention(a, stream));
}

bi_status bi_probe_read(const void *buf, size_t bytes, unsigned long long *out, bi_stream_t stream)
{
    if (!buf || !out || bytes == 0 || (bytes & 15u) != 0 || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
        return BI_ERR_INVALID_ARG;
    if (!aligned16(buf)) return BI_ERR_ALIGNMENT;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_probe_read(static_cast<const uint4 *>(buf), bytes / 16, out, stream));
}

bi_status bi_probe_copy(const void *src, void *dst, size_t bytes, bi_stream_t stream)
{
    if (!src || !dst || bytes == 0 || (bytes & 15u) != 0) return BI_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return BI_ERR_ALIGNMENT;
    const char *s = static_cast<const char *>(src), *d = static_cast<const char *>(dst);
    if (s < d + bytes && d < s + bytes) return BI_ERR_INVALID_ARG;     // the copy must not overlap
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_probe_copy(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), bytes / 16,
                                           stream));
}

bi_status bi_selftest_quotient(unsigned long long *out, bi_stream_t stream)
{
    if (!out || (reinterpret_cast<uintptr_t>(out) & 7u) != 0) return BI_ERR_INVALID_ARG;
    const bi_status st = device_info(nullptr);
    if (st != BI_OK) return st;
    return from_cuda(bi::launch_quotient_selftest(out, stream));
}

bi_status bi_workspace_status(void *ws, size_t ws_bytes, bi_stream_t stream)
{
    if (!ws || ws_bytes < bi::kWsBytes) return BI_ERR_WORKSPACE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BI_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
    if (word == bi::DEV_OK) return BI_OK;
    const int zero = 0;
    if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return BI_ERR_CUDA;
    return word == bi::DEV_BAD_PROGRAM ? BI_ERR_INVALID_ARG : BI_ERR_TIMEOUT;
}

}  // extern "C"
