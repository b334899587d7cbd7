"""CPU oracle for the batch-invariant W8A8 verify-pass linear (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The library under test never imports it, and it
imports nothing from the library.  Every function is a thin numpy/ctypes
wrapper over the plain C in ``oracle.c``, where each step cites the page it
follows.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16_rne_array.argtypes = [vp, i64, vp]
        L.oracle_f32_to_bf16_rne_array.restype = None
        L.oracle_quantize_act.argtypes = [vp, i64, ci, ci, vp, vp]
        L.oracle_quantize_act.restype = None
        L.oracle_quantize_weight.argtypes = [vp, ci, ci, vp, vp]
        L.oracle_quantize_weight.restype = None
        L.oracle_requant_pow2.argtypes = [vp, vp, ci, ci, vp, vp]
        L.oracle_requant_pow2.restype = None
        L.oracle_linear_w8a8.argtypes = [vp, vp, ci, ci, vp, vp, ci, vp]
        L.oracle_linear_w8a8.restype = ci
        L.oracle_lmhead_argmax.argtypes = [vp, vp, ci, ci, vp, vp, ci, vp, vp]
        L.oracle_lmhead_argmax.restype = ci
        L.oracle_residual_rescale.argtypes = [vp, vp, i64, ci, ci]
        L.oracle_residual_rescale.restype = None
        L.oracle_relu_mul.argtypes = [vp, i64, ci, ci, vp]
        L.oracle_relu_mul.restype = None
        L.oracle_greedy_verify.argtypes = [vp, vp, ci, vp]
        L.oracle_greedy_verify.restype = None
        L.oracle_quantize_q6.argtypes = [vp, ci, ci, vp, vp, vp, vp]
        L.oracle_quantize_q6.restype = None
        L.oracle_q6_code.argtypes = [vp, vp, ci, ci, ci]
        L.oracle_q6_code.restype = ci
        L.oracle_quantize_act_blocks.argtypes = [vp, i64, ci, ci, vp, vp]
        L.oracle_quantize_act_blocks.restype = None
        L.oracle_linear_q6.argtypes = [vp, vp, ci, ci, vp, vp, vp, vp, ci, vp]
        L.oracle_linear_q6.restype = None
        L.oracle_attn_exp.argtypes = [ctypes.c_float]
        L.oracle_attn_exp.restype = ctypes.c_float
        L.oracle_attention.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ctypes.c_float, vp]
        L.oracle_attention.restype = None
        L.oracle_attention_chunk.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ctypes.c_float, vp, vp, vp]
        L.oracle_attention_chunk.restype = None
        L.oracle_attention_merge.argtypes = [ci, vp, vp, vp, ci, vp]
        L.oracle_attention_merge.restype = None
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = ci
        L.oracle_set_num_threads.argtypes = [ci]
        L.oracle_set_num_threads.restype = None
        _LIB = L
    return _LIB


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def bf16_to_f32(b: int) -> float:
    return float(lib().oracle_bf16_to_f32(int(b)))


def f32_to_bf16_rne(f: float) -> int:
    return int(lib().oracle_f32_to_bf16_rne(float(np.float32(f))))


def f32_to_bf16_rne_array(f: np.ndarray) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().oracle_f32_to_bf16_rne_array(f.ctypes.data, f.size, out.ctypes.data)
    return out


def quantize_act(x_bf16: np.ndarray, K: int | None = None):
    """x_bf16: uint16 [M, ldx] bf16 patterns; the first K columns are the row.
    Returns (q int8 [M, K], s_a float32 [M])."""
    x = _c(x_bf16, np.uint16)
    M, ldx = x.shape
    K = ldx if K is None else K
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    lib().oracle_quantize_act(x.ctypes.data, ldx, M, K, q.ctypes.data, s.ctypes.data)
    return q, s


def quantize_weight(w_f32: np.ndarray):
    """Checkpoint-style absmax quantisation: (W_q int8 [N, K], s_w float32 [N])."""
    w = _c(w_f32, np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.int8)
    s = np.empty(N, np.float32)
    lib().oracle_quantize_weight(w.ctypes.data, N, K, q.ctypes.data, s.ctypes.data)
    return q, s


def requant_pow2(wq: np.ndarray, s_w: np.ndarray):
    wq = _c(wq, np.int8)
    s_w = _c(s_w, np.float32)
    N, K = wq.shape
    out = np.empty_like(wq)
    so = np.empty_like(s_w)
    lib().oracle_requant_pow2(wq.ctypes.data, s_w.ctypes.data, N, K, out.ctypes.data, so.ctypes.data)
    return out, so


def linear_w8a8(q: np.ndarray, s_a: np.ndarray, wq: np.ndarray, s_w: np.ndarray) -> np.ndarray:
    """bf16 patterns y [M, N]; raises OverflowError if the int32 bound is broken."""
    q = _c(q, np.int8)
    s_a = _c(s_a, np.float32)
    wq = _c(wq, np.int8)
    s_w = _c(s_w, np.float32)
    M, K = q.shape
    N, K2 = wq.shape
    assert K == K2
    y = np.empty((M, N), np.uint16)
    rc = lib().oracle_linear_w8a8(q.ctypes.data, s_a.ctypes.data, M, K, wq.ctypes.data,
                                  s_w.ctypes.data, N, y.ctypes.data)
    if rc != 0:
        raise OverflowError("an int8 dot product reached 2^31")
    return y


def lmhead_argmax(q, s_a, wq, s_w, want_logits: bool = True):
    q = _c(q, np.int8)
    s_a = _c(s_a, np.float32)
    wq = _c(wq, np.int8)
    s_w = _c(s_w, np.float32)
    M, K = q.shape
    N = wq.shape[0]
    logits = np.empty((M, N), np.uint16) if want_logits else None
    am = np.empty(M, np.int32)
    rc = lib().oracle_lmhead_argmax(q.ctypes.data, s_a.ctypes.data, M, K, wq.ctypes.data,
                                    s_w.ctypes.data, N,
                                    logits.ctypes.data if logits is not None else None,
                                    am.ctypes.data)
    if rc != 0:
        raise OverflowError("an int8 dot product reached 2^31")
    return am, logits


def residual_rescale(h: np.ndarray, y: np.ndarray) -> np.ndarray:
    """New residual stream: bf16_rne(h + y) rescaled by 2^-ilogb(row absmax).
    h: uint16 [M, K]; y: uint16 [M, >= K] (the first K columns are added)."""
    out = np.array(_c(h, np.uint16), copy=True)
    y = _c(y, np.uint16)
    M, K = out.shape
    assert y.shape[0] == M and y.shape[1] >= K
    lib().oracle_residual_rescale(out.ctypes.data, y.ctypes.data, y.shape[1], M, K)
    return out


def relu_mul(gu: np.ndarray, K: int) -> np.ndarray:
    """bf16_rne(relu(g) * u) for g = gu[:, :K], u = gu[:, K:2K]; uint16 [M, K]."""
    gu = _c(gu, np.uint16)
    M, ld = gu.shape
    assert ld >= 2 * K
    out = np.empty((M, K), np.uint16)
    lib().oracle_relu_mul(gu.ctypes.data, ld, M, K, out.ctypes.data)
    return out


def chain_layer(h: np.ndarray, L, q_rows: int):
    """One layer of the chained verify pass on the residual stream h (uint16
    [M, H] bf16).  L: dict of int8 codes and fp32 scales
        "qkv": (wq [q_rows + 2*kv, H], s_w)  q, k, v rows packed in that order,
        "o": (wq [H, q_rows], s_w), "gu": (wq [2*I, H], s_w)  gate rows then up rows,
        "down": (wq [H, I], s_w).
    Steps:  y_qkv = lin(quant(h), qkv);  a = y_qkv[:, :q_rows] (attention
    stand-in; k and v are computed, not used);  h = residual_rescale(h,
    lin(quant(a), o));  y_gu = lin(quant(h), gu);  h = residual_rescale(h,
    lin(quant(relu_mul(y_gu)), down)).  Returns (new h, dict of every linear
    output and of h after the first residual)."""
    q, s = quantize_act(h)
    y_qkv = linear_w8a8(q, s, *L["qkv"])
    qa, sa = quantize_act(np.ascontiguousarray(y_qkv[:, :q_rows]))
    y_o = linear_w8a8(qa, sa, *L["o"])
    h_mid = residual_rescale(h, y_o)
    q, s = quantize_act(h_mid)
    y_gu = linear_w8a8(q, s, *L["gu"])
    inter = L["gu"][0].shape[0] // 2
    mq, ms = quantize_act(relu_mul(y_gu, inter))
    y_d = linear_w8a8(mq, ms, *L["down"])
    h_new = residual_rescale(h_mid, y_d)
    return h_new, {"qkv": y_qkv, "o": y_o, "h_mid": h_mid, "gu": y_gu, "down": y_d, "h": h_new}


def verify_pass(h0: np.ndarray, layers, head, q_rows: int, record: bool = False):
    """Chained verify pass: chain_layer over `layers` from h0, then the greedy
    head (wq [V, H], s_w) on quant(h).  Returns (argmax int32 [M], final h,
    per-layer records of chain_layer if asked, else [])."""
    h = np.array(_c(h0, np.uint16), copy=True)
    recs = []
    for L in layers:
        h, rec = chain_layer(h, L, q_rows)
        if record:
            recs.append(rec)
    q, s = quantize_act(h)
    am, _ = lmhead_argmax(q, s, *head, want_logits=False)
    return am, h, recs


def greedy_verify(argmax: np.ndarray, draft: np.ndarray):
    """(accepted count L, next token) for the argmax rows [M] of a verify pass
    whose inputs after the first were the drafted tokens draft [M - 1]."""
    am = _c(argmax, np.int32)
    M = am.shape[0]
    d = _c(draft if len(draft) else np.zeros(1, np.int32), np.int32)
    assert len(draft) == M - 1
    out = np.empty(2, np.int32)
    lib().oracle_greedy_verify(am.ctypes.data, d.ctypes.data, M, out.ctypes.data)
    return int(out[0]), int(out[1])


# ------------------------------------------------------------ block-scaled variant
# ("why speculative decoding changed my output", "the mat-vec kernel"; the
# format and the fixed order of adds are defined in oracle.c)

def quantize_q6(w_f32: np.ndarray):
    """fp32 W [N, K] (K % 256 == 0) -> (ql uint8 [N, K/2], qh uint8 [N, K/4],
    sc int8 [N, K/16], d fp32 [N, K/256])."""
    w = _c(w_f32, np.float32)
    N, K = w.shape
    assert K % 256 == 0
    ql = np.zeros((N, K // 2), np.uint8)
    qh = np.zeros((N, K // 4), np.uint8)
    sc = np.zeros((N, K // 16), np.int8)
    d = np.zeros((N, K // 256), np.float32)
    lib().oracle_quantize_q6(w.ctypes.data, N, K, ql.ctypes.data, qh.ctypes.data, sc.ctypes.data, d.ctypes.data)
    return ql, qh, sc, d


def q6_codes(ql: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """The int8 codes [N, K] of a block-scaled matrix, one call per element."""
    ql, qh = _c(ql, np.uint8), _c(qh, np.uint8)
    N, K = ql.shape[0], 2 * ql.shape[1]
    L = lib()
    return np.array([[L.oracle_q6_code(ql.ctypes.data, qh.ctypes.data, K, n, k) for k in range(K)]
                     for n in range(N)], np.int8)


def quantize_act_blocks(x_bf16: np.ndarray):
    """bf16 x [M, K] (uint16 patterns, K % 32 == 0) -> (q int8 [M, K], d_a fp32 [M, K/32])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // 32), np.float32)
    lib().oracle_quantize_act_blocks(x.ctypes.data, K, M, K, q.ctypes.data, d.ctypes.data)
    return q, d


def linear_q6(qa, d_a, ql, qh, sc, d) -> np.ndarray:
    """y fp32 [M, N] of the block-scaled linear, in the fixed order of adds."""
    qa, d_a = _c(qa, np.int8), _c(d_a, np.float32)
    ql, qh, sc, d = _c(ql, np.uint8), _c(qh, np.uint8), _c(sc, np.int8), _c(d, np.float32)
    M, K = qa.shape
    N = ql.shape[0]
    y = np.empty((M, N), np.float32)
    lib().oracle_linear_q6(qa.ctypes.data, d_a.ctypes.data, M, K, ql.ctypes.data, qh.ctypes.data, sc.ctypes.data,
                           d.ctypes.data, N, y.ctypes.data)
    return y


# ------------------------------------------------------------ split-KV attention
# ("My speculative decoder got slower", split-KV attention; "why speculative
# decoding changed my output", "attention"; the readings are in oracle.c)

def attn_exp(x: float) -> float:
    """The attention's exp e(x) for x <= 0, as defined in oracle.c."""
    return float(lib().oracle_attn_exp(x))


def attention(q, k, v, T0: int, scale: float) -> np.ndarray:
    """q bf16 [M, Hq, D], k / v bf16 [S, Hkv, D] (S >= T0 + M) -> o bf16 [M, Hq, D]:
    query m attends to positions 0 .. T0 + m, in 256-position chunks merged in order."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    M, Hq, D = q.shape
    Hkv = k.shape[1]
    assert k.shape[0] >= T0 + M and Hq % Hkv == 0
    o = np.empty((M, Hq, D), np.uint16)
    lib().oracle_attention(q.ctypes.data, k.ctypes.data, v.ctypes.data, M, Hq, Hkv, D, T0, scale, o.ctypes.data)
    return o


def attention_chunk(q_row, k, v, hk: int, t0: int, t1: int, scale: float):
    """One chunk (positions t0 .. t1 - 1, at most 256) of kv head hk for one
    query row q_row bf16 [D]: (mx, l, a fp32 [D])."""
    q_row, k, v = _c(q_row, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    D = q_row.shape[0]
    assert 0 <= t0 < t1 <= k.shape[0] and t1 - t0 <= 256
    mx, l = np.zeros(1, np.float32), np.zeros(1, np.float32)
    a = np.empty(D, np.float32)
    lib().oracle_attention_chunk(q_row.ctypes.data, k.ctypes.data, v.ctypes.data, k.shape[1], hk, D, t0, t1, scale,
                                 mx.ctypes.data, l.ctypes.data, a.ctypes.data)
    return mx[0], l[0], a


def attention_merge(mx, l, a) -> np.ndarray:
    """The in-order merge of C chunk results: mx [C], l [C], a [C, D] (fp32) -> o bf16 [D]."""
    mx, l, a = _c(mx, np.float32), _c(l, np.float32), _c(a, np.float32)
    C, D = a.shape
    o = np.empty(D, np.uint16)
    lib().oracle_attention_merge(C, mx.ctypes.data, l.ctypes.data, a.ctypes.data, D, o.ctypes.data)
    return o


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the parallel loops (results do not depend on it)."""
    lib().oracle_set_num_threads(int(n))
