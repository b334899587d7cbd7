"""Helpers for the GPU tests: move generator output to the device and run the
library's entry points on it (through the Python binding, i.e. the C ABI)."""
import numpy as np
import torch

import gen

DEV = "cuda"


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def to_np(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a if dtype is None else a.view(dtype)


def quant_act(bi, x_np: np.ndarray, K: int | None = None, flags: int = 0):
    """x_np: uint16 [M, ldx] bf16 patterns -> device (q int8 [M, K], s_a fp32 [M])."""
    M, ldx = x_np.shape
    K = ldx if K is None else K
    x = to_dev(x_np)
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    bi.bi_quantize_act(x, q, s, K=K, flags=flags)
    return q, s


def weights(bi, w_f32: np.ndarray, pow2: bool):
    """fp32 [N, K] host weights -> device (w_q int8 [N, K], s_w fp32 [N]), quantised
    (and power-of-two requantised) by the library's own kernels."""
    N, K = w_f32.shape
    w = to_dev(w_f32)
    wq = torch.empty((N, K), dtype=torch.int8, device=DEV)
    sw = torch.empty(N, dtype=torch.float32, device=DEV)
    bi.bi_quantize_weight(w, wq, sw)
    if pow2:
        bi.bi_requant_pow2(wq, sw, wq, sw)
    del w
    return wq, sw


def weights_chunked(bi, make_rows, N: int, K: int, pow2: bool, chunk: int = 16384):
    """Same as weights() for matrices too large to hold in fp32 at once.
    make_rows(row0, rows) returns the fp32 rows [row0, row0+rows)."""
    wq = torch.empty((N, K), dtype=torch.int8, device=DEV)
    sw = torch.empty(N, dtype=torch.float32, device=DEV)
    for r0 in range(0, N, chunk):
        r = min(chunk, N - r0)
        part_q, part_s = weights(bi, make_rows(r0, r), pow2)
        wq[r0:r0 + r].copy_(part_q)
        sw[r0:r0 + r].copy_(part_s)
    return wq, sw


def linear(bi, q, s_a, wq, sw, flags: int = 0, ws=None):
    M = q.shape[0]
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.int16, device=DEV)
    if ws is None:
        ws = bi.new_workspace(M, N, q.shape[1])
    bi.bi_linear_w8a8(q, s_a, wq, sw, y, ws, flags=flags)
    return y


def lmhead(bi, q, s_a, wq, sw, want_logits=True, flags: int = 0, ws=None):
    M = q.shape[0]
    N = wq.shape[0]
    logits = torch.empty((M, N), dtype=torch.int16, device=DEV) if want_logits else None
    am = torch.empty(M, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = bi.new_workspace(M, N, q.shape[1])
    bi.bi_lmhead_argmax(q, s_a, wq, sw, logits, am, ws, flags=flags)
    return am, logits


def oracle_weights(oracle, w_f32: np.ndarray, pow2: bool):
    wq, sw = oracle.quantize_weight(w_f32)
    if pow2:
        wq, sw = oracle.requant_pow2(wq, sw)
    return wq, sw


def bf16_f32(a: np.ndarray) -> np.ndarray:
    return gen.bf16_bits_to_f32(a)
