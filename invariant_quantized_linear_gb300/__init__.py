"""Batch-invariant verify pass for GB300 (sm_103a): Python binding of the W8A8
linear and LM head, the verify-pass executor, the block-scaled variant and the
split-KV verify attention.

A thin ctypes layer over ``libbi.so`` (C ABI declared in ``include/bi.h``).
Each function has the name of the C entry point it calls and only marshals
arguments: tensor pointers, shapes and the current CUDA stream.  All
arithmetic runs in the library's CUDA kernels; there is no other code path.
If ``libbi.so`` is missing or fails to load, importing this package raises.

PyTorch supplies device memory and streams.  bf16 tensors may be passed as
``torch.bfloat16`` or as their ``int16``/``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbi.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libbi.so is not built: run invariant_quantized_linear_gb300/build.py "
                      "(or __graft_entry__.build()) first")

lib = ctypes.CDLL(LIB_PATH)

_vp, _i64, _ci, _cu, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
lib.bi_status_string.argtypes = [_ci]
lib.bi_status_string.restype = ctypes.c_char_p
lib.bi_quantize_act.argtypes = [_vp, _i64, _ci, _ci, _vp, _vp, _cu, _vp]
lib.bi_quantize_act.restype = _ci
lib.bi_residual_quantize.argtypes = [_vp, _vp, _i64, _ci, _ci, _vp, _vp, _cu, _vp]
lib.bi_residual_quantize.restype = _ci
lib.bi_relu_mul_quantize.argtypes = [_vp, _i64, _ci, _ci, _vp, _vp, _vp, _cu, _vp]
lib.bi_relu_mul_quantize.restype = _ci
lib.bi_quantize_weight.argtypes = [_vp, _i64, _ci, _ci, _vp, _vp, _vp]
lib.bi_quantize_weight.restype = _ci
lib.bi_requant_pow2.argtypes = [_vp, _vp, _ci, _ci, _vp, _vp, _vp]
lib.bi_requant_pow2.restype = _ci
lib.bi_linear_workspace_size.argtypes = [_ci, _ci, _ci]
lib.bi_linear_workspace_size.restype = _sz
lib.bi_lmhead_workspace_size.argtypes = [_ci, _ci, _ci]
lib.bi_lmhead_workspace_size.restype = _sz
lib.bi_linear_w8a8.argtypes = [_vp, _vp, _ci, _ci, _vp, _vp, _ci, _vp, _vp, _sz, _cu, _vp]
lib.bi_linear_w8a8.restype = _ci
lib.bi_lmhead_argmax.argtypes = [_vp, _vp, _ci, _ci, _vp, _vp, _ci, _vp, _vp, _vp, _sz, _cu, _vp]
lib.bi_lmhead_argmax.restype = _ci
lib.bi_greedy_verify.argtypes = [_vp, _vp, _ci, _vp, _vp]
lib.bi_greedy_verify.restype = _ci
lib.bi_selftest_wait_timeout.argtypes = [_vp, _sz, _vp]
lib.bi_selftest_wait_timeout.restype = _ci
lib.bi_selftest_quotient.argtypes = [_vp, _vp]
lib.bi_selftest_quotient.restype = _ci
lib.bi_workspace_status.argtypes = [_vp, _sz, _vp]
lib.bi_workspace_status.restype = _ci
lib.bi_linear_w8a8_noalloc.argtypes = [_vp, _vp, _ci, _ci, _vp, _vp, _ci, _vp, _cu, _vp]
lib.bi_linear_w8a8_noalloc.restype = _ci
lib.bi_linear_w8a8_noalloc_status.argtypes = [_vp]
lib.bi_linear_w8a8_noalloc_status.restype = _ci
lib.bi_quantize_weight_q6.argtypes = [_vp, _i64, _ci, _ci, _vp, _vp, _vp, _vp, _vp]
lib.bi_quantize_weight_q6.restype = _ci
lib.bi_quantize_act_blocks.argtypes = [_vp, _i64, _ci, _ci, _vp, _vp, _vp]
lib.bi_quantize_act_blocks.restype = _ci
lib.bi_linear_q6.argtypes = [_vp, _vp, _ci, _ci, _vp, _vp, _vp, _vp, _ci, _vp, _cu, _vp]
lib.bi_linear_q6.restype = _ci
lib.bi_attention_workspace_size.argtypes = [_ci, _ci, _ci, _ci]
lib.bi_attention_workspace_size.restype = _sz
lib.bi_attention_verify.argtypes = [_vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, ctypes.c_float, _vp, _vp, _sz,
                                    _vp]
lib.bi_attention_verify.restype = _ci
lib.bi_probe_read.argtypes = [_vp, _sz, _vp, _vp]
lib.bi_probe_read.restype = _ci
lib.bi_probe_copy.argtypes = [_vp, _vp, _sz, _vp]
lib.bi_probe_copy.restype = _ci

lib.bi_program_bytes.argtypes = [_ci]
lib.bi_program_bytes.restype = _sz
lib.bi_program_workspace_size.argtypes = []
lib.bi_program_workspace_size.restype = _sz


class bi_op(ctypes.Structure):
    """One op of a verify-pass program (struct bi_op of include/bi.h)."""
    _fields_ = [("kind", _ci), ("M", _ci), ("N", _ci), ("K", _ci),
                ("x", _vp), ("ldx", _i64), ("q", _vp), ("s_a", _vp),
                ("w_q", _vp), ("s_w", _vp), ("y", _vp), ("argmax", _vp),
                ("draft", _vp), ("accept", _vp)]


lib.bi_program_build.argtypes = [ctypes.POINTER(bi_op), _ci, _vp, _sz]
lib.bi_program_build.restype = _ci
lib.bi_program_run.argtypes = [_vp, _ci, _vp, _sz, _vp]
lib.bi_program_run.restype = _ci

BI_OP_QUANTIZE_ACT = 1
BI_OP_LINEAR = 2
BI_OP_LMHEAD = 3
BI_OP_RESIDUAL_QUANT = 4
BI_OP_RELU_MUL_QUANT = 5

BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_ALIGNMENT = 2
BI_ERR_INT32_BOUND = 3
BI_ERR_WORKSPACE = 4
BI_ERR_UNSUPPORTED = 5
BI_ERR_TIMEOUT = 6
BI_ERR_CUDA = 7
BI_FLAG_PDL = 1


class BiError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, lib.bi_status_string(status).decode()))


def _check(status: int, what: str) -> None:
    if status != BI_OK:
        raise BiError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def bi_status_string(status: int) -> str:
    return lib.bi_status_string(status).decode()


def bi_quantize_act(x: torch.Tensor, q: torch.Tensor, s_a: torch.Tensor, K: int | None = None,
                    flags: int = 0, stream=None) -> None:
    """x: bf16 [M, ldx] (row stride ldx = x.stride(0)); q: int8 [M, K]; s_a: fp32 [M]."""
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    _check(lib.bi_quantize_act(_ptr(x), x.stride(0), M, K, _ptr(q), _ptr(s_a), flags, _stream(stream)),
           "bi_quantize_act")


def bi_residual_quantize(h: torch.Tensor, y: torch.Tensor, q: torch.Tensor, s_a: torch.Tensor,
                         flags: int = 0, stream=None) -> None:
    """h: bf16 [M, K] contiguous, updated in place; y: bf16 [M, >= K] (row stride
    y.stride(0)), first K columns added; q: int8 [M, K]; s_a: fp32 [M]."""
    M, K = h.shape
    assert h.stride(0) == K
    _check(lib.bi_residual_quantize(_ptr(h), _ptr(y), y.stride(0), M, K, _ptr(q), _ptr(s_a), flags,
                                    _stream(stream)), "bi_residual_quantize")


def bi_relu_mul_quantize(gu: torch.Tensor, K: int, q: torch.Tensor, s_a: torch.Tensor,
                         m_out: torch.Tensor | None = None, flags: int = 0, stream=None) -> None:
    """gu: bf16 [M, >= 2K] packed gate|up (row stride gu.stride(0)); q: int8 [M, K];
    s_a: fp32 [M]; m_out: bf16 [M, K] or None."""
    M = gu.shape[0]
    _check(lib.bi_relu_mul_quantize(_ptr(gu), gu.stride(0), M, K, _ptr(q), _ptr(s_a), _ptr(m_out), flags,
                                    _stream(stream)), "bi_relu_mul_quantize")


def bi_quantize_weight(w: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor, stream=None) -> None:
    N, K = w.shape
    _check(lib.bi_quantize_weight(_ptr(w), w.stride(0), N, K, _ptr(w_q), _ptr(s_w), _stream(stream)),
           "bi_quantize_weight")


def bi_requant_pow2(w_q: torch.Tensor, s_w: torch.Tensor, w_q_out: torch.Tensor, s_w_out: torch.Tensor,
                    stream=None) -> None:
    N, K = w_q.shape
    _check(lib.bi_requant_pow2(_ptr(w_q), _ptr(s_w), N, K, _ptr(w_q_out), _ptr(s_w_out), _stream(stream)),
           "bi_requant_pow2")


def bi_linear_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib.bi_linear_workspace_size(M, N, K))


def bi_lmhead_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib.bi_lmhead_workspace_size(M, N, K))


def bi_linear_w8a8(q: torch.Tensor, s_a: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor,
                   y: torch.Tensor, ws: torch.Tensor, flags: int = 0, stream=None) -> None:
    M, K = q.shape
    N = w_q.shape[0]
    _check(lib.bi_linear_w8a8(_ptr(q), _ptr(s_a), M, K, _ptr(w_q), _ptr(s_w), N, _ptr(y), _ptr(ws),
                              ws.numel() * ws.element_size(), flags, _stream(stream)), "bi_linear_w8a8")


def bi_lmhead_argmax(q: torch.Tensor, s_a: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor,
                     logits: torch.Tensor | None, argmax: torch.Tensor, ws: torch.Tensor,
                     flags: int = 0, stream=None) -> None:
    M, K = q.shape
    N = w_q.shape[0]
    _check(lib.bi_lmhead_argmax(_ptr(q), _ptr(s_a), M, K, _ptr(w_q), _ptr(s_w), N, _ptr(logits),
                                _ptr(argmax), _ptr(ws), ws.numel() * ws.element_size(), flags,
                                _stream(stream)), "bi_lmhead_argmax")


def bi_quantize_weight_q6(w: torch.Tensor, ql: torch.Tensor, qh: torch.Tensor, sc: torch.Tensor, d: torch.Tensor,
                          stream=None) -> None:
    """w fp32 [N, K] -> block-scaled ql uint8 [N, K/2], qh uint8 [N, K/4], sc int8 [N, K/16], d fp32 [N, K/256]."""
    N, K = w.shape
    _check(lib.bi_quantize_weight_q6(_ptr(w), w.stride(0), N, K, _ptr(ql), _ptr(qh), _ptr(sc), _ptr(d),
                                     _stream(stream)), "bi_quantize_weight_q6")


def bi_quantize_act_blocks(x: torch.Tensor, q: torch.Tensor, d_a: torch.Tensor, stream=None) -> None:
    """x bf16 bits [M, K] (int16/uint16/bfloat16) -> q int8 [M, K], d_a fp32 [M, K/32]."""
    M, K = x.shape
    _check(lib.bi_quantize_act_blocks(_ptr(x), x.stride(0), M, K, _ptr(q), _ptr(d_a), _stream(stream)),
           "bi_quantize_act_blocks")


def bi_linear_q6(q: torch.Tensor, d_a: torch.Tensor, ql: torch.Tensor, qh: torch.Tensor, sc: torch.Tensor,
                 d: torch.Tensor, y: torch.Tensor, flags: int = 0, stream=None) -> None:
    """y fp32 [M, N] = the block-scaled linear (1 <= M <= 16)."""
    M, K = q.shape
    N = ql.shape[0]
    _check(lib.bi_linear_q6(_ptr(q), _ptr(d_a), M, K, _ptr(ql), _ptr(qh), _ptr(sc), _ptr(d), N, _ptr(y), flags,
                            _stream(stream)), "bi_linear_q6")


def bi_attention_workspace_size(M: int, Hq: int, D: int, T0: int) -> int:
    return int(lib.bi_attention_workspace_size(M, Hq, D, T0))


def bi_attention_verify(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, T0: int, scale: float, o: torch.Tensor,
                        ws: torch.Tensor | None = None, stream=None) -> None:
    """Split-KV verify attention: q bf16 [M, Hq, D], k/v bf16 [S, Hkv, D]
    (contiguous), o bf16 [M, Hq, D] out; query m sees positions 0 .. T0 + m.
    ws: device buffer of at least bi_attention_workspace_size(M, Hq, D, T0)
    bytes, or None when that is 0."""
    M, Hq, D = q.shape
    S, Hkv = k.shape[0], k.shape[1]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.bi_attention_verify(_ptr(q), _ptr(k), _ptr(v), M, Hq, Hkv, D, T0, S, scale, _ptr(o), _ptr(ws),
                                   nbytes, _stream(stream)), "bi_attention_verify")


def bi_probe_read(buf: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Read all of `buf` once (bandwidth probe); out: int64 device tensor, receives the xor of its 64-bit words."""
    _check(lib.bi_probe_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(out), _stream(stream)),
           "bi_probe_read")


def bi_probe_copy(src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """dst = src (bandwidth probe), same byte size, not overlapping."""
    _check(lib.bi_probe_copy(_ptr(src), _ptr(dst), src.numel() * src.element_size(), _stream(stream)),
           "bi_probe_copy")


def bi_linear_w8a8_noalloc(q: torch.Tensor, s_a: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor,
                           y: torch.Tensor, flags: int = 0, stream=None) -> None:
    """bi_linear_w8a8 without a workspace argument, for callers that cannot
    allocate device memory: the library keeps the kernel's scratch in a fixed
    array of its own (M <= 16; calls on one stream only, never overlapping)."""
    M, K = q.shape
    N = w_q.shape[0]
    _check(lib.bi_linear_w8a8_noalloc(_ptr(q), _ptr(s_a), M, K, _ptr(w_q), _ptr(s_w), N, _ptr(y), flags,
                                      _stream(stream)), "bi_linear_w8a8_noalloc")


def bi_linear_w8a8_noalloc_status(stream=None) -> int:
    """Status of the no-alloc entry point's scratch after `stream`: BI_OK, or
    BI_ERR_TIMEOUT (once; the scratch is then restored)."""
    return int(lib.bi_linear_w8a8_noalloc_status(_stream(stream)))


def bi_program_bytes(n_ops: int) -> int:
    return int(lib.bi_program_bytes(n_ops))


def bi_program_workspace_size() -> int:
    return int(lib.bi_program_workspace_size())


def bi_program_build(ops, program: torch.Tensor) -> None:
    """ops: a sequence of bi_op; program: device uint8 tensor of at least
    bi_program_bytes(len(ops)) bytes, 128-byte aligned."""
    arr = (bi_op * len(ops))(*ops)
    _check(lib.bi_program_build(arr, len(ops), _ptr(program), program.numel() * program.element_size()),
           "bi_program_build")


def bi_program_run(program: torch.Tensor, max_tokens: int, ws: torch.Tensor, stream=None) -> None:
    _check(lib.bi_program_run(_ptr(program), max_tokens, _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "bi_program_run")


def op_quantize_act(x: torch.Tensor, q: torch.Tensor, s_a: torch.Tensor, K: int | None = None) -> bi_op:
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    return bi_op(BI_OP_QUANTIZE_ACT, M, 0, K, _ptr(x), x.stride(0), _ptr(q), _ptr(s_a), None, None, None, None)


def op_residual_quant(h: torch.Tensor, y: torch.Tensor, q: torch.Tensor, s_a: torch.Tensor) -> bi_op:
    """h (in/out, contiguous [M, K]) <- rescale(bf16(h + y[:, :K])); q, s_a <- quant(h)."""
    M, K = h.shape
    assert h.stride(0) == K
    return bi_op(BI_OP_RESIDUAL_QUANT, M, 0, K, _ptr(y), y.stride(0), _ptr(q), _ptr(s_a), None, None, _ptr(h), None)


def op_relu_mul_quant(gu: torch.Tensor, K: int, q: torch.Tensor, s_a: torch.Tensor,
                      m_out: torch.Tensor | None = None) -> bi_op:
    """q, s_a <- quant(bf16(relu(gu[:, :K]) * gu[:, K:2K])); m_out receives the product if given."""
    M = gu.shape[0]
    return bi_op(BI_OP_RELU_MUL_QUANT, M, 0, K, _ptr(gu), gu.stride(0), _ptr(q), _ptr(s_a), None, None,
                 _ptr(m_out), None)


def op_linear(q: torch.Tensor, s_a: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor, y: torch.Tensor) -> bi_op:
    M, K = q.shape
    return bi_op(BI_OP_LINEAR, M, w_q.shape[0], K, None, 0, _ptr(q), _ptr(s_a), _ptr(w_q), _ptr(s_w), _ptr(y), None)


def op_lmhead(q: torch.Tensor, s_a: torch.Tensor, w_q: torch.Tensor, s_w: torch.Tensor,
              logits: torch.Tensor | None, argmax: torch.Tensor, draft: torch.Tensor | None = None,
              accept: torch.Tensor | None = None) -> bi_op:
    """LM head; with `accept` (int32 [2]) also greedy verification against `draft` (int32 [M - 1])."""
    M, K = q.shape
    return bi_op(BI_OP_LMHEAD, M, w_q.shape[0], K, None, 0, _ptr(q), _ptr(s_a), _ptr(w_q), _ptr(s_w),
                 _ptr(logits), _ptr(argmax), _ptr(draft), _ptr(accept))


def new_program(n_ops: int, device="cuda") -> torch.Tensor:
    """Device memory for a program of n_ops ops (128-byte aligned)."""
    n = bi_program_bytes(n_ops)
    buf = torch.empty(n + 128, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 128
    return buf[off:off + n]


def bi_greedy_verify(argmax: torch.Tensor, draft: torch.Tensor | None, out: torch.Tensor, stream=None) -> None:
    """argmax int32 [M], draft int32 [M - 1] (or None when M == 1), out int32 [2]:
    accepted draft count and next token."""
    _check(lib.bi_greedy_verify(_ptr(argmax), _ptr(draft), argmax.shape[0], _ptr(out), _stream(stream)),
           "bi_greedy_verify")


def bi_selftest_wait_timeout(ws: torch.Tensor, stream=None) -> None:
    """Launch a bounded wait that nothing satisfies (about 2 s); the workspace
    status then reads BI_ERR_TIMEOUT."""
    _check(lib.bi_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "bi_selftest_wait_timeout")


def bi_selftest_quotient(out: torch.Tensor, stream=None) -> None:
    """out int64 [3] on the device: pairs checked, mismatches, one mismatching
    (amax bits << 16 | v bits) of the executor's quotient against IEEE division."""
    assert out.dtype == torch.int64 and out.numel() >= 3 and out.is_cuda
    _check(lib.bi_selftest_quotient(_ptr(out), _stream(stream)), "bi_selftest_quotient")


def bi_workspace_status(ws: torch.Tensor, stream=None) -> int:
    """BI_OK or BI_ERR_TIMEOUT (returned, not raised); clears the status word."""
    return int(lib.bi_workspace_status(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def new_workspace(M: int, N: int, K: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace large enough for bi_linear_w8a8 and bi_lmhead_argmax."""
    n = max(bi_linear_workspace_size(M, N, K), bi_lmhead_workspace_size(M, N, K))
    return torch.zeros(n, dtype=torch.uint8, device=device)
