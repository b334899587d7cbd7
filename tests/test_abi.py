"""Host-side checks of the C ABI: the library loads, exports every entry point
include/bi.h declares, and rejects invalid calls on the host before any launch.

No call here reaches a kernel: every argument set fails validation (fake,
never-dereferenced pointers are used only where validation stops first)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import invariant_quantized_linear_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("bi_quantize_act", "bi_requant_pow2", "bi_linear_w8a8", "bi_lmhead_argmax",
                     "bi_linear_workspace_size", "bi_lmhead_workspace_size", "bi_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(bi):
    lib = ctypes.CDLL(bi.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(bi):
    for s in range(8):
        assert bi.bi_status_string(s).startswith("BI_")
    assert "unknown" in bi.bi_status_string(99)


def test_workspace_sizes_positive(bi):
    for M, N, K in ((1, 1, 16), (8, 151936, 4096), (2048, 12288, 4096)):
        assert bi.bi_linear_workspace_size(M, N, K) > 0
        assert bi.bi_lmhead_workspace_size(M, N, K) > 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced


def _lin(bi, q=FAKE, sa=FAKE, M=2, K=1024, w=FAKE, sw=FAKE, N=1024, y=FAKE, ws=FAKE, wsb=None):
    wsb = bi.bi_linear_workspace_size(M, N, K) if wsb is None else wsb
    return bi.lib.bi_linear_w8a8(q, sa, M, K, w, sw, N, y, ws, wsb, 0, None)


def test_linear_validation(bi):
    assert _lin(bi, q=None) == bi.BI_ERR_INVALID_ARG
    assert _lin(bi, y=None) == bi.BI_ERR_INVALID_ARG
    assert _lin(bi, M=0) == bi.BI_ERR_INVALID_ARG
    assert _lin(bi, N=0) == bi.BI_ERR_INVALID_ARG
    assert _lin(bi, K=8) == bi.BI_ERR_INVALID_ARG
    assert _lin(bi, K=1000) == bi.BI_ERR_INVALID_ARG           # K % 16 != 0
    assert _lin(bi, K=133152) == bi.BI_ERR_INT32_BOUND         # 133152 * 127^2 >= 2^31
    assert _lin(bi, q=FAKE + 8) == bi.BI_ERR_ALIGNMENT
    assert _lin(bi, w=FAKE + 1) == bi.BI_ERR_ALIGNMENT
    assert _lin(bi, sa=FAKE + 2) == bi.BI_ERR_ALIGNMENT
    assert _lin(bi, ws=None) == bi.BI_ERR_WORKSPACE
    assert _lin(bi, wsb=16) == bi.BI_ERR_WORKSPACE


def test_lmhead_validation(bi):
    L = bi.lib.bi_lmhead_argmax
    wsb = bi.bi_lmhead_workspace_size(8, 1024, 1024)
    assert L(FAKE, FAKE, 8, 1024, FAKE, FAKE, 1024, None, None, FAKE, wsb, 0, None) == bi.BI_ERR_INVALID_ARG
    assert L(FAKE, FAKE, 17, 1024, FAKE, FAKE, 1024, None, FAKE, FAKE, wsb, 0, None) == bi.BI_ERR_INVALID_ARG
    assert L(FAKE, FAKE, 8, 1024, FAKE, FAKE, 1024, None, FAKE + 2, FAKE, wsb, 0, None) == bi.BI_ERR_ALIGNMENT
    assert L(FAKE, FAKE, 8, 133152, FAKE, FAKE, 1024, None, FAKE, FAKE, wsb, 0, None) == bi.BI_ERR_INT32_BOUND


def test_quantize_validation(bi):
    Q = bi.lib.bi_quantize_act
    assert Q(None, 1024, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG
    assert Q(FAKE, 512, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG    # ldx < K
    assert Q(FAKE, 1028, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_ALIGNMENT     # ldx % 8 != 0
    assert Q(FAKE + 4, 1024, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_ALIGNMENT
    W = bi.lib.bi_quantize_weight
    assert W(FAKE, 1024, 4, 1000, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert W(FAKE, 1026, 4, 1024, FAKE, FAKE, None) == bi.BI_ERR_ALIGNMENT
    R = bi.lib.bi_requant_pow2
    assert R(FAKE, FAKE, 4, 1024, FAKE + 16, FAKE, None) == bi.BI_ERR_INVALID_ARG  # partial overlap
    assert R(FAKE, FAKE, 4, 1024, FAKE, FAKE + 4, None) == bi.BI_ERR_INVALID_ARG   # scales overlap
    assert R(FAKE, FAKE, 0, 1024, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG


def test_workspace_status_validation(bi):
    assert bi.lib.bi_workspace_status(None, 1 << 20, None) == bi.BI_ERR_WORKSPACE
    assert bi.lib.bi_workspace_status(FAKE, 16, None) == bi.BI_ERR_WORKSPACE


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_call_without_gpu_is_unsupported(bi):
    wsb = bi.bi_linear_workspace_size(2, 1024, 1024)
    assert _lin(bi, wsb=wsb) == bi.BI_ERR_UNSUPPORTED
