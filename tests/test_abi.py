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


def test_prefill_workspace_tiers(bi):
    """The linear workspace has three sizes: the weight-streaming one (M <= 16),
    plus the split-tile slots for 17 <= M <= 256 (independent of N and K), plus
    room for the f16 copies of q and W (each rounded up to 256 bytes) above
    256 tokens, where the TMA-fed prefill kernel reads them."""
    small = bi.bi_linear_workspace_size(16, 12288, 4096)
    mid = bi.bi_linear_workspace_size(17, 12288, 4096)
    assert mid > small and bi.bi_linear_workspace_size(256, 5, 4096) == mid
    f16 = lambda rows, K: (2 * rows * K + 255) // 256 * 256
    for M, N, K in ((257, 4096, 272), (512, 12288, 4096), (2048, 12288, 4096), (1100, 2500, 1024)):
        assert bi.bi_linear_workspace_size(M, N, K) == mid + f16(M, K) + f16(N, K)


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


def test_fused_quantize_validation(bi):
    R = bi.lib.bi_residual_quantize
    F2 = FAKE + (1 << 20)
    assert R(None, F2, 1024, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG
    assert R(FAKE, F2, 512, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG       # ldy < K
    assert R(FAKE, F2, 1024, 2, 1000, FAKE, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG      # K % 16
    assert R(FAKE, F2 + 8, 1024, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_ALIGNMENT
    assert R(FAKE, F2, 1028, 2, 1024, FAKE, FAKE, 0, None) == bi.BI_ERR_ALIGNMENT        # ldy % 8
    assert R(FAKE, FAKE + 2048, 1024, 2, 1024, F2, F2 + 4096, 0, None) == bi.BI_ERR_INVALID_ARG  # y inside h
    assert R(FAKE, F2, 1024, 2, 1024, FAKE + 1024, F2 + 8192, 0, None) == bi.BI_ERR_INVALID_ARG  # q inside h
    G = bi.lib.bi_relu_mul_quantize
    assert G(FAKE, 1024, 2, 1024, F2, F2 + 4096, None, 0, None) == bi.BI_ERR_INVALID_ARG   # ldgu < 2K
    assert G(FAKE, 2048, 2, 1024, F2 + 4, F2 + 4096, None, 0, None) == bi.BI_ERR_ALIGNMENT
    assert G(FAKE, 2048, 2, 1024, F2, F2 + 4096, FAKE + 4096, 0, None) == bi.BI_ERR_INVALID_ARG  # m_out in gu


def test_program_build_validation(bi):
    F2 = FAKE + (1 << 20)
    prog_bytes = bi.bi_program_bytes(1)
    prog = F2 + (1 << 20)          # never written: validation fails first
    def one(**kw):
        f = dict(kind=bi.BI_OP_RESIDUAL_QUANT, M=2, N=0, K=1024, x=FAKE, ldx=1024, q=F2, s_a=F2 + 4096,
                 w_q=None, s_w=None, y=FAKE + 8192, argmax=None)
        f.update(kw)
        op = bi.bi_op(*[f[k] for k in ("kind", "M", "N", "K", "x", "ldx", "q", "s_a", "w_q", "s_w", "y",
                                       "argmax")])
        return bi.lib.bi_program_build(ctypes.byref(op), 1, prog, prog_bytes)
    assert one(y=None) == bi.BI_ERR_INVALID_ARG                                # residual needs h
    assert one(y=FAKE + 1024) == bi.BI_ERR_INVALID_ARG                         # h overlaps x
    assert one(ldx=1028) == bi.BI_ERR_ALIGNMENT
    assert one(kind=bi.BI_OP_RELU_MUL_QUANT, ldx=1024, y=None) == bi.BI_ERR_INVALID_ARG   # ldx < 2K
    assert one(kind=bi.BI_OP_RELU_MUL_QUANT, ldx=2048, y=FAKE + 2048) == bi.BI_ERR_INVALID_ARG  # m in gu
    assert one(kind=bi.BI_OP_QUANTIZE_ACT, y=FAKE + 8192) == bi.BI_ERR_INVALID_ARG  # plain kind has no y
    assert one(kind=9) == bi.BI_ERR_INVALID_ARG


def test_greedy_verify_validation(bi):
    V = bi.lib.bi_greedy_verify
    assert V(None, FAKE, 4, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert V(FAKE, None, 4, FAKE, None) == bi.BI_ERR_INVALID_ARG          # drafts needed for M > 1
    assert V(FAKE, FAKE, 0, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert V(FAKE + 2, FAKE, 4, FAKE, None) == bi.BI_ERR_ALIGNMENT
    assert V(FAKE, FAKE, 4, FAKE + 1, None) == bi.BI_ERR_ALIGNMENT


def test_block_scaled_validation(bi):
    """The block-scaled entry points: K a multiple of 256 (weights, linear) or
    32 (activation blocks), 1 <= M <= 16 for the linear, aligned pointers."""
    W = bi.lib.bi_quantize_weight_q6
    assert W(FAKE, 1000, 4, 1000, FAKE, FAKE, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG      # K % 256
    assert W(FAKE, 4096, 0, 4096, FAKE, FAKE, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert W(FAKE, 2048, 4, 4096, FAKE, FAKE, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG      # ldw < K
    assert W(FAKE, 4096, 4, 4096, FAKE + 8, FAKE, FAKE, FAKE, None) == bi.BI_ERR_ALIGNMENT
    A = bi.lib.bi_quantize_act_blocks
    assert A(FAKE, 1024, 2, 1000, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG                 # K % 32
    assert A(FAKE, 512, 2, 1024, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG                  # ldx < K
    assert A(None, 1024, 2, 1024, FAKE, FAKE, None) == bi.BI_ERR_INVALID_ARG
    L = bi.lib.bi_linear_q6
    assert L(FAKE, FAKE, 17, 4096, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG   # M > 16
    assert L(FAKE, FAKE, 0, 4096, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG
    assert L(FAKE, FAKE, 4, 4000, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 0, None) == bi.BI_ERR_INVALID_ARG    # K % 256
    assert L(FAKE, FAKE, 4, 4096, FAKE, FAKE, FAKE, FAKE, 8, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert L(FAKE + 4, FAKE, 4, 4096, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 0, None) == bi.BI_ERR_ALIGNMENT


def test_attention_validation(bi):
    """The split-KV attention: D of 64 or 128, Hq a multiple of Hkv, the last
    query's positions inside the cache, a finite scale, k 16-byte aligned and a
    workspace once a query covers more than one chunk of 256 positions; q, k,
    v, o and the workspace 16-byte aligned."""
    Z = bi.lib.bi_attention_workspace_size
    assert Z(8, 32, 128, 100) == 0                       # 108 positions: one chunk
    assert Z(8, 32, 128, 1000) == 8 * 32 * 4 * 132 * 4   # 1008 positions: 4 chunks
    assert Z(1, 1, 64, 256) == 2 * 68 * 4
    assert Z(8, 32, 96, 1000) == 0 and Z(0, 32, 128, 1000) == 0
    F = bi.lib.bi_attention_verify
    args = dict(q=FAKE, k=FAKE, v=FAKE, M=8, Hq=32, Hkv=8, D=128, T0=1000, S=1008, scale=0.088, o=FAKE, ws=None,
                ws_bytes=0, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return F(a["q"], a["k"], a["v"], a["M"], a["Hq"], a["Hkv"], a["D"], a["T0"], a["S"], a["scale"], a["o"],
                 a["ws"], a["ws_bytes"], a["stream"])

    assert call(D=96) == bi.BI_ERR_INVALID_ARG
    assert call(Hkv=5) == bi.BI_ERR_INVALID_ARG
    assert call(S=1007) == bi.BI_ERR_INVALID_ARG          # T0 + M > S
    assert call(M=0) == bi.BI_ERR_INVALID_ARG
    assert call(T0=-1) == bi.BI_ERR_INVALID_ARG
    assert call(T0=(1 << 20) - 7, S=(1 << 20) + 1) == bi.BI_ERR_INVALID_ARG   # more than 2^20 positions
    assert Z(8, 32, 128, (1 << 20) - 7) == 0
    assert call(scale=float("nan")) == bi.BI_ERR_INVALID_ARG
    assert call(scale=float("inf")) == bi.BI_ERR_INVALID_ARG
    assert call(o=None) == bi.BI_ERR_INVALID_ARG
    assert call(k=FAKE + 2) == bi.BI_ERR_ALIGNMENT
    assert call(v=FAKE + 1) == bi.BI_ERR_ALIGNMENT
    assert call(q=FAKE + 8) == bi.BI_ERR_ALIGNMENT and call(o=FAKE + 4) == bi.BI_ERR_ALIGNMENT
    assert call() == bi.BI_ERR_WORKSPACE                  # 4 chunks, no workspace
    assert call(ws=FAKE, ws_bytes=Z(8, 32, 128, 1000) - 1) == bi.BI_ERR_WORKSPACE


def test_probe_validation(bi):
    """The bandwidth probes: a positive multiple of 16 bytes, 16-byte aligned
    buffers, an 8-byte aligned result word, no overlapping copy."""
    R = bi.lib.bi_probe_read
    assert R(FAKE, 0, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert R(FAKE, 100, FAKE, None) == bi.BI_ERR_INVALID_ARG
    assert R(FAKE, 4096, FAKE + 4, None) == bi.BI_ERR_INVALID_ARG
    assert R(FAKE + 8, 4096, FAKE, None) == bi.BI_ERR_ALIGNMENT
    assert R(None, 4096, FAKE, None) == bi.BI_ERR_INVALID_ARG
    C = bi.lib.bi_probe_copy
    assert C(FAKE, FAKE + 4096, 8192, None) == bi.BI_ERR_INVALID_ARG      # overlapping
    assert C(FAKE, FAKE + 8192, 24, None) == bi.BI_ERR_INVALID_ARG
    assert C(FAKE + 4, FAKE + 8192, 4096, None) == bi.BI_ERR_ALIGNMENT
