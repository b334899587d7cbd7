"""GPU parity of bi_linear_w8a8 (weight-streaming and prefill kernels) against
the CPU oracle, bit for bit, plus batch invariance across M."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV, linear, oracle_weights, quant_act, to_dev, to_np, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _case(seed, M, N, K, pow2, outliers=True):
    x = gen.act_bf16(seed, 1, M, K, outliers=gen.outlier_channels(seed, K) if outliers else (), gain=20.0)
    w = gen.weight_f32(seed, 0, 0, N, K)
    return x, w


def _check_linear(bi, x, w, pow2, flags=0):
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, pow2)
    want = oracle.linear_w8a8(q_o, s_o, wq_o, sw_o)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, pow2)
    got = to_np(linear(bi, q, s, wq, sw, flags=flags))
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, "%d mismatches, first at %s" % (len(bad), bad[:4].tolist())
    return got


# shapes span several row blocks (64 rows) and units (256 bytes of K), with
# ragged tails in N and K; M covers both token tiles of the skinny kernel and
# the prefill kernel (M > 16)
SKINNY = [(1, 1, 16), (2, 17, 48), (3, 100, 272), (8, 1000, 1024), (9, 1024, 1040), (16, 333, 4096),
          (4, 4096, 4096), (5, 64, 12288), (1, 12288, 256)]
PREFILL = [(17, 130, 256), (33, 257, 1024), (130, 300, 528), (200, 1000, 4096), (64, 64, 16),
           # exact fp32 chunks of 1024 K: a one-step last chunk, N tails on and
           # off the 16-byte store path, several token and weight tiles
           (129, 520, 1040), (300, 776, 3088)]
# above 256 tokens the TMA-fed kernel runs (f16 copies in the workspace); its
# last wave is cut into slices of 32 / 64 / 96 weight rows depending on how
# many tiles it holds, and a ragged q copy ends in a partial 512-code block
PREFILL_TMA = [(384, 300, 528), (400, 520, 1040), (520, 776, 3088), (257, 4096, 272), (1100, 2500, 1024)]


@pytest.mark.parametrize("M,N,K", SKINNY + PREFILL + PREFILL_TMA)
@pytest.mark.parametrize("pow2", [True, False])
def test_linear_matches_oracle(bi, M, N, K, pow2):
    x, w = _case(M * 7 + N, M, N, K, pow2)
    _check_linear(bi, x, w, pow2)


@pytest.mark.parametrize("M,N,K", PREFILL_TMA)
def test_prefill_kernels_agree(bi, M, N, K):
    """The TMA-fed prefill kernel above 256 tokens (f16 copies of the operands
    in the workspace) and the kernel that converts the codes in its tile loop
    (a workspace without room for the copies) give the same bits."""
    x, w = _case(M * 5 + N, M, N, K, True)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, True)
    full = bi.new_workspace(M, N, K)
    conv = bi.new_workspace(200, N, K)            # the size for M <= 256: no room for f16 copies
    assert conv.numel() < full.numel()
    assert torch.equal(linear(bi, q, s, wq, sw, ws=full), linear(bi, q, s, wq, sw, ws=conv))


def test_linear_near_int32_bound(bi):
    """K = 133136 (the largest multiple of 16 under the int32 bound) with
    all-127 operands: |acc| reaches 2,147,350,544 and must not wrap."""
    K, N = 133136, 70
    x = np.full((2, K), 0x42FE, np.uint16)        # 127.0 in bf16 -> q = 127
    x[1, ::2] = 0xC2FE                            # -127.0
    w = np.full((N, K), 0.02, np.float32)
    w[1::2, ::3] = -0.02
    _check_linear(bi, x, w, pow2=False)
    x3 = np.concatenate([x] * 10)[:20]            # prefill path too
    _check_linear(bi, x3, w, pow2=False)


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 12288), (333, 1040)])
def test_rows_are_batch_invariant(bi, N, K):
    """Row r of an M-row call equals the one-row call on row r alone, for
    M = 1..16 (both token tiles) and prefill sizes."""
    Ms = list(range(1, 17)) + [17, 64, 130]
    xall = gen.act_bf16(77, 1, max(Ms), K, outliers=gen.outlier_channels(77, K), gain=20.0)
    wq, sw = weights(bi, gen.weight_f32(77, 0, 0, N, K), pow2=True)
    single = []
    for r in range(max(Ms)):
        q, s = quant_act(bi, xall[r:r + 1])
        single.append(linear(bi, q, s, wq, sw))
    single = torch.cat(single)
    for M in Ms:
        q, s = quant_act(bi, xall[:M])
        y = linear(bi, q, s, wq, sw)
        assert torch.equal(y, single[:M]), M


def test_prefill_split_tiles_leave_workspace_zeroed(bi):
    """M = 200, N = 1000, K = 4096: 8 tiles on the GPU's SMs are split along K
    (the last wave is less than half full); the split tiles' counters return
    to zero (their partial-sum slots are scratch), and a workspace sized for
    M <= 16 (no split) gives the same bits."""
    M, N, K = 200, 1000, 4096
    x_np, w = _case(13, M, N, K, True)
    wq, sw = weights(bi, w, pow2=True)
    q, s = quant_act(bi, x_np)
    ws = bi.new_workspace(M, N, K)
    assert ws.numel() > bi.new_workspace(16, N, K).numel()
    ys = [linear(bi, q, s, wq, sw, ws=ws) for _ in range(3)]
    y_small = linear(bi, q, s, wq, sw, ws=bi.new_workspace(16, N, K))
    torch.cuda.synchronize()
    assert all(torch.equal(y, y_small) for y in ys)
    small = bi.new_workspace(16, N, K).numel()
    slots = 96 * 256 * 128 * 4
    counters = small + slots + 768          # after them: the f16 operand copies (scratch)
    assert int(ws[:small].count_nonzero()) == 0 and int(ws[small + slots:counters].count_nonzero()) == 0
    assert bi.bi_workspace_status(ws) == bi.BI_OK
    # without room for the f16 copies the converting kernel runs, with the split
    y_conv = linear(bi, q, s, wq, sw, ws=torch.zeros(counters, dtype=torch.uint8, device="cuda"))
    assert torch.equal(y_conv, y_small)


def test_pdl_flag_and_graph_capture_same_bits(bi):
    """PDL launches, and a CUDA graph of quantise + linear with PDL, give the
    same bits as plain launches."""
    M, N, K = 8, 4096, 4096
    x_np, w = _case(5, M, N, K, True)
    wq, sw = weights(bi, w, pow2=True)
    q, s = quant_act(bi, x_np)
    ref = linear(bi, q, s, wq, sw)
    ws = bi.new_workspace(M, N, K)
    y_pdl = linear(bi, q, s, wq, sw, flags=bi.BI_FLAG_PDL, ws=ws)
    assert torch.equal(ref, y_pdl)

    x = to_dev(x_np)
    q2 = torch.empty_like(q)
    s2 = torch.empty_like(s)
    y2 = torch.empty_like(ref)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        bi.bi_quantize_act(x, q2, s2, flags=bi.BI_FLAG_PDL)      # warm-up outside capture
        bi.bi_linear_w8a8(q2, s2, wq, sw, y2, ws, flags=bi.BI_FLAG_PDL)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    y2.zero_()
    with torch.cuda.graph(g, stream=stream):
        bi.bi_quantize_act(x, q2, s2, flags=bi.BI_FLAG_PDL)
        bi.bi_linear_w8a8(q2, s2, wq, sw, y2, ws, flags=bi.BI_FLAG_PDL)
    for _ in range(3):
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2, ref)


def test_workspace_left_zeroed(bi):
    M, N, K = 3, 1000, 1040   # row blocks straddle CTAs, so partial slots are used
    x_np, w = _case(9, M, N, K, True)
    wq, sw = weights(bi, w, pow2=True)
    q, s = quant_act(bi, x_np)
    ws = bi.new_workspace(M, N, K)
    for _ in range(3):
        linear(bi, q, s, wq, sw, ws=ws)
        lm = torch.empty(M, dtype=torch.int32, device=DEV)
        bi.bi_lmhead_argmax(q, s, wq, sw, None, lm, ws)
    torch.cuda.synchronize()
    # per-CTA argmax keys are scratch that is overwritten by every call; all
    # counters and partial sums must be back at zero
    from invariant_quantized_linear_gb300 import lib  # noqa: F401  (library loaded)
    G = 512   # per-CTA slots of the workspace (up to two CTAs per SM)
    head = ws[:256 + 4 * G]
    part = ws[256 + 4 * G + 8 * G * 16:]
    assert int(head.count_nonzero()) == 0 and int(part.count_nonzero()) == 0
    assert bi.bi_workspace_status(ws) == bi.BI_OK


def test_packed_weights_equal_separate_calls(bi):
    """q/k/v (or gate/up) rows stored back to back and run as one call give the
    same bits as one call per projection: output rows are independent."""
    K, M = 4096, 5
    x_np = gen.act_bf16(21, 1, M, K, outliers=gen.outlier_channels(21, K), gain=20.0)
    q, s = quant_act(bi, x_np)
    parts = [weights(bi, gen.weight_f32(21, 0, p, n, K), pow2=True) for p, n in ((0, 4096), (1, 1024), (2, 1024))]
    wq = torch.cat([w for w, _ in parts])
    sw = torch.cat([v for _, v in parts])
    packed = linear(bi, q, s, wq, sw, flags=bi.BI_FLAG_PDL)
    sep = torch.cat([linear(bi, q, s, w, v) for w, v in parts], dim=1)
    assert torch.equal(packed, sep)


def test_bounded_wait_reports_timeout_and_context_survives(bi):
    """A wait that nothing satisfies gives up after its limit and reports
    BI_ERR_TIMEOUT through the workspace; later work on the same context runs
    normally (no fault, no hang)."""
    ws = bi.new_workspace(1, 1, 16)
    bi.bi_selftest_wait_timeout(ws)
    assert bi.bi_workspace_status(ws) == bi.BI_ERR_TIMEOUT
    assert bi.bi_workspace_status(ws) == bi.BI_OK          # the status word was cleared
    x = gen.act_bf16(5, 1, 2, 256)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, gen.weight_f32(5, 0, 0, 64, 256), True)
    y = linear(bi, q, s, wq, sw, ws=ws)
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, gen.weight_f32(5, 0, 0, 64, 256), True)
    assert np.array_equal(to_np(y), oracle.linear_w8a8(q_o, s_o, wq_o, sw_o))
    assert bi.bi_workspace_status(ws) == bi.BI_OK


def test_executor_quotient_equals_ieee_division_exhaustively(bi):
    """The executor quantises with v / s formed from RN(1/s) and one fma
    correction; over every bf16 row maximum and every bf16 v with |v| <= amax
    the quotient and the code equal IEEE division's."""
    out = torch.zeros(3, dtype=torch.int64, device=DEV)
    bi.bi_selftest_quotient(out)
    torch.cuda.synchronize()
    checked, bad, example = (int(t) for t in out.cpu())
    # every pair of the domain, counted on the host by the same rule
    a = np.arange(1, 0x7F80, dtype=np.uint32)
    s = ((a << 16).view(np.float32) / np.float32(127)).astype(np.float32)
    keep = s >= np.float32(2.0 ** -64)
    assert checked == int((2 * (a[keep].astype(np.int64) + 1)).sum()), checked
    assert bad == 0, "%d mismatches, e.g. amax bits %#06x, v bits %#06x" % (bad, example >> 16, example & 0xFFFF)
