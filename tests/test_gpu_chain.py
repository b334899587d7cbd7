"""The chained verify pass on the GPU against the oracle (bitwise): the fused
residual and MLP quantisation kernels on their own, then whole passes run as
one program and as one call per op."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.chain_util import ChainStack
from tests.gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _bf16(v):
    import struct
    return struct.unpack("<I", struct.pack("<f", float(v)))[0] >> 16


def _edge_rows(h, y):
    """Plant the residual step's edge cases in rows 1..4 (when present)."""
    M, K = h.shape
    if M > 1:
        h[1], y[1, :K] = 0, 0                             # zero row: e = 0
    if M > 2:
        h[2], y[2, :K] = 0x8000, 0x8000                   # -0 + -0
    if M > 3:
        h[3], y[3, :K] = 0, 0
        h[3, :4] = [_bf16(2.0 ** -130), _bf16(-(2.0 ** -131)), _bf16(3 * 2.0 ** -133), _bf16(2.0 ** -128)]
    if M > 4:
        y[4, :K] = 0
        h[4, ::3] = _bf16(2.0 ** 100)                     # scale down; small entries underflow
        h[4, 1::7] = _bf16(-(2.0 ** -120))


@pytest.mark.parametrize("M,K,ldy", [(1, 4096, 4096), (5, 4096, 6144), (16, 48, 64), (3, 16400, 16400)])
def test_residual_quantize_matches_oracle(bi, M, K, ldy):
    h = gen.act_bf16(71 + M, 1, M, K, outliers=gen.outlier_channels(71, K), gain=20.0)
    y = gen.act_bf16(72 + M, 1, M, ldy, sigma=3.0)
    _edge_rows(h, y)
    want_h = oracle.residual_rescale(h, y)
    want_q, want_s = oracle.quantize_act(want_h)
    hd, yd = to_dev(h), to_dev(y)
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    for flags in (0, bi.BI_FLAG_PDL):
        hd.copy_(to_dev(h))
        bi.bi_residual_quantize(hd, yd, q, s, flags=flags)
        assert np.array_equal(to_np(hd), want_h)
        assert np.array_equal(to_np(q), want_q)
        assert np.array_equal(to_np(s).view(np.uint32), want_s.view(np.uint32))


@pytest.mark.parametrize("M,K,ld", [(1, 12288, 24576), (8, 12288, 24576), (4, 32, 80), (2, 17408, 34816)])
def test_relu_mul_quantize_matches_oracle(bi, M, K, ld):
    gu = gen.act_bf16(73 + M, 1, M, ld, sigma=2.0)
    if M > 1:
        gu[1, :K] = 0x8000                                 # relu(-0) = +0; sign from u
        gu[1, K:2 * K:2] ^= 0x8000
    want_m = oracle.relu_mul(gu, K)
    want_q, want_s = oracle.quantize_act(want_m)
    gd = to_dev(gu)
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    m_out = torch.full((M, K), -1, dtype=torch.int16, device=DEV)
    bi.bi_relu_mul_quantize(gd, K, q, s, m_out)
    assert np.array_equal(to_np(m_out), want_m)
    assert np.array_equal(to_np(q), want_q)
    assert np.array_equal(to_np(s).view(np.uint32), want_s.view(np.uint32))
    q2 = torch.empty_like(q)
    bi.bi_relu_mul_quantize(gd, K, q2, s, None, flags=bi.BI_FLAG_PDL)
    assert torch.equal(q, q2)


def test_fused_quantize_rejects_overlap(bi):
    h = torch.zeros((2, 64), dtype=torch.int16, device=DEV)
    q = torch.empty((2, 64), dtype=torch.int8, device=DEV)
    s = torch.empty(2, dtype=torch.float32, device=DEV)
    with pytest.raises(bi.BiError):
        bi.bi_residual_quantize(h, h, q, s)
    gu = torch.zeros((2, 128), dtype=torch.int16, device=DEV)
    with pytest.raises(bi.BiError):
        bi.bi_relu_mul_quantize(gu, 64, q, s, gu.view(-1)[:128].view(2, 64))   # m_out inside gu


SMALL = dict(H=256, QR=256, KV=64, I=400, V=1000)   # ragged row blocks and K units


@pytest.fixture(scope="module")
def small_stack(bi):
    return ChainStack(bi, layers=3, seed=3, **SMALL)


@pytest.mark.parametrize("M", [1, 5, 8, 16])
def test_chained_program_matches_oracle(bi, small_stack, M):
    st = small_stack
    h0 = gen.activations(gen.STACK36, 16, st.H)[:M]
    am_o, h_o, recs = st.oracle_pass(h0)
    b = st.buffers(M)
    st.run_program(b, to_dev(h0), M)
    assert np.array_equal(to_np(b["argmax"]), am_o)
    assert np.array_equal(to_np(b["h"]), h_o)
    for k in ("qkv", "o", "gu", "down"):
        assert np.array_equal(to_np(b["y_" + k]), recs[-1][k]), k


@pytest.mark.parametrize("M", [1, 5, 16])
def test_chained_calls_match_oracle_layer_by_layer(bi, small_stack, M):
    st = small_stack
    h0 = gen.activations(gen.STACK36, 16, st.H)[:M]
    am_o, h_o, recs = st.oracle_pass(h0)
    b = st.buffers(M)
    got = []
    for flags in (0, bi.BI_FLAG_PDL):
        got.clear()
        am = st.run_calls(b, to_dev(h0), M, flags=flags, record=got)
        for l, (g, r) in enumerate(zip(got, recs)):
            for k in ("qkv", "o", "h_mid", "gu", "down", "h"):
                assert np.array_equal(to_np(g[k]), r[k]), (flags, l, k)
        assert np.array_equal(to_np(am), am_o)


def test_chained_rows_are_batch_invariant(bi, small_stack):
    """Row r of a 16-row pass equals the 1-row pass on row r alone (GPU only)."""
    st = small_stack
    h0 = gen.activations(gen.STACK36, 16, st.H)
    b16 = st.buffers(16)
    st.run_program(b16, to_dev(h0), 16)
    am16, h16 = to_np(b16["argmax"]), to_np(b16["h"])
    for r in (0, 7, 15):
        b1 = st.buffers(1)
        st.run_program(b1, to_dev(h0[r:r + 1]), 1)
        assert to_np(b1["argmax"])[0] == am16[r]
        assert np.array_equal(to_np(b1["h"])[0], h16[r])


def test_chained_program_reruns_identically(bi, small_stack):
    st = small_stack
    h0 = to_dev(gen.activations(gen.STACK36, 8, st.H))
    b = st.buffers(8)
    prog, ws = st.run_program(b, h0, 8)
    first = (to_np(b["h"]).copy(), to_np(b["argmax"]).copy())
    for _ in range(3):
        b["h"].copy_(h0)
        bi.bi_program_run(prog, 8, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(b["h"]), first[0]) and np.array_equal(to_np(b["argmax"]), first[1])


def test_qwen3_8b_chained_layers_full_size(bi):
    """Two chained layers at the full Qwen3-8B shapes and the full 151,936-row
    head, M = 5 (the multi-token verify case): every output equals the oracle's."""
    st = ChainStack(bi, H=4096, QR=4096, KV=1024, I=12288, V=151936, layers=2, seed=3)
    M = 5
    h0 = gen.activations(gen.STACK36, M, st.H)
    am_o, h_o, recs = st.oracle_pass(h0)
    b = st.buffers(M)
    st.run_program(b, to_dev(h0), M)
    assert np.array_equal(to_np(b["argmax"]), am_o)
    assert np.array_equal(to_np(b["h"]), h_o)
    for k in ("qkv", "o", "gu", "down"):
        assert np.array_equal(to_np(b["y_" + k]), recs[-1][k]), k


def test_stack36_chained_full_size(bi):
    """The whole benchmark pass: 36 chained Qwen3-8B-shaped layers and the
    151,936-row head as one program, at M = 8 (the benchmarked verify batch),
    at every smaller M the benchmark sweeps, and at M = 1 (decode): the final
    residual stream and every argmax equal the oracle's eight-token pass,
    row for row (rows do not depend on how many tokens share the pass)."""
    st = ChainStack(bi, H=4096, QR=4096, KV=1024, I=12288, V=151936, layers=36, seed=3)
    h0 = gen.activations(gen.STACK36, 8, st.H)
    am_o, h_o, _ = st.oracle_pass(h0, record=False)
    for M in (8, 5, 4, 3, 2, 1):
        b = st.buffers(M)
        st.run_program(b, to_dev(h0[:M]), M)
        assert np.array_equal(to_np(b["argmax"]), am_o[:M]), M
        assert np.array_equal(to_np(b["h"]), h_o[:M]), M
