"""GPU parity of the quantisation entry points against the CPU oracle (bitwise)."""
import struct

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV, quant_act, to_dev, to_np, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _bf16(v):
    return struct.unpack("<I", struct.pack("<f", float(v)))[0] >> 16


@pytest.mark.parametrize("M,K,ldx", [(1, 16, 16), (3, 48, 64), (8, 4096, 4096), (16, 12288, 12288),
                                     (5, 1024, 1040), (130, 4096, 4096), (2, 133136, 133136)])
def test_quantize_act_matches_oracle(bi, M, K, ldx):
    x = gen.act_bf16(31 + M, 1, M, K, outliers=gen.outlier_channels(31, K), gain=20.0, ld=ldx)
    x[:, K:] = 0x7F80  # garbage (+inf) beyond K must be ignored
    if M >= 3:
        x[1, :K] = 0                                   # zero row -> s = 1, q = 0
        x[2, :K] = 0
        x[2, 0], x[2, 1], x[2, 2] = _bf16(127.0), _bf16(2.5), _bf16(-1.5)   # half-integer quotients
    if M >= 5:
        x[4, :K] = 0
        x[4, :3] = [_bf16(2.0 ** -130), _bf16(-(2.0 ** -131)), _bf16(2.0 ** -133)]  # subnormal absmax
    q_o, s_o = oracle.quantize_act(x, K)
    q_g, s_g = quant_act(bi, x, K)
    assert np.array_equal(to_np(q_g), q_o)
    assert np.array_equal(to_np(s_g).view(np.uint32), s_o.view(np.uint32))


@pytest.mark.parametrize("N,K", [(1, 16), (100, 272), (1024, 4096), (7, 12288)])
def test_quantize_weight_matches_oracle(bi, N, K):
    w = gen.weight_f32(40 + N, 0, 0, N, K)
    w[0, :] = 0.0
    q_o, s_o = oracle.quantize_weight(w)
    q_g, s_g = weights(bi, w, pow2=False)
    assert np.array_equal(to_np(q_g), q_o)
    assert np.array_equal(to_np(s_g).view(np.uint32), s_o.view(np.uint32))


@pytest.mark.parametrize("N,K,inplace", [(257, 1024, False), (257, 1024, True), (64, 48, True)])
def test_requant_pow2_matches_oracle(bi, N, K, inplace):
    w = gen.weight_f32(50 + N, 0, 1, N, K)
    wq_o, sw_o = oracle.quantize_weight(w)
    # a spread of scales, including subnormal, tiny, huge and degenerate ones
    sw_o[0:8] = np.array([1.0, 0.0, np.inf, 2.0 ** -140, 3.0e-39, 1.0e38, 3.0e38, 0.7071067],
                         dtype=np.float32)
    want_q, want_s = oracle.requant_pow2(wq_o, sw_o)
    wq = to_dev(wq_o)
    sw = to_dev(sw_o)
    if inplace:
        bi.bi_requant_pow2(wq, sw, wq, sw)
        got_q, got_s = wq, sw
    else:
        got_q = torch.empty_like(wq)
        got_s = torch.empty_like(sw)
        bi.bi_requant_pow2(wq, sw, got_q, got_s)
    assert np.array_equal(to_np(got_q), want_q)
    assert np.array_equal(to_np(got_s).view(np.uint32), want_s.view(np.uint32))


def test_weight_pipeline_matches_oracle_pow2(bi):
    w = gen.weight_f32(0, 0, 0, 1024, 1024)
    from tests.gpu_util import oracle_weights
    q_o, s_o = oracle_weights(oracle, w, pow2=True)
    q_g, s_g = weights(bi, w, pow2=True)
    assert np.array_equal(to_np(q_g), q_o)
    assert np.array_equal(to_np(s_g).view(np.uint32), s_o.view(np.uint32))


def test_quantize_act_pdl_flag_same_bits(bi):
    x = gen.act_bf16(3, 1, 8, 4096)
    q0, s0 = quant_act(bi, x, flags=0)
    q1, s1 = quant_act(bi, x, flags=bi.BI_FLAG_PDL)
    torch.cuda.synchronize()
    assert torch.equal(q0, q1) and torch.equal(s0, s1)
