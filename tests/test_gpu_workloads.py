"""The benchmark workloads at their full sizes, checked against the oracle
(every output where the oracle finishes in seconds, sampled rows otherwise)."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV, linear, oracle_weights, quant_act, to_np, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def test_single_linear_workload(bi):
    """M = 2, K = N = 1024, pow2 scales, four outlier channels x20, seed 0."""
    wl = gen.SINGLE
    x = gen.activations(wl, 2, 1024)
    w = gen.weight_f32(wl.seed, 0, 0, 1024, 1024)
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, True)
    want = oracle.linear_w8a8(q_o, s_o, wq_o, sw_o)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, True)
    assert np.array_equal(to_np(linear(bi, q, s, wq, sw)), want)


@pytest.mark.parametrize("lin", gen.QWEN3_8B_LINEARS, ids=lambda l: l.name)
def test_qwen3_8b_layer_linears(bi, lin):
    """Each Qwen3-8B-shaped linear with its own absmax scales, M in {1,2,3,4,5,8};
    every row of every M equals the oracle's row."""
    wl = gen.QWEN3_8B
    x = gen.activations(wl, 8, lin.K, stream=gen.STREAM_ACT + lin.proj)
    w = gen.weight_f32(wl.seed, 0, lin.proj, lin.N, lin.K)
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, False)
    want = oracle.linear_w8a8(q_o, s_o, wq_o, sw_o)
    wq, sw = weights(bi, w, False)
    for M in wl.Ms:
        q, s = quant_act(bi, x[:M])
        for flags in (0, bi.BI_FLAG_PDL):
            assert np.array_equal(to_np(linear(bi, q, s, wq, sw, flags=flags)), want[:M]), (M, flags)


@pytest.mark.parametrize("M", gen.PREFILL.Ms)
def test_prefill_workload(bi, M):
    """M in {512, 2048}, K = 4096, N = 12288: every row equals the M = 16
    weight-streaming kernel's row (itself M-invariant), and 48 sampled rows
    equal the oracle's."""
    wl = gen.PREFILL
    K, N = 4096, 12288
    x = gen.activations(wl, M, K)
    w = gen.weight_f32(wl.seed, 0, 0, N, K)
    wq, sw = weights(bi, w, True)
    q, s = quant_act(bi, x)
    y = linear(bi, q, s, wq, sw)
    ws = bi.new_workspace(16, N, K)
    for r0 in range(0, M, 16):
        ys = linear(bi, q[r0:r0 + 16].contiguous(), s[r0:r0 + 16].contiguous(), wq, sw, ws=ws)
        assert torch.equal(ys, y[r0:r0 + 16]), r0
    rows = np.random.default_rng(M).choice(M, 48, replace=False)
    q_o, s_o = oracle.quantize_act(x[rows])
    wq_o, sw_o = oracle_weights(oracle, w, True)
    want = oracle.linear_w8a8(q_o, s_o, wq_o, sw_o)
    assert np.array_equal(to_np(y)[rows], want)
