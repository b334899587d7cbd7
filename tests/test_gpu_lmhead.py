"""GPU parity of bi_lmhead_argmax (bf16 logits and lowest-index greedy argmax)
against the CPU oracle, at the full LM-head size with planted near ties."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV, lmhead, oracle_weights, quant_act, to_dev, to_np, weights, weights_chunked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (3, 100, 48), (8, 1000, 1024), (16, 5000, 272), (9, 64, 4096)])
def test_lmhead_small_matches_oracle(bi, M, N, K):
    x = gen.act_bf16(M + N, 1, M, K)
    w = gen.weight_f32(M + N, 0, 2, N, K)
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, True)
    am_o, lg_o = oracle.lmhead_argmax(q_o, s_o, wq_o, sw_o)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, True)
    am, lg = lmhead(bi, q, s, wq, sw)
    assert np.array_equal(to_np(lg), lg_o)
    assert np.array_equal(to_np(am), am_o)
    am2, _ = lmhead(bi, q, s, wq, sw, want_logits=False)
    assert torch.equal(am, am2)


def test_lmhead_ties_pick_lowest_index(bi):
    """Duplicate weight rows give exactly tied logits; the lower index wins,
    wherever the two rows fall relative to CTA ranges."""
    M, N, K = 4, 20000, 1024
    x = gen.act_bf16(5, 1, M, K)
    w = gen.weight_f32(5, 0, 2, N, K)
    xs = gen.bf16_bits_to_f32(x)
    for m, (a, b) in enumerate([(19000, 3), (100, 15000), (7, 8), (12345, 12346)]):
        w[a] = np.sign(xs[m]) * 0.05
        w[b] = w[a]
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, True)
    am_o, _ = oracle.lmhead_argmax(q_o, s_o, wq_o, sw_o)
    assert am_o.tolist() == [3, 100, 7, 12345]
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, True)
    am, _ = lmhead(bi, q, s, wq, sw, want_logits=False)
    assert to_np(am).tolist() == am_o.tolist()


def test_lmhead_full_size_with_near_ties(bi):
    """LM head 4096 -> 151936, power-of-two scales, M = 8 rows with planted
    exact and near ties; logits and argmax bitwise against the oracle, and
    every M = 1..8 prefix gives the same rows."""
    wl = gen.LMHEAD_WL
    N, K = gen.LMHEAD.N, gen.LMHEAD.K
    x = gen.activations(wl, 8, K)
    make = lambda r0, r: gen.lmhead_weight_f32(wl.seed, x, r0, r, N=N, K=K)
    wq, sw = weights_chunked(bi, make, N, K, pow2=True)
    wq_o = np.empty((N, K), np.int8)
    sw_o = np.empty(N, np.float32)
    for r0 in range(0, N, 16384):
        r = min(16384, N - r0)
        wq_o[r0:r0 + r], sw_o[r0:r0 + r] = oracle_weights(oracle, make(r0, r), True)
    assert np.array_equal(to_np(wq), wq_o) and np.array_equal(to_np(sw).view(np.uint32), sw_o.view(np.uint32))
    q_o, s_o = oracle.quantize_act(x)
    am_o, lg_o = oracle.lmhead_argmax(q_o, s_o, wq_o, sw_o)
    rows = gen.lmhead_special_rows(N)
    assert am_o[0] == min(rows[0]) and am_o[4] == min(rows[4])   # exact ties resolved low
    q, s = quant_act(bi, x)
    for M in range(1, 9):
        am, lg = lmhead(bi, q[:M].contiguous(), s[:M].contiguous(), wq, sw, flags=bi.BI_FLAG_PDL)
        assert np.array_equal(to_np(am), am_o[:M]), M
        assert np.array_equal(to_np(lg), lg_o[:M]), M


@pytest.mark.parametrize("M", [1, 2, 5, 16, 40, 100])
def test_greedy_verify_matches_oracle(bi, M):
    rng = np.random.default_rng(200 + M)
    for trial in range(20):
        am = rng.integers(0, 5, M).astype(np.int32)
        dr = am[:M - 1].copy()
        cut = int(rng.integers(0, M))
        if cut < M - 1:
            dr[cut] = dr[cut] + 1
        out = torch.full((2,), -1, dtype=torch.int32, device=DEV)
        bi.bi_greedy_verify(to_dev(am), to_dev(dr) if M > 1 else None, out)
        assert tuple(to_np(out).tolist()) == oracle.greedy_verify(am, dr), (trial, cut)


@pytest.mark.parametrize("M,cut", [(8, 3), (8, 7), (5, 0), (1, 0), (16, 11)])
def test_program_head_greedy_verify(bi, M, cut):
    """An LM-head op with drafted tokens reports the accepted count and the
    next token, as the oracle computes them from the oracle's argmax."""
    K, N = 1024, 3000
    x = gen.act_bf16(300 + M, 1, M, K)
    w = gen.weight_f32(300 + M, 0, 0, N, K)
    q_o, s_o = oracle.quantize_act(x)
    wq_o, sw_o = oracle_weights(oracle, w, True)
    am_o, _ = oracle.lmhead_argmax(q_o, s_o, wq_o, sw_o, want_logits=False)
    dr = am_o[:M - 1].copy()
    if cut < M - 1:
        dr[cut] = (dr[cut] + 1) % N
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, w, True)
    am = torch.full((M,), -1, dtype=torch.int32, device=DEV)
    acc = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    dd = to_dev(dr) if M > 1 else None
    ops = [bi.op_lmhead(q, s, wq, sw, None, am, draft=dd, accept=acc)]
    prog = bi.new_program(1)
    bi.bi_program_build(ops, prog)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    bi.bi_program_run(prog, M, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(am), am_o)
    assert tuple(to_np(acc).tolist()) == oracle.greedy_verify(am_o, dr)
