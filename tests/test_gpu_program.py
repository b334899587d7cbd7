"""The verify-pass executor (bi_program_*) gives exactly the bits of the same
ops issued one call at a time, including ops that read what earlier ops of
the same program wrote."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV, linear, lmhead, oracle_weights, quant_act, to_dev, to_np, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _chain(bi, M, dims, seed, head_n=None):
    """x0 -> quant -> linear(W1) -> y1 -> quant(y1) -> linear(W2) -> ... -> head.
    Returns (ops, buffers) for the program and the per-call reference."""
    K0 = dims[0]
    x0 = to_dev(gen.act_bf16(seed, 1, M, K0, outliers=gen.outlier_channels(seed, K0), gain=20.0))
    Ws = [weights(bi, gen.weight_f32(seed, i, 0, dims[i + 1], dims[i]), pow2=(i % 2 == 0))
          for i in range(len(dims) - 1)]
    head = None
    if head_n:
        head = weights(bi, gen.weight_f32(seed, 99, 0, head_n, dims[-1]), pow2=True)
    return x0, Ws, head


def _reference(bi, M, dims, x0, Ws, head):
    x = x0
    ys = []
    for i, (wq, sw) in enumerate(Ws):
        q = torch.empty((M, dims[i]), dtype=torch.int8, device=DEV)
        s = torch.empty(M, dtype=torch.float32, device=DEV)
        bi.bi_quantize_act(x, q, s)
        y = linear(bi, q, s, wq, sw)
        ys.append(y)
        x = y
    am = lg = None
    if head is not None:
        q = torch.empty((M, dims[-1]), dtype=torch.int8, device=DEV)
        s = torch.empty(M, dtype=torch.float32, device=DEV)
        bi.bi_quantize_act(x, q, s)
        am, lg = lmhead(bi, q, s, head[0], head[1])
    torch.cuda.synchronize()
    return ys, am, lg


def _program(bi, M, dims, x0, Ws, head):
    ops, keep = [], []
    x = x0
    ys = []
    for i, (wq, sw) in enumerate(Ws):
        q = torch.empty((M, dims[i]), dtype=torch.int8, device=DEV)
        s = torch.empty(M, dtype=torch.float32, device=DEV)
        y = torch.full((M, wq.shape[0]), -1, dtype=torch.int16, device=DEV)
        ops += [bi.op_quantize_act(x, q, s), bi.op_linear(q, s, wq, sw, y)]
        keep += [q, s, y]
        ys.append(y)
        x = y
    am = lg = None
    if head is not None:
        q = torch.empty((M, dims[-1]), dtype=torch.int8, device=DEV)
        s = torch.empty(M, dtype=torch.float32, device=DEV)
        am = torch.full((M,), -1, dtype=torch.int32, device=DEV)
        lg = torch.full((M, head[0].shape[0]), -1, dtype=torch.int16, device=DEV)
        ops += [bi.op_quantize_act(x, q, s), bi.op_lmhead(q, s, head[0], head[1], lg, am)]
        keep += [q, s]
    prog = bi.new_program(len(ops))
    bi.bi_program_build(ops, prog)
    return prog, ys, am, lg, keep


@pytest.mark.parametrize("M,dims,head_n", [
    (1, [1024, 4096, 1024], None),
    (5, [4096, 1008, 1040, 272], 3000),
    (8, [4096, 6144, 4096, 12288, 4096], 20000),
    (16, [2048, 336, 2048], 5000),
    (9, [48, 64, 16], 100),
])
def test_program_matches_single_calls(bi, M, dims, head_n):
    x0, Ws, head = _chain(bi, M, dims, 3 + M, head_n)
    ref_y, ref_am, ref_lg = _reference(bi, M, dims, x0, Ws, head)
    prog, ys, am, lg, keep = _program(bi, M, dims, x0, Ws, head)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    for run in range(3):                       # repeated runs reuse the workspace
        for y in ys:
            y.fill_(-1)
        bi.bi_program_run(prog, M, ws)
        torch.cuda.synchronize()
        assert bi.bi_workspace_status(ws) == bi.BI_OK
        for i, (a, b) in enumerate(zip(ys, ref_y)):
            assert torch.equal(a, b), (run, i)
        if head is not None:
            assert torch.equal(am, ref_am) and torch.equal(lg, ref_lg), run


def test_program_against_oracle_two_layers(bi):
    """A 2-linear chain checked directly against the CPU oracle."""
    M, dims = 4, [1024, 2048, 512]
    x0_np = gen.act_bf16(8, 1, M, dims[0], outliers=gen.outlier_channels(8, dims[0]), gain=20.0)
    w = [gen.weight_f32(8, i, 0, dims[i + 1], dims[i]) for i in range(2)]
    x = x0_np
    for wi in w:
        q, s = oracle.quantize_act(x)
        wq, sw = oracle_weights(oracle, wi, True)
        x = oracle.linear_w8a8(q, s, wq, sw)
    Ws = [weights(bi, wi, True) for wi in w]
    prog, ys, _, _, keep = _program(bi, M, dims, to_dev(x0_np), Ws, None)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    bi.bi_program_run(prog, M, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(ys[-1]), x)


def test_program_wrong_token_tiles_is_reported(bi):
    """Running a program with a max_tokens that selects the other kernel
    variant launches nothing useful and reports BI_ERR_INVALID_ARG."""
    M, dims = 12, [256, 256]
    x0, Ws, _ = _chain(bi, M, dims, 1)
    prog, ys, _, _, keep = _program(bi, M, dims, x0, Ws, None)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    bi.bi_program_run(prog, 4, ws)            # built for 9..16 tokens
    torch.cuda.synchronize()
    assert bi.bi_workspace_status(ws) == bi.BI_ERR_INVALID_ARG
    bi.bi_program_run(prog, M, ws)
    torch.cuda.synchronize()
    assert bi.bi_workspace_status(ws) == bi.BI_OK


def test_program_in_cuda_graph(bi):
    M, dims = 8, [4096, 4096, 4096]
    x0, Ws, head = _chain(bi, M, dims, 2, 8000)
    ref_y, ref_am, _ = _reference(bi, M, dims, x0, Ws, head)
    prog, ys, am, lg, keep = _program(bi, M, dims, x0, Ws, head)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        bi.bi_program_run(prog, M, ws)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bi.bi_program_run(prog, M, ws)
    for _ in range(3):
        for y in ys:
            y.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ys, ref_y))
        assert torch.equal(am, ref_am)


def test_program_quantize_crafted_rows_match_oracle(bi):
    """Quantisation inside a program: half-integer quotients (ties to even),
    quotients a hair either side of a half-integer, zero and subnormal rows."""
    import struct
    K = 4096
    rng = np.random.default_rng(4)

    def bf(v):
        return struct.unpack("<I", struct.pack("<f", float(v)))[0] >> 16

    x = gen.act_bf16(12, 1, 6, K)
    x[0, 0] = bf(127.0)                            # s = 1: x / s = x exactly
    for i, v in enumerate(np.arange(-126.5, 126.5, 0.5)[:K - 1]):
        x[0, 1 + i] = bf(v)
    x[1, :] = 0                                     # zero row
    x[2, :] = 0
    x[2, :3] = [bf(2.0 ** -130), bf(-(2.0 ** -131)), bf(2.0 ** -133)]
    x[3, 0] = bf(100.0)                             # quotients near half-integers for s = 100/127
    vals = (np.arange(1, K) - 0.5) * np.float32(100.0 / 127.0) * (1 + rng.uniform(-1e-6, 1e-6, K - 1))
    x[3, 1:] = [bf(v) for v in np.clip(vals, -99.0, 99.0)]
    q_o, s_o = oracle.quantize_act(x)
    xd = to_dev(x)
    q = torch.empty((6, K), dtype=torch.int8, device=DEV)
    s = torch.empty(6, dtype=torch.float32, device=DEV)
    prog = bi.new_program(1)
    bi.bi_program_build([bi.op_quantize_act(xd, q, s)], prog)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    bi.bi_program_run(prog, 1, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(q), q_o)
    assert np.array_equal(to_np(s).view(np.uint32), s_o.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [(3, 1040, 528), (8, 4096, 1008), (1, 272, 48)])
def test_program_linear_on_external_codes(bi, M, K, N):
    """A program whose first linear reads codes quantised outside it (so they
    arrive as int8, including a K that ends inside a 256-byte unit), followed
    by a quantisation and a linear that read the program's own codes: both
    equal the single calls."""
    x = gen.act_bf16(21 + M, 1, M, K, outliers=gen.outlier_channels(21, K), gain=20.0)
    w1 = weights(bi, gen.weight_f32(21, 1, 0, N, K), pow2=True)
    w2 = weights(bi, gen.weight_f32(21, 2, 0, 2 * N, N), pow2=False)
    q0, s0 = quant_act(bi, x)
    y1_ref = linear(bi, q0, s0, *w1)
    q1_ref = torch.empty((M, N), dtype=torch.int8, device=DEV)
    s1_ref = torch.empty(M, dtype=torch.float32, device=DEV)
    bi.bi_quantize_act(y1_ref, q1_ref, s1_ref)
    y2_ref = linear(bi, q1_ref, s1_ref, *w2)
    y1 = torch.full((M, N), -1, dtype=torch.int16, device=DEV)
    y2 = torch.full((M, 2 * N), -1, dtype=torch.int16, device=DEV)
    q1 = torch.empty((M, N), dtype=torch.int8, device=DEV)
    s1 = torch.empty(M, dtype=torch.float32, device=DEV)
    ops = [bi.op_linear(q0, s0, *w1, y1), bi.op_quantize_act(y1, q1, s1), bi.op_linear(q1, s1, *w2, y2)]
    prog = bi.new_program(len(ops))
    bi.bi_program_build(ops, prog)
    ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
    for _ in range(2):
        bi.bi_program_run(prog, M, ws)
        torch.cuda.synchronize()
        assert bi.bi_workspace_status(ws) == bi.BI_OK
        assert torch.equal(y1, y1_ref)
        assert torch.equal(q1, q1_ref) and torch.equal(s1, s1_ref)
        assert torch.equal(y2, y2_ref)
