"""GPU parity of the block-scaled variant ("why speculative decoding changed
my output", "the mat-vec kernel") against the CPU oracle, bit for bit:
weight and activation quantisation, the linear (fp32 outputs compared as bit
patterns), and batch invariance over M = 1 .. 16."""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_util import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _weights_gpu(bi, w):
    N, K = w.shape
    wt = torch.from_numpy(np.ascontiguousarray(w)).to(DEV)
    ql = torch.empty((N, K // 2), dtype=torch.uint8, device=DEV)
    qh = torch.empty((N, K // 4), dtype=torch.uint8, device=DEV)
    sc = torch.empty((N, K // 16), dtype=torch.int8, device=DEV)
    d = torch.empty((N, K // 256), dtype=torch.float32, device=DEV)
    bi.bi_quantize_weight_q6(wt, ql, qh, sc, d)
    return ql, qh, sc, d


def _act_gpu(bi, x_bits):
    M, K = x_bits.shape
    xt = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(DEV)
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    d_a = torch.empty((M, K // 32), dtype=torch.float32, device=DEV)
    bi.bi_quantize_act_blocks(xt, q, d_a)
    return q, d_a


def _linear_gpu(bi, q, d_a, W, flags=0):
    ql, qh, sc, d = W
    y = torch.empty((q.shape[0], ql.shape[0]), dtype=torch.float32, device=DEV)
    bi.bi_linear_q6(q, d_a, ql, qh, sc, d, y, flags=flags)
    return y


def _np(t):
    return t.cpu().numpy()


def _case(seed, M, N, K):
    w = gen.weight_f32(seed, 0, 0, N, K)
    x = gen.act_bf16(seed, 1, M, K, outliers=gen.outlier_channels(seed, K), gain=20.0)
    return w, x


@pytest.mark.parametrize("N,K", [(1, 256), (17, 512), (100, 4096), (5, 12288)])
def test_weight_quantisation_matches_oracle(bi, N, K):
    w, _ = _case(N + K, 1, N, K)
    w = w.copy()
    w[0, 256 - 16:256] = 0.0                     # a zero sub-block
    if N > 2:
        w[2, :256] = 0.0                         # a zero super-block
    ql, qh, sc, d = _weights_gpu(bi, w)
    o = oracle.quantize_q6(w)
    for got, want in zip((ql, qh, sc, d), o):
        assert np.array_equal(_np(got).view(want.dtype), want)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 4096), (8, 12288)])
def test_activation_blocks_match_oracle(bi, M, K):
    _, x = _case(M * 3 + K, M, 1, K)
    x = x.copy()
    x[0, 32:64] = 0                              # an all-zero block (bit pattern +0)
    q, d_a = _act_gpu(bi, x)
    q_o, d_o = oracle.quantize_act_blocks(x)
    assert np.array_equal(_np(q), q_o)
    assert np.array_equal(_np(d_a), d_o)


# every token tile of the kernel (M = 1, 2-4, 5-8, 9-16), with 72 blocks per row
# (lanes with three and with two blocks), 8 blocks (most lanes empty) and 256
# or 384 blocks
SHAPES = [(1, 1, 256), (2, 17, 512), (5, 100, 4096), (8, 1000, 4096), (16, 333, 1024), (3, 64, 12288),
          (9, 31, 2304), (8, 40, 256), (6, 77, 12288), (12, 129, 8192), (16, 20, 12288)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_matches_oracle(bi, M, N, K):
    w, x = _case(M * 5 + N, M, N, K)
    W = _weights_gpu(bi, w)
    q, d_a = _act_gpu(bi, x)
    y = _linear_gpu(bi, q, d_a, W)
    want = oracle.linear_q6(_np(q), _np(d_a), *(_np(t) for t in W))
    got = _np(y)
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, "%d mismatches, first at %s" % (len(bad), bad[:4].tolist())


def test_rows_are_batch_invariant(bi):
    """Row r of an M-row call equals the one-row call on row r alone, M = 1 .. 16."""
    K, N = 4096, 513
    w, x = _case(91, 16, N, K)
    W = _weights_gpu(bi, w)
    q, d_a = _act_gpu(bi, x)
    single = torch.cat([_linear_gpu(bi, q[r:r + 1].contiguous(), d_a[r:r + 1].contiguous(), W) for r in range(16)])
    for M in range(1, 17):
        y = _linear_gpu(bi, q[:M].contiguous(), d_a[:M].contiguous(), W)
        assert torch.equal(y.view(torch.int32), single[:M].view(torch.int32)), M


@pytest.mark.parametrize("M", [1, 8, 16])
def test_full_size_gate_up_sampled_rows(bi, M):
    """gate/up of a Qwen3-8B layer (N = 24576, K = 4096) at M = 1, 8 and 16 (the
    sizes the benchmark times), with PDL: 48 sampled output rows equal the
    oracle's."""
    N, K = 24576, 4096
    w, x = _case(7, M, N, K)
    W = _weights_gpu(bi, w)
    q, d_a = _act_gpu(bi, x)
    y = _np(_linear_gpu(bi, q, d_a, W, flags=bi.BI_FLAG_PDL))
    rows = np.sort(np.random.default_rng(5).choice(N, 48, replace=False))
    Wn = [_np(t)[rows] for t in W]
    want = oracle.linear_q6(_np(q), _np(d_a), *Wn)
    assert np.array_equal(y[:, rows].view(np.uint32), want.view(np.uint32))
