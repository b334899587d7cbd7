"""bi_linear_w8a8_noalloc: the linear layer for callers that cannot allocate
device memory (allocator callbacks, plugins handed only their tensors,
processes with a frozen device footprint).  It keeps the kernel's scratch in a
fixed array inside the library instead of taking a workspace.

Called through the C ABI (ctypes, raw pointers) twice in a row, its output must
equal bi_linear_w8a8's bit for bit.  The file sorts last so that a run which
stops at the first failure has already run every other test."""
import pytest
import torch

import gen
from tests.gpu_util import DEV, linear, quant_act, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


def _noalloc(bi, q, s, wq, sw, y, flags=0):
    M, K = q.shape
    N = wq.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return bi.lib.bi_linear_w8a8_noalloc(q.data_ptr(), s.data_ptr(), M, K, wq.data_ptr(), sw.data_ptr(), N,
                                         y.data_ptr(), flags, stream)


@pytest.mark.parametrize("M,N,K", [(8, 1000, 1040), (3, 4096, 4096), (16, 333, 12288)])
def test_noalloc_matches_workspace_entry_point(bi, M, N, K):
    x = gen.act_bf16(M + N, 1, M, K, outliers=gen.outlier_channels(M + N, K), gain=20.0)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, gen.weight_f32(M + N, 0, 0, N, K), pow2=True)
    ref = linear(bi, q, s, wq, sw)
    for flags in (0, bi.BI_FLAG_PDL):          # two calls in a row on the shared scratch
        y = torch.full((M, N), -1, dtype=torch.int16, device=DEV)
        assert _noalloc(bi, q, s, wq, sw, y, flags) == bi.BI_OK
        torch.cuda.synchronize()
        assert torch.equal(y, ref)


def test_noalloc_rejects_more_tokens_than_the_scratch_holds(bi):
    K, N, M = 1024, 64, 17
    q = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    s = torch.ones(M, dtype=torch.float32, device=DEV)
    wq = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    sw = torch.ones(N, dtype=torch.float32, device=DEV)
    y = torch.zeros((M, N), dtype=torch.int16, device=DEV)
    assert _noalloc(bi, q, s, wq, sw, y) == bi.BI_ERR_UNSUPPORTED


def test_noalloc_reports_a_timeout_through_its_scratch(bi):
    """A bounded wait that gives up on the fixed scratch (the library's wait
    self-test, pointed at the scratch) is reported once by
    bi_linear_w8a8_noalloc_status, which restores the scratch: the status then
    reads BI_OK again and the next two calls equal bi_linear_w8a8.  Nothing
    faults or hangs."""
    M, N, K = 5, 777, 2080
    x = gen.act_bf16(5, 1, M, K, outliers=gen.outlier_channels(5, K), gain=20.0)
    q, s = quant_act(bi, x)
    wq, sw = weights(bi, gen.weight_f32(5, 1, 0, N, K), pow2=True)
    ref = linear(bi, q, s, wq, sw)
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.full((M, N), -1, dtype=torch.int16, device=DEV)
    assert _noalloc(bi, q, s, wq, sw, y) == bi.BI_OK
    assert bi.lib.bi_linear_w8a8_noalloc_status(stream) == bi.BI_OK
    assert bi.lib.bi_selftest_wait_timeout(None, 0, stream) == bi.BI_OK
    assert bi.lib.bi_linear_w8a8_noalloc_status(stream) == bi.BI_ERR_TIMEOUT
    assert bi.lib.bi_linear_w8a8_noalloc_status(stream) == bi.BI_OK
    for _ in range(2):
        y.fill_(-1)
        assert _noalloc(bi, q, s, wq, sw, y) == bi.BI_OK
        assert bi.lib.bi_linear_w8a8_noalloc_status(stream) == bi.BI_OK
        assert torch.equal(y, ref)
