"""The bandwidth probes read and copy every byte they are given."""
import numpy as np
import pytest
import torch

from tests.gpu_util import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import invariant_quantized_linear_gb300 as m
    return m


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 37 * 1024 * 1024 + 48])
def test_probe_read_sees_every_word(bi, nbytes):
    host = np.random.default_rng(nbytes).integers(0, 2 ** 63, nbytes // 8, dtype=np.int64)
    buf = torch.from_numpy(host).to(DEV)
    out = torch.zeros(1, dtype=torch.int64, device=DEV)
    bi.bi_probe_read(buf, out)
    want = np.bitwise_xor.reduce(host.view(np.uint64))
    assert int(out.cpu().numpy().view(np.uint64)[0]) == int(want)


def test_probe_copy_copies_exactly(bi):
    src = torch.randint(-2 ** 31, 2 ** 31 - 1, (9 * 1024 * 1024 + 4,), dtype=torch.int32, device=DEV)
    dst = torch.zeros_like(src)
    bi.bi_probe_copy(src, dst)
    assert torch.equal(src, dst)
