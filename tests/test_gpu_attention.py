"""GPU parity of the split-KV verify attention ("My speculative decoder got
slower", split-KV attention in 256-token chunks with a merge; "why speculative
decoding changed my output", "attention") against the CPU oracle, bit for bit
on every output element; batch invariance over M and over the cache length
beyond a query's positions."""
import math

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


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def _attn_gpu(bi, q, k, v, T0, scale):
    M, Hq, D = q.shape
    o = torch.empty((M, Hq, D), dtype=torch.int16, device=DEV)
    n = bi.bi_attention_workspace_size(M, Hq, D, T0)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV) if n else None
    if ws is not None:
        ws.fill_(0xFF)                          # the workspace needs no initialisation
    bi.bi_attention_verify(_t(q), _t(k), _t(v), T0, scale, o, ws)
    return o.cpu().numpy().view(np.uint16)


def _assert_same(got, want):
    bad = np.argwhere(got != want)
    assert bad.size == 0, "%d of %d outputs differ, first at %s" % (len(bad), got.size, bad[:4].tolist())


# (M, Hq, Hkv, D, T0, extra cache positions past the last query)
SHAPES = [
    (1, 1, 1, 64, 0, 0),          # one position
    (5, 4, 2, 64, 0, 3),          # a few positions, cache longer than needed
    (8, 32, 8, 128, 250, 0),      # queries on both sides of the first chunk boundary
    (4, 8, 2, 128, 700, 17),      # three chunks, ragged last chunk
    (3, 4, 4, 64, 1030, 0),       # five chunks, no grouping
    (16, 8, 1, 128, 4095, 1),     # sixteen queries over one kv head, 17 chunks
    (2, 6, 3, 128, 255, 0),       # the second query starts chunk 2 with one position
    (7, 16, 8, 64, 511, 5),       # 512 positions exactly for the first query
    # at most 8 rows per kv head: heads of 128 on a grid of at most two CTAs
    # per SM run the four-CTA cluster kernel, the rest the small-row kernel
    (1, 4, 1, 64, 300, 2),        # 4 rows of 64: half the value warps have no row
    (2, 8, 2, 64, 700, 0),        # 8 rows of 64 over three chunks
    (2, 3, 1, 128, 260, 1),       # odd group: a row pair holds rows of two queries
    (1, 8, 8, 128, 4095, 0),      # one row per kv head, the last chunk a single position
    (2, 16, 4, 128, 1023, 3),     # 8 rows of 128, the second query starts a new chunk
]


@pytest.mark.parametrize("M,Hq,Hkv,D,T0,extra", SHAPES)
def test_attention_matches_oracle(bi, M, Hq, Hkv, D, T0, extra):
    S = T0 + M + extra
    q, k, v = gen.attn_qkv(M * 7 + T0, M, Hq, Hkv, D, S)
    scale = 1.0 / math.sqrt(D)
    _assert_same(_attn_gpu(bi, q, k, v, T0, scale), oracle.attention(q, k, v, T0, scale))


@pytest.mark.parametrize("sigma_k", [3.0, 12.0])
def test_peaked_scores_match_oracle(bi, sigma_k):
    """Keys scaled up make the scores spread over tens to hundreds: most
    weights flush to 0 (e of an argument below -87) and the chunks' merge
    weights w_c span many orders of magnitude or vanish."""
    M, Hq, Hkv, D, T0 = 6, 8, 2, 128, 1500
    q, k, v = gen.attn_qkv(11, M, Hq, Hkv, D, T0 + M, sigma_k=sigma_k)
    scale = 1.0 / math.sqrt(D)
    _assert_same(_attn_gpu(bi, q, k, v, T0, scale), oracle.attention(q, k, v, T0, scale))


def test_queries_are_batch_invariant(bi):
    """Query m of an M-query call equals the one-query call whose cache holds
    its T0 + m earlier positions, for M = 1 .. 16, and does not depend on the
    positions the cache holds after it."""
    Mx, Hq, Hkv, D, T0 = 16, 8, 2, 128, 760
    S = T0 + Mx + 40
    q, k, v = gen.attn_qkv(13, Mx, Hq, Hkv, D, S)
    scale = 1.0 / math.sqrt(D)
    alone = np.stack([_attn_gpu(bi, q[m:m + 1], k, v, T0 + m, scale)[0] for m in range(Mx)])
    for M in (1, 2, 3, 5, 8, 13, 16):
        _assert_same(_attn_gpu(bi, q[:M], k, v, T0, scale), alone[:M])
    k2, v2 = k.copy(), v.copy()
    k2[T0 + Mx:] = k2[:S - T0 - Mx]
    v2[T0 + Mx:] = 0
    _assert_same(_attn_gpu(bi, q, k2, v2, T0, scale), alone)


def test_later_queries_start_later(bi):
    """Shifting the batch: queries m .. M-1 of a call at T0 equal the queries
    of a call at T0 + m over the same cache."""
    M, Hq, Hkv, D, T0 = 8, 4, 4, 64, 300
    q, k, v = gen.attn_qkv(17, M, Hq, Hkv, D, T0 + M)
    scale = 0.125
    o = _attn_gpu(bi, q, k, v, T0, scale)
    for m in (1, 4, 7):
        _assert_same(_attn_gpu(bi, q[m:], k, v, T0 + m, scale), o[m:])


@pytest.mark.parametrize("M", [16, 8, 4, 3, 2, 1])
def test_full_size_verify_attention(bi, M):
    """A Qwen3-8B-shaped layer's verify attention (32 query heads over 8 kv heads
    of 128), M queries after 4096 cached positions: every output equals the
    oracle's.  M = 1, 2 run the small-row chunk kernel (4 and 8 rows per kv
    head; 17 chunks x 8 kv heads is too large a grid for the cluster kernel),
    M = 3 .. 8 the 32-row one, M = 16 two 32-row blocks per kv head."""
    Hq, Hkv, D, T0 = 32, 8, 128, 4096
    q, k, v = gen.attn_qkv(5, M, Hq, Hkv, D, T0 + M)
    scale = 1.0 / math.sqrt(D)
    _assert_same(_attn_gpu(bi, q, k, v, T0, scale), oracle.attention(q, k, v, T0, scale))


@pytest.mark.parametrize("M", [8, 4, 1])
def test_long_context_sampled_heads(bi, M):
    """32768 cached positions (129 chunks): heads sampled across the kv groups,
    each compared with the oracle on that head alone (the heads of a group
    share a kv head, so a single-head oracle call on kv head h // 4 is exact)."""
    Hq, Hkv, D, T0 = 32, 8, 128, 32768
    q, k, v = gen.attn_qkv(19, M, Hq, Hkv, D, T0 + M)
    scale = 1.0 / math.sqrt(D)
    o = _attn_gpu(bi, q, k, v, T0, scale)
    for h in (0, 5, 14, 31):
        g = h // (Hq // Hkv)
        want = oracle.attention(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], T0, scale)
        _assert_same(o[:, h:h + 1], want)


def test_maximum_positions(bi):
    """The largest cache the entry point takes: T0 + M = 2^20 positions (4096
    chunks, the widest merge), two queries, 8 q heads over one kv head; two
    sampled heads equal the oracle's."""
    M, Hq, Hkv, D = 2, 8, 1, 128
    T0 = (1 << 20) - M
    q, k, v = gen.attn_qkv(29, M, Hq, Hkv, D, T0 + M)
    scale = 1.0 / math.sqrt(D)
    o = _attn_gpu(bi, q, k, v, T0, scale)
    for h in (0, 5):
        want = oracle.attention(q[:, h:h + 1], k, v, T0, scale)
        _assert_same(o[:, h:h + 1], want)
