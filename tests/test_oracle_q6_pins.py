"""Pins of the block-scaled oracle ("why speculative decoding changed my
output", "the mat-vec kernel": q6_k-style weight blocks of 256, int8
activation blocks of 32, integer products per block, fp32 scale-and-add in a
fixed order).  The format, quantisers and order are this library's readings,
stated in oracle.c; each pin below checks the oracle against what that
definition or the arithmetic fixes, not against a retyped copy of the code."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _bf16(x):
    """fp32 -> bf16 bit patterns (values chosen exactly representable)."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "test values must be exact bf16"
    return (u >> 16).astype(np.uint16)


def _f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- weights

def test_q6_codes_round_within_half_a_step():
    """|w - c * e_j| <= e_j / 2 for every unclamped weight, with e_j the fp32
    product d * sc_j of its super-block scale and sub-block scale; codes lie in
    [-32, 31], sub-scales in [0, 127], and each super-block's largest sub-block
    scale is 127."""
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((6, 768)) * 0.02).astype(np.float32)
    w[2, 256:512] *= 50.0                       # super-blocks of very different magnitude
    w[3, 16:32] = 0.0                           # one all-zero sub-block
    ql, qh, sc, d = oracle.quantize_q6(w)
    c = oracle.q6_codes(ql, qh).astype(np.int64)
    assert c.min() >= -32 and c.max() <= 31
    assert sc.min() >= 0 and sc.max() <= 127
    N, K = w.shape
    for n in range(N):
        for s in range(K // 256):
            assert sc[n, 16 * s:16 * s + 16].max() == 127
            for j in range(16):
                e = np.float32(d[n, s]) * np.float32(sc[n, 16 * s + j])
                seg = slice(256 * s + 16 * j, 256 * s + 16 * j + 16)
                if e == 0:
                    assert np.all(c[n, seg] == 0)
                    continue
                ratio = w[n, seg].astype(np.float64) / float(e)
                ok = np.abs(ratio) <= 31.5
                err = np.abs(w[n, seg].astype(np.float64) - c[n, seg] * float(e))
                assert np.all(err[ok] <= float(e) / 2 * (1 + 1e-6)), (n, s, j)
    assert np.all(sc[3, 1] == 0) and np.all(c[3, 16:32] == 0)


def test_q6_zero_super_block():
    w = np.zeros((2, 256), np.float32)
    ql, qh, sc, d = oracle.quantize_q6(w)
    assert np.all(d == 1.0) and np.all(sc == 0)
    assert np.all(oracle.q6_codes(ql, qh) == 0)


def test_q6_known_codes_and_byte_layout():
    """Every sub-block of one super-block has the same maximum, so every
    sub-scale is 127 and e_j = d * 127 ~ absmax / 31: weights k * absmax / 31
    quantise to code k.  The stored bytes are then fixed by the layout: low 4
    bits of c + 32 in byte k / 2 (bits 4 (k & 1)), high 2 bits in byte k / 4
    (bits 2 (k & 3))."""
    amax = 0.75
    codes = np.array([((k * 7) % 63) - 31 for k in range(256)], np.int64)
    for j in range(16):                          # every sub-block reaches +-31
        codes[16 * j] = 31 if j % 2 else -31
    w = (codes * (amax / 31)).astype(np.float32)[None, :]
    ql, qh, sc, d = oracle.quantize_q6(w)
    assert np.all(sc == 127)
    assert np.array_equal(oracle.q6_codes(ql, qh)[0].astype(np.int64), codes)
    u = codes + 32
    want_ql = (u[0::2] & 0xF) | ((u[1::2] & 0xF) << 4)
    want_qh = sum(((u[i::4] >> 4) & 3) << (2 * i) for i in range(4))
    assert np.array_equal(ql[0], want_ql.astype(np.uint8))
    assert np.array_equal(qh[0], want_qh.astype(np.uint8))


# ---------------------------------------------------------------- activations

def test_act_blocks_follow_the_per_token_rule_per_block():
    """Each block of 32: its largest magnitude maps to +-127, an all-zero block
    has scale 1 and codes 0, and a block's codes do not depend on any other
    block."""
    rng = np.random.default_rng(2)
    x = _f32((rng.standard_normal((3, 128)) * 4).astype(np.float32).view(np.uint32) >> 16)
    x[1, 32:64] = 0.0
    xb = _bf16(x)
    q, d = oracle.quantize_act_blocks(xb)
    for m in range(3):
        for b in range(4):
            blk = x[m, 32 * b:32 * b + 32]
            if np.all(blk == 0):
                assert d[m, b] == 1.0 and np.all(q[m, 32 * b:32 * b + 32] == 0)
                continue
            i = int(np.argmax(np.abs(blk)))
            assert abs(int(q[m, 32 * b + i])) == 127
    x2 = x.copy()
    x2[:, 64:] *= 4.0                             # other blocks change
    q2, d2 = oracle.quantize_act_blocks(_bf16(x2))
    assert np.array_equal(q2[:, :64], q[:, :64]) and np.array_equal(d2[:, :2], d[:, :2])


def test_act_block_half_integer_quotients_round_to_even():
    """absmax = 127 * 2^-3 makes the scale exactly 2^-3, so x = (k + 1/2) * 2^-3
    divides exactly and must round to the even neighbour."""
    scale = 2.0 ** -3
    ks = np.arange(-20, 11)
    x = np.zeros(32, np.float32)
    x[0] = 127 * scale
    x[1:] = (ks + 0.5) * scale
    q, d = oracle.quantize_act_blocks(_bf16(x)[None, :])
    assert d[0, 0] == np.float32(scale)
    want = [int(np.round(k + 0.5)) for k in ks]   # numpy rounds half to even
    assert q[0, 1:].tolist() == want


# ---------------------------------------------------------------- the linear

def _pack(codes):
    """ql, qh of int codes [N, K] (the stored layout; checked above)."""
    u = np.asarray(codes, np.int64) + 32
    ql = ((u[:, 0::2] & 0xF) | ((u[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    qh = sum(((u[:, i::4] >> 4) & 3) << (2 * i) for i in range(4)).astype(np.uint8)
    return ql, qh


def test_linear_equals_the_exact_sum_when_every_step_is_exact():
    """With power-of-two scales and small codes every fp32 operation is exact,
    so y must equal the exact rational sum over k of (c * sc * d) * (q * d_a):
    which scale multiplies which element, and every sign, is pinned."""
    rng = np.random.default_rng(3)
    N, K, M = 3, 512, 2
    codes = rng.integers(-32, 32, (N, K))
    sc = rng.integers(0, 4, (N, K // 16)).astype(np.int8)
    d = (2.0 ** rng.integers(-6, -2, (N, K // 256))).astype(np.float32)
    qa = rng.integers(-127, 128, (M, K)).astype(np.int8)
    d_a = (2.0 ** rng.integers(-8, -4, (M, K // 32))).astype(np.float32)
    ql, qh = _pack(codes)
    y = oracle.linear_q6(qa, d_a, ql, qh, sc, d)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(int(codes[n, k]) * int(sc[n, k // 16])) * Fraction(float(d[n, k // 256]))
                        * Fraction(int(qa[m, k])) * Fraction(float(d_a[m, k // 32])) for k in range(K))
            assert Fraction(float(y[m, n])) == exact, (m, n)


def _one_hot_linear(contribs, K):
    """A 1 x 1 linear whose 32-block b contributes exactly contribs[b]
    (a power of two times +-1): one nonzero product per block, sc = 1, d = 1,
    d_a = |contribs[b]|."""
    nb = K // 32
    codes = np.zeros((1, K), np.int64)
    qa = np.zeros((1, K), np.int8)
    d_a = np.ones((1, nb), np.float32)
    for b, v in contribs.items():
        codes[0, 32 * b] = 1 if v > 0 else -1
        qa[0, 32 * b] = 1
        d_a[0, b] = abs(v)
    sc = np.ones((1, K // 16), np.int8)
    d = np.ones((1, K // 256), np.float32)
    ql, qh = _pack(codes)
    return float(oracle.linear_q6(qa, d_a, ql, qh, sc, d)[0, 0])


def test_lane_order_pin():
    """K = 4096 (128 blocks): lane 0 adds blocks 0 then 32, lane 1 holds block 1.
    2^24 + 1 rounds to 2^24 (ties to even) inside lane 0, and the lane tree then
    cancels it against -2^24: the defined order gives 0, a left-to-right sum
    over the blocks would give 1."""
    assert _one_hot_linear({0: 2.0 ** 24, 1: -2.0 ** 24, 32: 1.0}, 4096) == 0.0


def test_tree_order_pin():
    """K = 256 (8 blocks, one per lane 0..7): the xor tree adds
    ((v0 + v4) + (v2 + v6)) + ((v1 + v5) + (v3 + v7)).  With v0 = 2^24, v4 = 1,
    v1 = -2^24, v5 = 1 that is 2^24 + (1 - 2^24) = 1; a left-to-right sum gives 2."""
    assert _one_hot_linear({0: 2.0 ** 24, 4: 1.0, 1: -2.0 ** 24, 5: 1.0}, 256) == 1.0


def test_rows_do_not_depend_on_the_batch():
    rng = np.random.default_rng(4)
    K, N = 768, 5
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    ql, qh, sc, d = oracle.quantize_q6(w)
    x = rng.standard_normal((6, K)).astype(np.float32)
    qa, d_a = oracle.quantize_act_blocks((x.view(np.uint32) >> 16).astype(np.uint16))
    y = oracle.linear_q6(qa, d_a, ql, qh, sc, d)
    for r in range(6):
        assert np.array_equal(oracle.linear_q6(qa[r:r + 1], d_a[r:r + 1], ql, qh, sc, d)[0], y[r])


def test_block_scale_multiply_order_pin():
    """A block's contribution is ((float)isum * d_a) * d, in that order.  With
    isum = 3, d_a = fl(1/3) and d = fl(0.1) the two orders give different fp32
    results; the oracle must give the first."""
    K = 256
    codes = np.zeros((1, K), np.int64)
    codes[0, 0] = 3
    qa = np.zeros((1, K), np.int8)
    qa[0, 0] = 1
    third = np.float32(1) / np.float32(3)
    d_a = np.ones((1, K // 32), np.float32)
    d_a[0, 0] = third
    sc = np.ones((1, K // 16), np.int8)
    d = np.full((1, 1), 0.1, np.float32)
    ql, qh = _pack(codes)
    y = oracle.linear_q6(qa, d_a, ql, qh, sc, d)[0, 0]
    stated = (np.float32(3) * third) * np.float32(0.1)
    other = (np.float32(3) * np.float32(0.1)) * third
    assert stated != other
    assert y == stated
