"""Pins of the split-KV attention oracle ("My speculative decoder got slower",
split-KV attention in 256-token chunks with a merge; "why speculative decoding
changed my output", "attention").  The readings (causal positions, chunking,
order of adds, the exp) are stated in oracle.c; each pin checks the oracle
against the mathematics: the true exponential within a bound, closed forms,
an fp64 reference, causality, head grouping and batch invariance."""
import math

import numpy as np
import pytest

import oracle


def _bf16_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16          # round to nearest even
    return u.astype(np.uint16)


def _f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def _rand(shape, rng, sigma=1.0):
    return _bf16_bits(rng.standard_normal(shape) * sigma)


# ---------------------------------------------------------------- exp

def test_exp_is_one_at_zero_and_flushes_below_the_normal_range():
    assert oracle.attn_exp(0.0) == 1.0
    assert oracle.attn_exp(-88.0) == 0.0 and oracle.attn_exp(-1000.0) == 0.0


def test_exp_error_bound_and_monotonicity():
    """|e(x) - exp(x)| <= 1e-5 exp(x) on [-87, 0]: the degree-6 Taylor
    remainder on |f ln 2| <= 0.35 is below 2e-8, eight fp32 roundings add
    about 5e-7, and rounding t = x log2(e) costs at most |t| 2^-24 ln 2
    < 5.3e-6 relative at |t| <= 126.  e is non-increasing on a sorted grid."""
    xs = np.concatenate([-np.logspace(-8, math.log10(87.0), 4000), np.linspace(-87.0, 0.0, 4001)])
    xs = np.sort(xs.astype(np.float32))
    es = np.array([oracle.attn_exp(float(x)) for x in xs])
    ex = np.exp(xs.astype(np.float64))
    assert np.all(np.abs(es - ex) <= 1e-5 * ex)
    assert np.all(np.diff(es) >= 0.0)


# ---------------------------------------------------------------- attention

def _exact_attention(q, k, v, T0, scale):
    """fp64 softmax attention of the bf16 inputs (no chunks), positions 0 .. T0 + m."""
    qf, kf, vf = _f32(q).astype(np.float64), _f32(k).astype(np.float64), _f32(v).astype(np.float64)
    M, Hq, D = q.shape
    g = Hq // k.shape[1]
    o = np.empty((M, Hq, D))
    for m in range(M):
        T = T0 + m + 1
        for h in range(Hq):
            s = (kf[:T, h // g] @ qf[m, h]) * scale
            p = np.exp(s - s.max())
            o[m, h] = (p @ vf[:T, h // g]) / p.sum()
    return o


def test_single_position_returns_its_value():
    rng = np.random.default_rng(1)
    q, k, v = _rand((1, 2, 64), rng), _rand((4, 1, 64), rng), _rand((4, 1, 64), rng)
    o = oracle.attention(q, k, v, 0, 0.125)
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])


def test_equal_scores_give_the_exact_mean():
    """q = 0 makes every score 0, so every weight is e(0) = 1 and o is the mean
    of the values; with small integers and 8 positions it is exact."""
    rng = np.random.default_rng(2)
    D, T = 32, 8
    vals = rng.integers(-8, 9, (T, 1, D)).astype(np.float32)
    v = _bf16_bits(vals)
    k = _rand((T, 1, D), rng)
    q = _bf16_bits(np.zeros((1, 1, D)))
    o = oracle.attention(q, k, v, T - 1, 0.125)
    assert np.array_equal(_f32(o[0, 0]), vals.mean(axis=0)[0].astype(np.float32))


@pytest.mark.parametrize("T0,M", [(0, 5), (250, 8), (700, 4), (1030, 3)])
def test_close_to_fp64_attention_across_chunks(T0, M):
    """Against fp64 softmax attention (no chunks) rounded to bf16: every output
    within one bf16 step, and almost all equal.  T0 = 250 puts the queries on
    both sides of the first chunk boundary; 700 and 1030 need 3 to 5 chunks."""
    rng = np.random.default_rng(T0 + M)
    Hq, Hkv, D = 4, 2, 64
    S = T0 + M
    q, k, v = _rand((M, Hq, D), rng), _rand((S, Hkv, D), rng), _rand((S, Hkv, D), rng)
    scale = 1.0 / math.sqrt(D)
    o = _f32(oracle.attention(q, k, v, T0, scale)).astype(np.float64)
    ref = _exact_attention(q, k, v, T0, scale)
    ref_b = _f32(_bf16_bits(ref)).astype(np.float64)
    ulp = np.maximum(np.abs(ref_b), 1e-30) * 2.0 ** -7
    assert np.all(np.abs(o - ref_b) <= ulp)
    assert np.mean(o == ref_b) > 0.97


def test_causal_positions_only():
    """Query m sees positions 0 .. T0 + m: changing later keys and values leaves
    it alone, changing position T0 + m does not."""
    rng = np.random.default_rng(3)
    M, Hq, Hkv, D, T0 = 4, 2, 1, 64, 300
    S = T0 + M
    q, k, v = _rand((M, Hq, D), rng), _rand((S, Hkv, D), rng), _rand((S, Hkv, D), rng)
    o = oracle.attention(q, k, v, T0, 0.125)
    k2, v2 = k.copy(), v.copy()
    k2[T0 + 2:], v2[T0 + 2:] = _rand(k2[T0 + 2:].shape, rng), _rand(v2[T0 + 2:].shape, rng)
    o2 = oracle.attention(q, k2, v2, T0, 0.125)
    assert np.array_equal(o2[:2], o[:2])
    assert not np.array_equal(o2[2], o[2])


def test_query_heads_share_their_group_kv_head():
    """With Hq = 4 and Hkv = 2, q heads 0-1 read kv head 0 and 2-3 kv head 1:
    changing kv head 1 changes exactly q heads 2 and 3."""
    rng = np.random.default_rng(4)
    M, Hq, Hkv, D, T0 = 2, 4, 2, 64, 40
    S = T0 + M
    q, k, v = _rand((M, Hq, D), rng), _rand((S, Hkv, D), rng), _rand((S, Hkv, D), rng)
    o = oracle.attention(q, k, v, T0, 0.125)
    v2 = v.copy()
    v2[:, 1] = _rand(v2[:, 1].shape, rng)
    o2 = oracle.attention(q, k, v2, T0, 0.125)
    assert np.array_equal(o2[:, :2], o[:, :2])
    assert not np.array_equal(o2[:, 2], o[:, 2]) and not np.array_equal(o2[:, 3], o[:, 3])


def test_queries_do_not_depend_on_the_batch():
    """Query m of a batch equals a one-query call whose cache holds T0 + m
    earlier positions."""
    rng = np.random.default_rng(5)
    M, Hq, Hkv, D, T0 = 6, 2, 2, 64, 254
    S = T0 + M
    q, k, v = _rand((M, Hq, D), rng), _rand((S, Hkv, D), rng), _rand((S, Hkv, D), rng)
    o = oracle.attention(q, k, v, T0, 0.125)
    for m in range(M):
        alone = oracle.attention(q[m:m + 1], k[:T0 + m + 1], v[:T0 + m + 1], T0 + m, 0.125)
        assert np.array_equal(alone[0], o[m])


# ---------------------------------------------------------------- fused steps

def _rn32(fr):
    """Round a Fraction to the nearest fp32, ties to even (exact: the answer is
    one of the three fp32 values around the double-rounded candidate)."""
    from fractions import Fraction
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_exp_matches_two_to_the_rounded_t():
    """The polynomial part: e(x) is within 3e-7 (relative) of 2^t for the fp32
    t = x log2(e) it rounds first; a wrong or dropped Taylor term (the x^6 term
    alone is 2e-6 at |f| = 1/2) fails this."""
    xs = np.concatenate([-np.logspace(-8, math.log10(87.0), 2000), np.linspace(-87.0, 0.0, 20001)])
    xs = xs.astype(np.float32)
    t = xs * np.float32(1.44269502162933349609375)
    keep = t >= -126.0
    es = np.array([oracle.attn_exp(float(x)) for x in xs[keep]])
    ref = np.exp2(t[keep].astype(np.float64))
    assert np.max(np.abs(es - ref) / ref) <= 3e-7


def test_chunk_value_sums_are_fused():
    """Two positions: q = e_0, k_0 = 0, k_1 = c e_0, so s = (0, c), p = (1, e(c))
    and l = 1 + e(c); each a_d is then the single rounding of v_0d + e(c) v_1d
    (a fused multiply-add), computed here in exact rational arithmetic.  Over
    4096 components some differ from the unfused RN(v_0 + RN(e(c) v_1))."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    D = 4096
    q = np.zeros(D, np.uint16)
    q[0] = 0x3F80                                          # 1.0
    k = np.zeros((2, 1, D), np.uint16)
    k[1, 0, 0] = 0xBE99                                    # -0.298828125
    v = _rand((2, 1, D), rng)
    mx, l, a = oracle.attention_chunk(q, k, v, 0, 0, 2, 1.0)
    p1 = np.float32(oracle.attn_exp(float(_f32(0xBE99))))
    assert mx == 0.0 and l == np.float32(1.0) + p1
    v0, v1 = _f32(v[0, 0]), _f32(v[1, 0])
    fused = np.array([_rn32(Fraction(float(x)) + Fraction(float(p1)) * Fraction(float(y))) for x, y in zip(v0, v1)],
                     np.float32)
    unfused = v0 + p1 * v1
    assert np.array_equal(a.view(np.uint32), fused.view(np.uint32))
    assert np.any(fused != unfused)


def test_merge_is_fused_at_a_bf16_tie():
    """Two chunk results with mx = (0, y), l = (1, 0): w = (1, e(y)), L = 1, and
    o = bf16(a_0 + e(y) a_1) with one rounding before the bf16 step.  a_0 =
    1 + 2^-8 is a bf16 tie and e(y) a_1 is just above 2^-24, half an fp32 step
    at a_0: the fused sum rounds up to a_0 + 2^-23 and the bf16 result to
    1 + 2^-7 (0x3F81); rounding e(y) a_1 to 2^-24 first would leave the tie
    and round to 1.0 (0x3F80)."""
    from fractions import Fraction
    target = Fraction(1, 2 ** 24)
    found = None
    for y in np.linspace(-0.9, -0.1, 81).astype(np.float32):
        w = np.float32(oracle.attn_exp(float(y)))
        a1 = np.float32(float(target / Fraction(float(w))))
        for cand in (a1, np.nextafter(a1, np.float32(np.inf)), np.nextafter(a1, np.float32(2.0))):
            prod = Fraction(float(w)) * Fraction(float(cand))
            if target < prod < target * (1 + Fraction(1, 2 ** 25)) and w * cand == np.float32(2.0 ** -24):
                found = (y, cand)
                break
        if found:
            break
    assert found is not None
    y, a1 = found
    D = 2
    a = np.array([[1.0 + 2.0 ** -8, 1.0 + 2.0 ** -8], [a1, 0.0]], np.float32)
    o = oracle.attention_merge(np.array([0.0, y], np.float32), np.array([1.0, 0.0], np.float32), a)
    assert o[0] == 0x3F81 and o[1] == 0x3F80


def test_equal_scores_across_chunks_give_the_rounded_mean():
    """q = 0 over 700 positions (three chunks): every weight is 1, every chunk
    maximum 0, so every merge weight is e(0) = 1; with small integer values all
    sums are exact and o is bf16(RN32(sum(v) / 700)), the rounded mean."""
    from fractions import Fraction
    rng = np.random.default_rng(8)
    D, T = 16, 700
    vals = rng.integers(-8, 9, (T, 1, D)).astype(np.float32)
    v = _bf16_bits(vals)
    k = _rand((T, 1, D), rng)
    q = _bf16_bits(np.zeros((1, 1, D)))
    o = oracle.attention(q, k, v, T - 1, 0.125)
    for d in range(D):
        mean = _rn32(Fraction(int(vals[:, 0, d].sum()), T))
        assert o[0, 0, d] == _bf16_bits(np.float32(mean))
