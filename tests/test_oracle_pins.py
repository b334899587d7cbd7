"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden), an exact-rational restatement (tests/exact_ref.py),
closed forms, invariants, brute force on tiny inputs, or a library routine.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import gen
import oracle
from tests import exact_ref as ex


def f32(x):
    return np.float32(x)


def bf16_pattern(x: float) -> int:
    u = struct.unpack("<I", struct.pack("<f", float(x)))[0]
    assert u & 0xFFFF == 0, x
    return u >> 16


def bf16_array(vals) -> np.ndarray:
    return np.array([bf16_pattern(v) for v in vals], dtype=np.uint16)


def ulp_dist_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


# --------------------------------------------------------------- fp32 order

def test_fp32_order_example(golden):
    """Page "why speculative decoding changed my output", "floats care about order"."""
    g = golden("fp32_order.txt")
    a, b = f32(float(g["a"])), f32(float(g["b"]))
    assert float(np.spacing(a)) == float(g["spacing_near_a"])
    assert float((a + b) - a) == float(g["(a + b) - a"])
    assert float((a - a) + b) == float(g["(a - a) + b"])


def test_integer_accumulation_is_order_independent():
    """The Integer Alibi: the int32 dot product of shared int8 operands is exact,
    so any permutation of k gives the same bits; an fp32 sum of the same
    products in two orders need not."""
    rng = np.random.default_rng(7)
    K, N, M = 4096, 16, 3
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    s_a = rng.uniform(0.01, 0.1, M).astype(np.float32)
    s_w = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    y = oracle.linear_w8a8(q, s_a, w, s_w)
    for seed in range(3):
        perm = np.random.default_rng(seed).permutation(K)
        assert np.array_equal(oracle.linear_w8a8(q[:, perm], s_a, w[:, perm], s_w), y)
    # the same sums in fp32, forwards and backwards, do differ somewhere
    prod = (q[:, None, :].astype(np.float32) * w[None, :, :].astype(np.float32)) * f32(1e-3)
    fwd = np.zeros((M, N), np.float32)
    bwd = np.zeros((M, N), np.float32)
    for k in range(K):
        fwd += prod[:, :, k]
        bwd += prod[:, :, K - 1 - k]
    assert not np.array_equal(fwd, bwd)


# --------------------------------------------------------------- bf16 rounding

def test_bf16_rne_against_torch_structured_exhaustive():
    """Every bf16 high half x the rounding-relevant low halves (below, at and
    above the midpoint, both ends), plus 2^22 random patterns, against torch's
    float32 -> bfloat16 conversion (round to nearest even).  NaN patterns are
    excluded (the oracle canonicalises them, torch keeps a payload)."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x3FFF, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFE, 0xFFFF],
                    dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    pats = np.concatenate([pats, np.random.default_rng(1).integers(0, 1 << 32, 1 << 22,
                                                                   dtype=np.uint64).astype(np.uint32)])
    f = pats.view(np.float32)
    keep = ~np.isnan(f)
    f = np.ascontiguousarray(f[keep])
    ours = oracle.f32_to_bf16_rne_array(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rne_against_exact_rational():
    rng = np.random.default_rng(3)
    pats = rng.integers(0, 0x7F800000, 3000, dtype=np.uint64).astype(np.uint32)
    pats = np.concatenate([pats, pats | np.uint32(0x80000000)])
    for u in pats:
        x = np.array([u], np.uint32).view(np.float32)[0]
        want = ex.rn_bf16(Fraction(float(x)))
        got = oracle.f32_to_bf16_rne(x)
        if want in (ex.INF, -ex.INF):
            assert got == (0x7F80 if want > 0 else 0xFF80)
        else:
            assert got == ex.bf16_bits(want)


def test_bf16_rne_special_cases():
    assert oracle.f32_to_bf16_rne(float("nan")) == 0x7FC0
    assert oracle.f32_to_bf16_rne(float("inf")) == 0x7F80
    assert oracle.f32_to_bf16_rne(-0.0) == 0x8000
    # largest finite fp32 rounds up to infinity under round-to-nearest
    assert oracle.f32_to_bf16_rne(np.finfo(np.float32).max) == 0x7F80
    # 1 + 2^-8 is exactly halfway between 1 and 1 + 2^-7: ties go to the even 1.0
    assert oracle.f32_to_bf16_rne(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.f32_to_bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82


# --------------------------------------------------------------- quantisation

def _exact_quant_rows(x_bits: np.ndarray):
    rows_q, rows_s = [], []
    for row in x_bits:
        codes, s = ex.quantize_row([ex.bf16_value(b) for b in row])
        rows_q.append(codes)
        rows_s.append(s)
    return rows_q, rows_s


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_quantize_act_against_exact_rational(seed):
    x = gen.act_bf16(seed, 1, 4, 64, outliers=gen.outlier_channels(seed, 64), gain=20.0)
    q, s = oracle.quantize_act(x)
    eq, es = _exact_quant_rows(x)
    assert np.array_equal(q, np.array(eq, np.int8))
    assert [Fraction(float(v)) for v in s] == es


def test_quantize_act_half_integer_quotients_round_to_even():
    """absmax = 127 gives s_a = 1 exactly, so x / s_a = x and x.5 values must go
    to the even neighbour; -0.5 goes to 0."""
    vals = [127.0, 2.5, 3.5, -0.5, -1.5, 0.5, 126.5, -125.5, 1.0, 0.0]
    x = bf16_array(vals)[None, :]
    q, s = oracle.quantize_act(np.pad(x, ((0, 0), (0, 6))))
    assert s[0] == np.float32(1.0)
    assert q[0, :10].tolist() == [127, 2, 4, 0, -2, 0, 126, -126, 1, 0]


def test_quantize_act_zero_row_and_absmax_maps_to_127():
    x = np.zeros((2, 32), np.uint16)
    x[1] = gen.act_bf16(5, 1, 1, 32)[0]
    q, s = oracle.quantize_act(x)
    assert s[0] == 1.0 and not q[0].any()
    i = int(np.argmax(np.abs(gen.bf16_bits_to_f32(x[1]))))
    assert abs(int(q[1, i])) == 127
    assert q.min() >= -127


def test_quantize_act_subnormal_row():
    """absmax in the subnormal range: s_a is a subnormal fp32 (no flush to zero)."""
    vals = [2.0 ** -130, -2.0 ** -131, 2.0 ** -133, 0.0] + [0.0] * 12
    x = bf16_array(vals)[None, :]
    q, s = oracle.quantize_act(x)
    eq, es = _exact_quant_rows(x)
    assert Fraction(float(s[0])) == es[0] and float(s[0]) < 2.0 ** -126
    assert q[0].tolist() == eq[0]


def test_quantize_weight_round_trip_bound():
    """|w - q*s| <= s/2 (+ the fp32 rounding of w/s) for every element."""
    w = gen.weight_f32(11, 0, 0, 64, 256)
    wq, s = oracle.quantize_weight(w)
    err = np.abs(w.astype(np.float64) - wq.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-6))
    eq = [ex.quantize_row([Fraction(float(v)) for v in row]) for row in w[:8]]
    for n in range(8):
        assert wq[n].tolist() == eq[n][0]
        assert Fraction(float(s[n])) == eq[n][1]


# --------------------------------------------------------------- pow2 requant

def _own_scale_weights(seed=21, N=256, K=128):
    w = gen.weight_f32(seed, 0, 0, N, K)
    return oracle.quantize_weight(w)


def test_requant_pow2_scale_is_nearest_power_of_two_brute_force():
    wq, s = _own_scale_weights()
    _, sp = oracle.requant_pow2(wq, s)
    for a, b in zip(s, sp):
        assert float(b) == ex.nearest_pow2_log(float(a))
        assert abs(math.log2(float(b) / float(a))) <= 0.5


def test_requant_pow2_codes_exact_rational():
    wq, s = _own_scale_weights(N=32, K=64)
    wq2, sp = oracle.requant_pow2(wq, s)
    for n in range(32):
        ratio = Fraction(float(s[n])) / Fraction(float(sp[n]))
        want = [max(-127, min(127, round(int(c) * ratio))) for c in wq[n]]
        assert wq2[n].tolist() == want


def test_requant_pow2_invariants():
    wq, s = _own_scale_weights()
    wq2, sp = oracle.requant_pow2(wq, s)
    # idempotent, and the identity on power-of-two scales
    wq3, sp3 = oracle.requant_pow2(wq2, sp)
    assert np.array_equal(wq3, wq2) and np.array_equal(sp3, sp)
    m, _ = np.frexp(sp)
    assert np.all(m == 0.5)
    # dequantised values move by at most half a new step where not clamped
    old = wq.astype(np.float64) * s[:, None]
    new = wq2.astype(np.float64) * sp[:, None]
    unclamped = np.abs(wq2) < 127
    assert np.all(np.abs(new - old)[unclamped] <= (sp[:, None] / 2 + 0 * old)[unclamped])
    # rewriting the scales without requantising the codes is a different layer
    assert not np.allclose(wq.astype(np.float64) * sp[:, None], old, rtol=1e-3)


def test_requant_pow2_degenerate_scales():
    wq = np.array([[1, -2, 3, 4]] * 3, np.int8)
    s = np.array([1.0, 0.0, np.inf], np.float32)
    out, so = oracle.requant_pow2(wq, s)
    assert np.array_equal(out, wq) and so[0] == 1.0 and so[1] == 0.0 and np.isinf(so[2])


# --------------------------------------------------------------- linear

def _tiny_case(seed, M, N, K, pow2):
    x = gen.act_bf16(seed, 1, M, K, outliers=gen.outlier_channels(seed, K, 2), gain=20.0)
    w = gen.weight_f32(seed, 0, 0, N, K)
    wq, s_w = oracle.quantize_weight(w)
    if pow2:
        wq, s_w = oracle.requant_pow2(wq, s_w)
    q, s_a = oracle.quantize_act(x)
    return x, q, s_a, wq, s_w


@pytest.mark.parametrize("seed,M,N,K,pow2", [(0, 4, 8, 64, True), (1, 3, 8, 48, False),
                                              (2, 1, 5, 16, False), (3, 4, 8, 64, False)])
def test_linear_against_exact_rational(seed, M, N, K, pow2):
    x, q, s_a, wq, s_w = _tiny_case(seed, M, N, K, pow2)
    y = oracle.linear_w8a8(q, s_a, wq, s_w)
    want = ex.linear(q.tolist(), [Fraction(float(v)) for v in s_a], wq.tolist(),
                     [Fraction(float(v)) for v in s_w])
    assert y.tolist() == want


def test_linear_large_accumulators_against_exact_rational():
    """|acc| above 2^24, where int32 -> fp32 itself rounds."""
    rng = np.random.default_rng(5)
    K = 2048
    q = np.full((2, K), 127, np.int8)
    q[1, ::3] = -127
    w = rng.integers(100, 128, (4, K)).astype(np.int8)
    w[2] = -w[2]
    s_a = np.array([0.0301, 1.0], np.float32)
    s_w = np.array([3.1e-4, 2.0 ** -11, 7.7e-5, 1.0], np.float32)
    y = oracle.linear_w8a8(q, s_a, w, s_w)
    accs = q.astype(np.int64) @ w.astype(np.int64).T
    assert np.abs(accs).max() > 2 ** 24
    want = ex.linear(q.tolist(), [Fraction(float(v)) for v in s_a], w.tolist(),
                     [Fraction(float(v)) for v in s_w])
    assert y.tolist() == want


def test_linear_zero_row_gives_positive_zero():
    x, q, s_a, wq, s_w = _tiny_case(4, 2, 8, 32, True)
    q[1] = 0
    s_a[1] = 1.0
    y = oracle.linear_w8a8(q, s_a, wq, s_w)
    assert np.all(y[1] == 0)


def test_linear_rows_are_batch_invariant():
    """Row r of an M-row call equals the one-row call on row r alone."""
    x = gen.act_bf16(9, 1, 8, 256, outliers=gen.outlier_channels(9, 256), gain=20.0)
    wq, s_w = oracle.quantize_weight(gen.weight_f32(9, 0, 0, 64, 256))
    q, s_a = oracle.quantize_act(x)
    full = oracle.linear_w8a8(q, s_a, wq, s_w)
    for r in range(8):
        q1, s1 = oracle.quantize_act(x[r:r + 1])
        assert np.array_equal(q1[0], q[r]) and s1[0] == s_a[r]
        assert np.array_equal(oracle.linear_w8a8(q1, s1, wq, s_w)[0], full[r])


def test_int32_bound(golden):
    g = golden("int32_bound.txt")
    kmax = int(g["max_k"])
    assert kmax * 127 * 127 == int(g["acc_at_max_k_all_127"]) < int(g["int32_limit"]) == 2 ** 31
    assert (kmax + 1) * 127 * 127 == int(g["acc_at_max_k_plus_1_all_127"]) >= 2 ** 31
    ones = np.ones(1, np.float32)
    q = np.full((1, kmax), 127, np.int8)
    y = oracle.linear_w8a8(q, ones, q.copy(), ones)
    assert y[0, 0] == oracle.f32_to_bf16_rne(float(np.float32(kmax * 16129)))
    q = np.full((1, kmax + 1), 127, np.int8)
    with pytest.raises(OverflowError):
        oracle.linear_w8a8(q, ones, q.copy(), ones)


# ---------------------------------------------------- epilogue fault catalogue

def _bf16_trunc(f: np.ndarray) -> np.ndarray:
    return (f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_rne(f: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _epilogue_variants(q, s_a, wq, s_w):
    """The correct epilogue and the five faults of Table II of "Deterministic
    LLM Inference Across GPU Kernels", in numpy/torch (not the oracle's code)."""
    acc = (q.astype(np.float64) @ wq.astype(np.float64).T)   # exact: |acc| < 2^53
    assert np.abs(acc).max() < 2 ** 31
    acc = acc.astype(np.int64)
    facc = acc.astype(np.int32).astype(np.float32)
    sa = s_a[:, None].astype(np.float32)
    sw = s_w[None, :].astype(np.float32)
    def bf16r(v):
        return gen.bf16_bits_to_f32(_bf16_rne(v))
    out = {"correct": _bf16_rne((facc * sa) * sw)}
    out["F1 scale precision"] = _bf16_rne((facc * bf16r(sa)) * bf16r(sw))
    out["F2 double rounding"] = _bf16_rne(bf16r(facc * sa) * sw)
    out["F3 scale order"] = _bf16_rne(facc * (sa * sw))
    out["F4 output truncation"] = _bf16_trunc((facc * sa) * sw)
    # F5: the per-column scale enters the reduction, which becomes an fp32 sum
    M, K = q.shape
    fsum = np.zeros((M, wq.shape[0]), np.float32)
    wscaled = wq.astype(np.float32) * s_w[:, None].astype(np.float32)
    for k in range(K):
        fsum += q[:, k:k + 1].astype(np.float32) * wscaled[None, :, k][0]
    out["F5 fused order"] = _bf16_rne(fsum * sa)
    return out


def test_epilogue_faults_are_caught_by_zero_ulp_compare():
    """Each single epilogue fault moves some outputs and the oracle's bitwise
    comparison flags every one.  F2-F4 provably stay within one bf16 spacing
    (a one-spacing tolerance is blind to them); F1 and F5 are measured and
    printed (the paper saw at most one spacing on its layers; these synthetic
    scales can reach two for F1)."""
    # F3 moves an output only when two fp32 values one fp32 step apart straddle
    # a bf16 rounding midpoint (about 1 output in 2^16), hence many outputs
    x, q, s_a, wq, s_w = _tiny_case(13, 8, 1 << 19, 64, pow2=False)
    y = oracle.linear_w8a8(q, s_a, wq, s_w)
    var = _epilogue_variants(q, s_a, wq, s_w)
    assert np.array_equal(var["correct"], y)
    for name, v in var.items():
        if name == "correct":
            continue
        d = ulp_dist_bf16(v, y)
        print(f"{name}: {int((d > 0).sum())} of {d.size} outputs moved, max {int(d.max())} ULP")
        assert d.max() >= 1, name                 # observable: 0-ULP compare fires
        if name in ("F2 double rounding", "F3 scale order", "F4 output truncation"):
            assert d.max() == 1, (name, d.max())  # within one spacing


def test_pow2_scales_make_f1_and_f3_vanish():
    """With power-of-two scales, bf16(s) = s and acc*(s_a*s_w) is exact, so F1
    and F3 cannot move an output: the reason pow2 scales give bitwise agreement
    across kernels with different scale handling."""
    x, q, s_a, wq, s_w = _tiny_case(14, 4, 512, 1024, pow2=True)
    s_a = np.exp2(np.round(np.log2(s_a))).astype(np.float32)
    var = _epilogue_variants(q, s_a, wq, s_w)
    assert np.array_equal(var["F1 scale precision"], var["correct"])
    assert np.array_equal(var["F3 scale order"], var["correct"])
    assert np.array_equal(var["F2 double rounding"], var["correct"])


# --------------------------------------------------------------- argmax

def test_bf16_tie_from_the_pages(golden):
    """Logits 30.0 / 29.875 pick the 30.0 row; a 29.875 / 29.875 tie picks the
    lower index.  With s_a = 1 (absmax 127) and s_w = 1/8, acc = 240 -> 30.0
    and acc = 239 -> 29.875 exactly."""
    g = golden("bf16_tie.txt")
    K = 16
    xrow = np.zeros(K)
    xrow[0], xrow[1] = 127.0, 1.0
    x = bf16_array(list(xrow))[None, :]
    q, s_a = oracle.quantize_act(x)
    assert s_a[0] == 1.0 and q[0, 0] == 127 and q[0, 1] == 1
    w = np.zeros((4, K), np.int8)
    w[:, 0] = 1
    w[0, 1], w[1, 1], w[2, 1], w[3, 1] = 100, 112, 113, 112   # acc 227, 239, 240, 239
    s_w = np.full(4, 0.125, np.float32)
    am, logits = oracle.lmhead_argmax(q, s_a, w, s_w)
    vals = gen.bf16_bits_to_f32(logits[0])
    assert float(vals[2]) == float(g["alone_top1"]) and float(vals[1]) == float(g["alone_top2"])
    assert am[0] == 2
    w[2, 1] = 112                                             # now rows 1, 2, 3 tie at 29.875
    am, logits = oracle.lmhead_argmax(q, s_a, w, s_w)
    assert float(gen.bf16_bits_to_f32(logits[0])[1]) == float(g["batched_top1"])
    assert am[0] == 1
    assert float(g["alone_top1"]) - float(g["alone_top2"]) == float(g["bf16_spacing_at_30"])


def test_argmax_matches_numpy_first_occurrence_and_signed_zero():
    rng = np.random.default_rng(17)
    K, N, M = 64, 300, 5
    q = rng.integers(-5, 6, (M, K), dtype=np.int8)
    w = rng.integers(-3, 4, (N, K), dtype=np.int8)
    w[10] = w[200]                                            # exact duplicate rows
    s_a = np.ones(M, np.float32)
    s_w = np.full(N, 0.5, np.float32)
    am, logits = oracle.lmhead_argmax(q, s_a, w, s_w)
    assert np.array_equal(am, np.argmax(gen.bf16_bits_to_f32(logits), axis=1))
    # -0 and +0 compare equal: an all-zero logit row picks index 0
    neg = np.full(N, -1.0, np.float32)
    q0 = np.zeros((1, K), np.int8)
    am0, lg0 = oracle.lmhead_argmax(q0, np.ones(1, np.float32), w, neg)
    assert am0[0] == 0 and set(np.unique(lg0[0])) <= {0x0000, 0x8000}


def test_lmhead_near_tie_workload_structure():
    """The generator's planted rows produce the intended ties on a reduced head
    (N = 4096): exact-copy rows tie in bf16 and the lower index wins."""
    N, K = 4096, 4096
    x = gen.activations(gen.LMHEAD_WL, 8, K)
    w = gen.lmhead_weight_f32(gen.LMHEAD_WL.seed, x, 0, N, N=N, K=K)
    wq, s_w = oracle.requant_pow2(*oracle.quantize_weight(w))
    q, s_a = oracle.quantize_act(x)
    am, logits = oracle.lmhead_argmax(q, s_a, wq, s_w)
    rows = gen.lmhead_special_rows(N)
    for m in (0, 4):
        a, b = rows[m]
        assert am[m] == min(a, b)
        assert logits[m, a] == logits[m, b]
    for m in (1, 5):
        a, b = rows[m]
        va, vb = gen.bf16_bits_to_f32(logits[m, [a, b]])
        assert abs(float(va) - float(vb)) <= 0.25
        assert am[m] in (a, b)


# --------------------------------------------------------------- chained pass

def _crafted_rows(K):
    """Rows of (h, y) bf16 patterns that reach the edge cases of the residual step."""
    rng = np.random.default_rng(77)
    rows = []
    h = gen.act_bf16(61, 1, 1, K)[0]
    y = gen.act_bf16(62, 1, 1, K, sigma=0.3)[0]
    rows.append((h, y))                                          # ordinary
    rows.append((np.zeros(K, np.uint16), np.zeros(K, np.uint16)))  # all +0: e = 0
    nz = np.full(K, 0x8000, np.uint16)
    rows.append((nz, nz.copy()))                                 # -0 + -0 stays -0
    rows.append((h, h ^ 0x8000))                                 # exact cancellation: +0
    tiny = np.array([bf16_pattern(v) for v in rng.choice([2.0 ** -130, -(2.0 ** -131), 3 * 2.0 ** -133, 0.0], K)],
                    np.uint16)
    rows.append((tiny, np.zeros(K, np.uint16)))                  # subnormal absmax: scale up by 2^130
    big = np.array([bf16_pattern(v) for v in rng.choice([2.0 ** 100, -3 * 2.0 ** 90, 2.0 ** -30, 1.5], K)],
                   np.uint16)
    rows.append((big, h))                                        # large values: scale down
    ones = np.full(K, bf16_pattern(1.0), np.uint16)
    ties = np.array([bf16_pattern(v) for v in rng.choice([2.0 ** -8, 3 * 2.0 ** -8, -(2.0 ** -9), 2.0 ** -7], K)],
                    np.uint16)
    rows.append((ones, ties))                                    # sums on bf16 ties
    mixed = np.array([bf16_pattern(v) for v in rng.choice([2.0 ** 100, 2.0 ** -30, -(2.0 ** -33), 3 * 2.0 ** -40,
                                                           -(2.0 ** -126), 255 * 2.0 ** -40], K)], np.uint16)
    rows.append((mixed, np.zeros(K, np.uint16)))                 # rescale pushes elements under the normal range
    return rows


def test_residual_rescale_against_exact_rational():
    K = 48
    rows = _crafted_rows(K)
    h = np.stack([r[0] for r in rows])
    y = np.stack([r[1] for r in rows])
    got = oracle.residual_rescale(h, y)
    for i in range(len(rows)):
        assert got[i].tolist() == ex.residual_rescale_row(h[i].tolist(), y[i].tolist()), i


def test_residual_rescale_row_stride_and_range():
    """y may be wider than h (its first K columns are added); a nonzero row ends
    with absmax in [1, 2), and the codes of per-row quantisation do not change."""
    M, K = 6, 256
    h = gen.act_bf16(63, 1, M, K, outliers=gen.outlier_channels(63, K), gain=20.0)
    y = gen.act_bf16(64, 1, M, 3 * K, sigma=4.0)
    got = oracle.residual_rescale(h, y)
    for m in range(M):
        assert got[m].tolist() == ex.residual_rescale_row(h[m].tolist(), y[m, :K].tolist())
        vals = gen.bf16_bits_to_f32(got[m])
        assert 1.0 <= np.abs(vals).max() < 2.0
        t = np.array(ex.residual_rescale_row(h[m].tolist(), y[m, :K].tolist()), np.uint16)
        # quantisation of the unscaled sum gives the same codes as of the rescaled row
        unscaled = oracle.f32_to_bf16_rne_array(gen.bf16_bits_to_f32(h[m]) + gen.bf16_bits_to_f32(y[m, :K]))
        qa, _ = oracle.quantize_act(unscaled[None, :])
        qb, _ = oracle.quantize_act(t[None, :])
        assert np.array_equal(qa, qb)


def test_relu_mul_against_exact_rational():
    rng = np.random.default_rng(78)
    M, K = 4, 40
    gu = gen.act_bf16(65, 1, M, 2 * K + 8, sigma=2.0)
    # signed zeros, negative gates, tiny products that leave the normal range
    special = [0.0, -0.0, -1.5, 2.0 ** -70, -(2.0 ** -70), 2.0 ** -66, 3.0, 2.0 ** 60]
    gu[0, :K] = [bf16_pattern(v) for v in rng.choice(special, K)]
    gu[0, K:2 * K] = [bf16_pattern(v) for v in rng.choice(special, K)]
    got = oracle.relu_mul(gu, K)
    for m in range(M):
        assert got[m].tolist() == ex.relu_mul_row(gu[m, :K].tolist(), gu[m, K:2 * K].tolist()), m


def _tiny_stack(seed, H=32, I=48, QR=32, KV=16, V=64, layers=2):
    def wq(layer, proj, N, K):
        q, s = oracle.quantize_weight(gen.weight_f32(seed, layer, proj, N, K))
        return oracle.requant_pow2(q, s)
    Ls = []
    for l in range(layers):
        Ls.append({"qkv": wq(l, 0, QR + 2 * KV, H), "o": wq(l, 3, H, QR),
                   "gu": wq(l, 4, 2 * I, H), "down": wq(l, 6, H, I)})
    head = wq(99, 0, V, H)
    return Ls, head, QR


def _exact_lin(q_rows, s_a, wq, s_w):
    return ex.linear(q_rows, [Fraction(float(v)) for v in s_a], wq.tolist(), [Fraction(float(v)) for v in s_w])


def _exact_quant(bits_rows):
    out_q, out_s = [], []
    for row in bits_rows:
        c, s = ex.quantize_row([ex.bf16_value(b) for b in row])
        out_q.append(c)
        out_s.append(s)
    return out_q, out_s


def test_verify_pass_tiny_against_exact_rational():
    """Two chained layers and the head, every step recomputed with exact rationals."""
    Ls, head, QR = _tiny_stack(5)
    M = 3
    h0 = gen.act_bf16(66, 1, M, 32, outliers=gen.outlier_channels(66, 32, 2), gain=20.0)
    am, h_end, recs = oracle.verify_pass(h0, Ls, head, QR, record=True)

    def lin(bits_rows, w):
        q, s = _exact_quant(bits_rows)
        return ex.linear(q, s, w[0].tolist(), [Fraction(float(v)) for v in w[1]])

    h = h0.tolist()
    for L, rec in zip(Ls, recs):
        y_qkv = lin(h, L["qkv"])
        assert rec["qkv"].tolist() == y_qkv
        y_o = lin([r[:QR] for r in y_qkv], L["o"])
        assert rec["o"].tolist() == y_o
        h = [ex.residual_rescale_row(hr, yr) for hr, yr in zip(h, y_o)]
        assert rec["h_mid"].tolist() == h
        y_gu = lin(h, L["gu"])
        assert rec["gu"].tolist() == y_gu
        inter = len(y_gu[0]) // 2
        m = [ex.relu_mul_row(r[:inter], r[inter:]) for r in y_gu]
        y_d = lin(m, L["down"])
        assert rec["down"].tolist() == y_d
        h = [ex.residual_rescale_row(hr, yr) for hr, yr in zip(h, y_d)]
        assert rec["h"].tolist() == h
    logits = lin(h, head)
    assert am.tolist() == [ex.argmax_bf16(r) for r in logits]
    assert h_end.tolist() == h


def test_verify_pass_rows_are_batch_invariant():
    """Each row of a 5-row chained pass equals the 1-row pass on that row alone,
    layer by layer."""
    Ls, head, QR = _tiny_stack(6, H=64, I=96, QR=64, KV=32, V=256, layers=3)
    h0 = gen.act_bf16(67, 1, 5, 64, outliers=gen.outlier_channels(67, 64), gain=20.0)
    am, h_end, recs = oracle.verify_pass(h0, Ls, head, QR, record=True)
    for r in range(5):
        am1, h1, recs1 = oracle.verify_pass(h0[r:r + 1], Ls, head, QR, record=True)
        assert am1[0] == am[r] and np.array_equal(h1[0], h_end[r])
        for a, b in zip(recs, recs1):
            for k in a:
                assert np.array_equal(a[k][r], b[k][0]), k


# --------------------------------------------------------------- greedy verify

def _plain_greedy_accept(argmax, draft):
    """Restatement from the definition: step through the drafts one position
    at a time, as plain greedy decoding would emit tokens."""
    emitted = []
    for i in range(len(argmax)):
        emitted.append(int(argmax[i]))
        if i == len(draft) or int(draft[i]) != int(argmax[i]):
            return i, emitted[-1]
    raise AssertionError


@pytest.mark.parametrize("M", [1, 2, 5, 8, 16])
def test_greedy_verify_against_step_by_step_restatement(M):
    rng = np.random.default_rng(90 + M)
    for trial in range(200):
        am = rng.integers(0, 6, M).astype(np.int32)      # a small vocabulary makes matches common
        dr = am[:M - 1].copy()
        cut = rng.integers(0, M)
        if cut < M - 1:
            dr[cut] = (dr[cut] + 1 + rng.integers(0, 4)) % 6
        got = oracle.greedy_verify(am, dr)
        assert got == _plain_greedy_accept(am, dr), (trial, am, dr)
        L, tok = got
        assert 0 <= L <= M - 1 and tok == am[L]
        assert all(am[i] == dr[i] for i in range(L))


def test_greedy_verify_edge_cases():
    assert oracle.greedy_verify(np.array([7], np.int32), np.array([], np.int32)) == (0, 7)       # decode: no drafts
    assert oracle.greedy_verify(np.array([3, 4, 5], np.int32), np.array([3, 4], np.int32)) == (2, 5)  # all accepted
    assert oracle.greedy_verify(np.array([3, 4, 5], np.int32), np.array([9, 4], np.int32)) == (0, 3)  # first rejected
