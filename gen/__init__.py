"""Seeded synthetic inputs for the W8A8 verify-pass linear workloads.

This module is shared by the CPU oracle (through the tests) and by the GPU
library's tests and benchmark.  It holds no step of the method: it produces
raw fp32 weights and bf16 activations (plus the near-tie row structure of the
LM-head workload), never quantised codes, scales or outputs.

Workloads (shapes and seeds; every one synthetic, no checkpoint or dataset):

* ``single``     - one linear, M=2, K=N=1024, seed 0, power-of-two scales.
* ``qwen3_8b``   - the seven linears of a Qwen3-8B-shaped layer (hidden 4096,
  GQA 32/8 heads of 128, intermediate 12288), seed 1, the weights' own
  absmax scales, M in {1,2,3,4,5,8}.
* ``lmhead``     - LM head 4096 -> 151936, power-of-two scales, seed 2,
  M = 1..8, with near-tie rows injected.
* ``stack36``    - all linears of a 36-layer Qwen3-8B-shaped stack plus the
  LM head, power-of-two scales, seed 3, M in {1,5}.
* ``prefill``    - M in {512, 2048}, K=4096, N=12288, seed 4.
* ``attention``  - verify-pass attention of a Qwen3-8B-shaped layer: 32 query
  heads over 8 kv heads of 128, M = 8 queries after T0 = 4096 cached
  positions, seed 5; q, k, v ~ N(0, 1) as bf16 (``attn_qkv``).

Weights are ~N(0, 0.02) and activations ~N(0, 1) (Irwin-Hall(8) approximation,
see gen.c); ``single``, ``qwen3_8b`` and ``prefill`` activations carry four
outlier channels scaled by 20.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.gen_key.argtypes = [u64, u64]
        L.gen_key.restype = u64
        L.gen_draw.argtypes = [u64, u64]
        L.gen_draw.restype = u64
        L.gen_normal_f32.argtypes = [u64, u64, i64, i64, dbl, vp]
        L.gen_normal_f32.restype = None
        L.gen_u64.argtypes = [u64, u64, i64, i64, vp]
        L.gen_u64.restype = None
        L.gen_act_bf16.argtypes = [u64, u64, i64, i64, i64, i64, dbl, vp, ctypes.c_int, dbl, vp]
        L.gen_act_bf16.restype = None
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---------------------------------------------------------------- primitives

def normal_f32(seed: int, stream: int, count: int, sigma: float, offset: int = 0,
               out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(count, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == count
    lib().gen_normal_f32(seed, stream, offset, count, sigma, _ptr(out))
    return out


def u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    lib().gen_u64(seed, stream, offset, count, _ptr(out))
    return out


def outlier_channels(seed: int, K: int, n: int = 4) -> np.ndarray:
    """n distinct channel indices in [0, K), drawn from stream 2 of `seed`."""
    chosen: list[int] = []
    j = 0
    while len(chosen) < n:
        c = int(u64(seed, 2, 1, offset=j)[0] % np.uint64(K))
        j += 1
        if c not in chosen:
            chosen.append(c)
    return np.array(chosen, dtype=np.int64)


def act_bf16(seed: int, stream: int, rows: int, cols: int, sigma: float = 1.0,
             outliers=(), gain: float = 20.0, row0: int = 0, ld: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of shape [rows, ld]; columns >= cols are zero."""
    ld = cols if ld is None else ld
    assert ld >= cols
    out = np.zeros((rows, ld), dtype=np.uint16)
    o = np.ascontiguousarray(np.asarray(outliers, dtype=np.int64))
    lib().gen_act_bf16(seed, stream, row0, rows, cols, ld, sigma,
                       _ptr(o) if o.size else None, int(o.size), gain, _ptr(out))
    return out


ATTENTION_SEED = 5


def attn_qkv(seed: int, M: int, Hq: int, Hkv: int, D: int, S: int, sigma_q: float = 1.0,
             sigma_k: float = 1.0) -> tuple:
    """bf16 bit patterns of q [M, Hq, D] (stream 20), k [S, Hkv, D] (stream 21,
    standard deviation sigma_k) and v [S, Hkv, D] (stream 22, N(0, 1))."""
    q = act_bf16(seed, 20, M, Hq * D, sigma_q).reshape(M, Hq, D)
    k = act_bf16(seed, 21, S, Hkv * D, sigma_k).reshape(S, Hkv, D)
    v = act_bf16(seed, 22, S, Hkv * D, 1.0).reshape(S, Hkv, D)
    return q, k, v


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a bit shift, no rounding)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- workloads

WEIGHT_SIGMA = 0.02
ACT_SIGMA = 1.0
OUTLIER_GAIN = 20.0
STREAM_ACT = 1


def weight_stream(layer: int, proj: int) -> int:
    return 1000 + 16 * layer + proj


@dataclass(frozen=True)
class Linear:
    name: str
    K: int
    N: int
    proj: int  # index of the weight stream inside a layer


QWEN3_8B_LINEARS = (
    Linear("q", 4096, 4096, 0),
    Linear("k", 4096, 1024, 1),
    Linear("v", 4096, 1024, 2),
    Linear("o", 4096, 4096, 3),
    Linear("gate", 4096, 12288, 4),
    Linear("up", 4096, 12288, 5),
    Linear("down", 12288, 4096, 6),
)
LMHEAD = Linear("lm_head", 4096, 151936, 15)
HIDDEN = 4096
INTERMEDIATE = 12288
N_LAYERS = 36


# A layer of the chained verify pass: members that read the same input are
# stored as one packed weight matrix (rows of the members back to back, in
# this order), so each group is one linear.
CHAIN_GROUPS = (("qkv", ("q", "k", "v")), ("o", ("o",)), ("gu", ("gate", "up")), ("down", ("down",)))


def chain_linears(H: int, QR: int, KV: int, I: int) -> tuple:
    """The seven projections of a layer with hidden H, q rows QR, k/v rows KV
    and intermediate I (Qwen3-8B: 4096, 4096, 1024, 12288), with the weight
    stream indices of QWEN3_8B_LINEARS."""
    return (Linear("q", H, QR, 0), Linear("k", H, KV, 1), Linear("v", H, KV, 2), Linear("o", QR, H, 3),
            Linear("gate", H, I, 4), Linear("up", H, I, 5), Linear("down", I, H, 6))


def chain_group_f32(seed: int, layer: int, group: str, linears=QWEN3_8B_LINEARS) -> np.ndarray:
    """fp32 weights of one packed group of a layer: its members' matrices
    (each from its own weight stream) stacked in CHAIN_GROUPS order."""
    byname = {l.name: l for l in linears}
    members = dict(CHAIN_GROUPS)[group]
    mats = [weight_f32(seed, layer, byname[m].proj, byname[m].N, byname[m].K) for m in members]
    return mats[0] if len(mats) == 1 else np.concatenate(mats, axis=0)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    pow2: bool
    outliers: bool
    Ms: tuple = field(default_factory=tuple)


SINGLE = Workload("single", 0, True, True, (2,))
QWEN3_8B = Workload("qwen3_8b", 1, False, True, (1, 2, 3, 4, 5, 8))
LMHEAD_WL = Workload("lmhead", 2, True, False, tuple(range(1, 9)))
STACK36 = Workload("stack36", 3, True, False, (1, 5))
PREFILL = Workload("prefill", 4, True, True, (512, 2048))


def weight_f32(seed: int, layer: int, proj: int, N: int, K: int, row0: int = 0,
               rows: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+rows) of an fp32 weight matrix W[N, K] ~ N(0, 0.02).
    `out`, if given, is a float32 buffer of at least rows*K elements."""
    rows = N - row0 if rows is None else rows
    if out is not None:
        out = out.reshape(-1)[:rows * K]
    flat = normal_f32(seed, weight_stream(layer, proj), rows * K, WEIGHT_SIGMA, offset=row0 * K, out=out)
    return flat.reshape(rows, K)


def activations(wl: Workload, rows: int, K: int, stream: int = STREAM_ACT, ld: int | None = None) -> np.ndarray:
    outl = outlier_channels(wl.seed, K) if wl.outliers else ()
    return act_bf16(wl.seed, stream, rows, K, ACT_SIGMA, outl, OUTLIER_GAIN, ld=ld)


# LM-head near ties.  For activation row m (m < 8) the generator plants a
# "dominant" weight row aligned with the signs of x[m] (so it very likely wins
# the argmax) and a second row that is either an exact copy (m % 4 == 0) or a
# copy with one element nudged at the channel where |x[m]| is closest to 0.1
# (m % 4 == 1), giving a top-2 logit gap far below 0.01.  Rows m % 4 in {2, 3}
# keep their natural argmax.  Half of the copies sit below the dominant row,
# half above, so the lowest-index tie-break is exercised both ways.
def lmhead_special_rows(N: int) -> dict:
    rows = {}
    for m in range(8):
        a = (N // 8) * m + N // 16 + 3 * m
        if m % 4 in (0, 1):
            b = a - N // 64 if (m // 4) == 0 else a + N // 64
            rows[m] = (a, b)
        else:
            rows[m] = (a, None)
    return rows


def lmhead_weight_f32(seed: int, x_bf16: np.ndarray, row0: int, rows: int,
                      N: int = LMHEAD.N, K: int = LMHEAD.K, out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+rows) of the LM-head weights, near-tie rows included.

    x_bf16 holds the (up to 8) activation rows the ties are planted for."""
    W = weight_f32(seed, 0, LMHEAD.proj, N, K, row0=row0, rows=rows, out=out)
    xs = bf16_bits_to_f32(x_bf16[:, :K])
    mag = np.abs(normal_f32(seed, 9, 8 * K, WEIGHT_SIGMA).reshape(8, K))
    for m, (a, b) in lmhead_special_rows(N).items():
        if m >= xs.shape[0]:
            continue
        dom = (np.sign(xs[m]) * mag[m]).astype(np.float32)
        dom[dom == 0] = np.float32(WEIGHT_SIGMA)
        if row0 <= a < row0 + rows:
            W[a - row0] = dom
        if b is not None and row0 <= b < row0 + rows:
            cp = dom.copy()
            if m % 4 == 1:
                kstar = int(np.argmin(np.abs(np.abs(xs[m]) - np.float32(0.1))))
                cp[kstar] = np.float32(cp[kstar] + np.float32(3 * WEIGHT_SIGMA))
            W[b - row0] = cp
    return W
