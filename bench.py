#!/usr/bin/env python3
"""Benchmark: one chained verify pass of a 36-layer Qwen3-8B-shaped W8A8 stack.

A step is one pass of the whole hot path over one batch of M tokens (the last
accepted token and M - 1 drafted ones): the
residual stream h (bf16 [M, 4096]) runs through 36 layers, each
    y_qkv = linear(quant(h), W_qkv)          q, k, v packed (6144 rows)
    y_o   = linear(quant(y_qkv[:, :4096]), W_o)   (q slice: attention stand-in)
    h     = rescale(bf16(h + y_o));  y_gu = linear(quant(h), W_gu)   gate, up packed
    y_d   = linear(quant(bf16(relu(gate) * up)), W_down)
    h     = rescale(bf16(h + y_d))
and then the LM head's greedy argmax over 151,936 rows with the greedy
verification of the drafts (accepted count and next token).  Every quantisation is
fused with the elementwise step before it.  Weights (7,568,097,280 bytes of
int8 plus power-of-two scales) come from the seeded recipe, are quantised on
the GPU and stay resident; the step reads all of them, far more than the L2
cache, so no explicit flush is needed.

`value` is weight GB/s over the step (weight codes + scales / step time) with
the step in a CUDA graph; `e2e` is the same metric measured on the host clock
with, every step, the input rows copied from pinned host memory, the library
call made through the C ABI, the argmax and verification result copied back
and waited for.  `per_config` times the public calls alone on every
configuration's shapes (one linear, each Qwen3-8B projection at M = 1..8, the
LM head at M = 1..8).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--m M] [--mode program|calls]
    python bench.py --impl reference     # the CPU oracle on a bounded sample

Under torchrun (N > 1) each rank runs an independent replica on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W8A8 verify-pass linear weight GB/s & % of HBM roofline at M=1–8, bit-exact"
UNIT = "GB/s"
WORKLOAD = "qwen3_8b_stack36_chained_verify_pass"

# DRAM traffic of the weight-streaming kernel from one ncu capture (bytes read +
# written per launch, scaled to the given launch) and the hash of the kernel
# source it was taken on; reported only while the source is unchanged.
NCU_TRAFFIC = {"source_sha256": "2bef6809b49ee2e7ade214a45bf08e5beb1f8b83a8f5de38b4fb6c5654d789d5",
               "bytes_per_launch": 7654890260,
               "launch": "program_kernel, M=8; captured at 3 layers (1,210,151,168 B read+written vs 1,208,084,868 B "
                         "algorithmic) and scaled by the algorithmic bytes to 36 layers"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--m", type=int, default=8, help="tokens per verify pass (1..16)")
    p.add_argument("--layers", type=int, default=36)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-sweep", action="store_true", help="skip the per-M sweep")
    p.add_argument("--prefill-only", type=int, default=0, metavar="M",
                   help="time only the prefill contraction at M tokens and print its figures")
    p.add_argument("--blockq-only", action="store_true",
                   help="time only the block-scaled variant and print its figures")
    p.add_argument("--attn-only", action="store_true",
                   help="time only the split-KV verify attention and print its figures")
    p.add_argument("--attn-cases", default="",
                   help="with --attn-only: comma-separated M:T0:copies cases (default: the four of the sweep)")
    p.add_argument("--mode", default="program", choices=["program", "calls"],
                   help="program: the step as one verify-pass program launch; calls: one launch per op")
    p.add_argument("--per-config-only", action="store_true",
                   help="time only the public calls on each configuration's shapes and print their figures")
    p.add_argument("--linear-only", default="", metavar="NAME:M",
                   help="time only one linear of the stack (q, k, v, o, gate, up, down, qkv, gu or head) at M "
                        "tokens, through bi_linear_w8a8 (bi_lmhead_argmax for head), rotating over the layers")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples (clocks and throttle reasons), each stamped with the
    host time it arrived, so that the ones taken during the timed region can be
    picked out afterwards."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.first = threading.Event()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self.first.wait(timeout=10.0)        # sampling is running before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line))
            self.first.set()

    def stop(self, t0, t1):
        """Summary of the samples taken in [t0, t1] (host monotonic seconds); if
        the region was shorter than the sampling period, the first sample after
        t0."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.samples:
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((t, float(f[1]), float(f[2]),
                             {n for n, v in zip(names, f[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:
            after = [r for r in rows if r[0] >= t0]
            inside = after[:1]
            window = "first sample after the timed region began"
        if not inside:
            return None
        reasons = set().union(*(r[3] for r in inside))
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ------------------------------------------------------------------- model

class Stack:
    """Resident int8 weights of the chained stack and the pass's buffers
    (sized for up to 16 tokens; a pass over M tokens uses the first M rows)."""

    H, QR, KV, I, V = 4096, 4096, 1024, 12288, 151936
    MAXM = 16

    def __init__(self, bi, torch, layers: int, device):
        import gen
        self.bi, self.torch, self.dev, self.layers = bi, torch, device, layers
        wl = gen.STACK36
        lins = {l.name: l for l in gen.QWEN3_8B_LINEARS}
        self.chunk = 8192
        self.stage = torch.empty(self.chunk * self.I, dtype=torch.float32).pin_memory()
        stage_np = self.stage.numpy()
        self.W = []        # per layer: group -> (wq, sw), member rows packed in order
        self.weight_bytes = 0
        for l in range(layers):
            d = {}
            for gname, members in gen.CHAIN_GROUPS:
                mats = [lins[m] for m in members]
                K = mats[0].K
                N = sum(m.N for m in mats)
                wq = torch.empty((N, K), dtype=torch.int8, device=device)
                sw = torch.empty(N, dtype=torch.float32, device=device)
                off = 0
                for m in mats:
                    self._quantise_rows(lambda r0, r, m=m, l=l: gen.weight_f32(
                        wl.seed, l, m.proj, m.N, m.K, row0=r0, rows=r, out=stage_np), m.N, K,
                        wq[off:off + m.N], sw[off:off + m.N])
                    off += m.N
                d[gname] = (wq, sw)
                self.weight_bytes += N * K + 4 * N
            self.W.append(d)
        hq = torch.empty((self.V, self.H), dtype=torch.int8, device=device)
        hs = torch.empty(self.V, dtype=torch.float32, device=device)
        self._quantise_rows(lambda r0, r: gen.weight_f32(wl.seed, 0, gen.LMHEAD.proj, self.V, self.H, row0=r0,
                                                         rows=r, out=stage_np), self.V, self.H, hq, hs)
        self.head = (hq, hs)
        self.weight_bytes += self.V * self.H + 4 * self.V
        del self.stage
        # the pass's input rows and buffers
        self.h0_np = gen.activations(wl, self.MAXM, self.H)
        t, M16 = torch, self.MAXM
        self.h0 = t.from_numpy(self.h0_np.view(np.int16)).to(device)
        self.h = t.empty((M16, self.H), dtype=t.int16, device=device)
        self.y, self.q, self.s = {}, {}, {}
        for name, N, K in (("qkv", self.QR + 2 * self.KV, self.H), ("o", self.H, self.QR),
                           ("gu", 2 * self.I, self.H), ("down", self.H, self.I), ("head", 0, self.H)):
            if N:
                self.y[name] = t.zeros((M16, N), dtype=t.int16, device=device)
            self.q[name] = t.empty((M16, K), dtype=t.int8, device=device)
            self.s[name] = t.empty(M16, dtype=t.float32, device=device)
        self.argmax = t.empty(M16, dtype=t.int32, device=device)
        # drafted tokens of the verify pass (synthetic) and the verification result
        self.draft = t.from_numpy(gen.u64(wl.seed, 11, M16).astype(np.int64) % self.V).to(t.int32).to(device)
        self.accept = t.zeros(2, dtype=t.int32, device=device)
        self.ws = bi.new_workspace(M16, self.V, self.I, device=device)
        torch.cuda.synchronize()

    def _quantise_rows(self, rows_fn, N, K, wq, sw):
        """Generate fp32 rows chunk by chunk into pinned memory and quantise
        them on the GPU (absmax, then power-of-two requantisation)."""
        torch, bi = self.torch, self.bi
        for r0 in range(0, N, self.chunk):
            r = min(self.chunk, N - r0)
            rows_fn(r0, r)
            w = self.stage[:r * K].view(r, K).to(self.dev, non_blocking=True)
            bi.bi_quantize_weight(w, wq[r0:r0 + r], sw[r0:r0 + r])
            bi.bi_requant_pow2(wq[r0:r0 + r], sw[r0:r0 + r], wq[r0:r0 + r], sw[r0:r0 + r])
            torch.cuda.synchronize()

    def ops(self, M):
        """The pass as executor ops, in order."""
        bi, y, q, s = self.bi, self.y, self.q, self.s
        h = self.h[:M]
        ops = [bi.op_quantize_act(h, q["qkv"][:M], s["qkv"][:M])]
        for l, W in enumerate(self.W):
            nxt = "head" if l == self.layers - 1 else "qkv"
            ops += [bi.op_linear(q["qkv"][:M], s["qkv"][:M], *W["qkv"], y["qkv"][:M]),
                    bi.op_quantize_act(y["qkv"][:M], q["o"][:M], s["o"][:M], K=self.QR),
                    bi.op_linear(q["o"][:M], s["o"][:M], *W["o"], y["o"][:M]),
                    bi.op_residual_quant(h, y["o"][:M], q["gu"][:M], s["gu"][:M]),
                    bi.op_linear(q["gu"][:M], s["gu"][:M], *W["gu"], y["gu"][:M]),
                    bi.op_relu_mul_quant(y["gu"][:M], self.I, q["down"][:M], s["down"][:M]),
                    bi.op_linear(q["down"][:M], s["down"][:M], *W["down"], y["down"][:M]),
                    bi.op_residual_quant(h, y["down"][:M], q[nxt][:M], s[nxt][:M])]
        ops.append(bi.op_lmhead(q["head"][:M], s["head"][:M], *self.head, None, self.argmax[:M],
                                draft=self.draft[:M - 1] if M > 1 else None, accept=self.accept))
        return ops

    def build_program(self, M):
        bi = self.bi
        ops = self.ops(M)
        prog = bi.new_program(len(ops), device=self.dev)
        bi.bi_program_build(ops, prog)
        return prog

    def reset(self, M):
        """Start the pass from the input rows (a device copy, part of the step)."""
        self.h[:M].copy_(self.h0[:M])

    def step_calls(self, M, flags, linears_only=False):
        """The same pass as one library call per op (or just its linears)."""
        bi, y, q, s, ws = self.bi, self.y, self.q, self.s, self.ws
        h = self.h[:M]
        if not linears_only:
            bi.bi_quantize_act(h, q["qkv"][:M], s["qkv"][:M], flags=flags)
        for l, W in enumerate(self.W):
            nxt = "head" if l == self.layers - 1 else "qkv"
            bi.bi_linear_w8a8(q["qkv"][:M], s["qkv"][:M], *W["qkv"], y["qkv"][:M], ws, flags=flags)
            if not linears_only:
                bi.bi_quantize_act(y["qkv"][:M], q["o"][:M], s["o"][:M], K=self.QR, flags=flags)
            bi.bi_linear_w8a8(q["o"][:M], s["o"][:M], *W["o"], y["o"][:M], ws, flags=flags)
            if not linears_only:
                bi.bi_residual_quantize(h, y["o"][:M], q["gu"][:M], s["gu"][:M], flags=flags)
            bi.bi_linear_w8a8(q["gu"][:M], s["gu"][:M], *W["gu"], y["gu"][:M], ws, flags=flags)
            if not linears_only:
                bi.bi_relu_mul_quantize(y["gu"][:M], self.I, q["down"][:M], s["down"][:M], flags=flags)
            bi.bi_linear_w8a8(q["down"][:M], s["down"][:M], *W["down"], y["down"][:M], ws, flags=flags)
            if not linears_only:
                bi.bi_residual_quantize(h, y["down"][:M], q[nxt][:M], s[nxt][:M], flags=flags)
        if not linears_only:
            bi.bi_lmhead_argmax(q["head"][:M], s["head"][:M], *self.head, None, self.argmax[:M], ws,
                                flags=flags)
            bi.bi_greedy_verify(self.argmax[:M], self.draft[:M - 1] if M > 1 else None, self.accept)

    def launches_per_step(self, mode):
        return 2 if mode == "program" else 3 + 8 * self.layers

    def op_bytes(self, op):
        """Algorithmic bytes of one op: what it must read and write."""
        bi = self.bi
        M, N, K = op.M, op.N, op.K
        if op.kind == bi.BI_OP_QUANTIZE_ACT:
            return 2 * M * K + M * K + 4 * M
        if op.kind == bi.BI_OP_RESIDUAL_QUANT:
            return 3 * 2 * M * K + M * K + 4 * M
        if op.kind == bi.BI_OP_RELU_MUL_QUANT:
            return 2 * 2 * M * K + M * K + 4 * M + (2 * M * K if op.y else 0)
        tot = N * K + 4 * N + M * K + 4 * M
        if op.kind == bi.BI_OP_LINEAR:
            return tot + 2 * M * N
        return tot + 4 * M + (2 * M * N if op.y else 0) + (4 * (M - 1) + 8 if op.accept else 0)

    def step_bytes(self, M):
        """Algorithmic bytes of one step: the input copy and every op."""
        return 4 * M * self.H + sum(self.op_bytes(o) for o in self.ops(M))

    def linear_bytes(self, M):
        bi = self.bi
        return sum(self.op_bytes(o) for o in self.ops(M) if o.kind == bi.BI_OP_LINEAR)


# The stack's projections as row slices of its packed weight groups:
# name -> (group, first row, rows).  K is the group's.
STACK_LINEARS = {"q": ("qkv", 0, 4096), "k": ("qkv", 4096, 1024), "v": ("qkv", 5120, 1024), "o": ("o", 0, 4096),
                 "gate": ("gu", 0, 12288), "up": ("gu", 12288, 12288), "down": ("down", 0, 4096),
                 "qkv": ("qkv", 0, 6144), "gu": ("gu", 0, 24576)}


def linear_measure(bi, torch, st, stream, peaks, name, M, reps=3):
    """One public call on one of the stack's shapes at M tokens, timed through
    the C ABI: bi_linear_w8a8 for a projection (the weights of layer l for the
    l-th call, so the matrices rotate over all the stack's layers, far more
    than L2), bi_lmhead_argmax for the head (622 MB, more than L2 by itself).
    A CUDA graph of the calls (programmatic dependent launch), timed with
    events on the launching stream; returns microseconds per call and weight
    GB/s."""
    import gen
    dev = st.dev
    peak = float(peaks["hbm_gbs"])
    if name == "head":
        wq, sw = st.head
        K, N, layers = wq.shape[1], wq.shape[0], [st.head]
    else:
        g, r0, n = STACK_LINEARS[name]
        layers = [(W[g][0][r0:r0 + n], W[g][1][r0:r0 + n]) for W in st.W]
        K, N = layers[0][0].shape[1], n
    x = torch.from_numpy(gen.activations(gen.QWEN3_8B, M, K).view(np.int16)).to(dev)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    s = torch.empty(M, dtype=torch.float32, device=dev)
    bi.bi_quantize_act(x, q, s)
    y = torch.empty((M, N), dtype=torch.int16, device=dev)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    calls = max(len(layers) * reps, 12)

    def enqueue():
        for i in range(calls):
            wq, sw = layers[i % len(layers)]
            if name == "head":
                bi.bi_lmhead_argmax(q, s, wq, sw, None, am, st.ws, flags=bi.BI_FLAG_PDL)
            else:
                bi.bi_linear_w8a8(q, s, wq, sw, y, st.ws, flags=bi.BI_FLAG_PDL)

    with torch.cuda.stream(stream):
        enqueue()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue()
    with torch.cuda.stream(stream):    # replays run on the current stream
        for _ in range(3):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_rep = 3
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_rep):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (n_rep * calls)
    wbytes = N * K + 4 * N
    gbs = wbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "weight_gbs": round(gbs, 1), "frac_of_hbm_copy": round(gbs / peak, 4),
            "N": N, "K": K, "weight_bytes": wbytes, "rotating_copies": len(layers)}


def per_config_measure(bi, torch, st, stream, peaks):
    """The public calls on the shapes of each workload configuration.

    single_linear: M = 2, K = N = 1024 (L2-resident: a latency case), the
    activation quantisation and the linear back to back in a CUDA graph.
    qwen3_8b_linears: every projection of a Qwen3-8B layer (and the packed
    q/k/v and gate/up groups the verify pass uses) at M in {1,2,3,4,5,8}.
    lm_head: bi_lmhead_argmax over 151,936 rows at M = 1..8."""
    import gen
    dev = st.dev
    out = {}
    # single linear (its own weights: the recipe of that configuration)
    wl = gen.SINGLE
    M, K, N = 2, 1024, 1024
    w = torch.from_numpy(gen.weight_f32(wl.seed, 0, 0, N, K)).to(dev)
    wq = torch.empty((N, K), dtype=torch.int8, device=dev)
    sw = torch.empty(N, dtype=torch.float32, device=dev)
    bi.bi_quantize_weight(w, wq, sw)
    bi.bi_requant_pow2(wq, sw, wq, sw)
    x = torch.from_numpy(gen.activations(wl, M, K).view(np.int16)).to(dev)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    s = torch.empty(M, dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.int16, device=dev)
    reps = 200

    def pair():
        for _ in range(reps):
            bi.bi_quantize_act(x, q, s, flags=bi.BI_FLAG_PDL)
            bi.bi_linear_w8a8(q, s, wq, sw, y, st.ws, flags=bi.BI_FLAG_PDL)

    def linear_alone():
        for _ in range(reps):
            bi.bi_linear_w8a8(q, s, wq, sw, y, st.ws, flags=bi.BI_FLAG_PDL)

    single = {}
    for key, fn in (("quantize_and_linear_us", pair), ("linear_us", linear_alone)):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        with torch.cuda.stream(stream):    # replays run on the current stream
            g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        single[key] = round(e0.elapsed_time(e1) * 1e3 / (5 * reps), 2)
    single["note"] = ("M=2, K=N=1024 (1 MB of weights: L2-resident), back to back in a CUDA graph with "
                      "programmatic dependent launch; a latency figure, not a roofline one")
    out["single_linear"] = single
    # the Qwen3-8B projections
    lins = {}
    for name in ("q", "k", "v", "o", "gate", "up", "down", "qkv", "gu"):
        lins[name] = {str(m): linear_measure(bi, torch, st, stream, peaks, name, m) for m in (1, 2, 3, 4, 5, 8)}
    out["qwen3_8b_linears"] = lins
    out["lm_head"] = {str(m): linear_measure(bi, torch, st, stream, peaks, "head", m) for m in range(1, 9)}
    out["note"] = ("each call through the C ABI (bi_linear_w8a8 / bi_lmhead_argmax); projections are row "
                   "slices of the stack's packed groups, layer l's weights for the l-th call (rotating over "
                   "all layers, more than L2); weight_gbs = (N*K + 4N) bytes / time per call")
    return out


def prefill_measure(bi, torch, st, stream, peaks, Ms=(512, 2048)):
    """The prefill contraction (M = 512 and 2048 tokens, K = 4096, N = 12288:
    layer 0's gate projection) through bi_linear_w8a8, timed alone: int
    operations per second against the measured dense bf16 tensor peak (the
    kernel runs the int8 products on the f16 tensor-core MMA)."""
    import gen
    out = {}
    K, N = 4096, 12288
    wq = st.W[0]["gu"][0][:N]
    sw = st.W[0]["gu"][1][:N]
    for Mp in Ms:
        x = torch.from_numpy(gen.activations(gen.PREFILL, Mp, K).view(np.int16)).to(st.dev)
        q = torch.empty((Mp, K), dtype=torch.int8, device=st.dev)
        s = torch.empty(Mp, dtype=torch.float32, device=st.dev)
        y = torch.empty((Mp, N), dtype=torch.int16, device=st.dev)
        ws = bi.new_workspace(Mp, N, K, device=st.dev)
        with torch.cuda.stream(stream):
            bi.bi_quantize_act(x, q, s)
            for _ in range(3):
                bi.bi_linear_w8a8(q, s, wq, sw, y, ws)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = 20
            e0.record(stream)
            for _ in range(reps):
                bi.bi_linear_w8a8(q, s, wq, sw, y, ws)
            e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tops = 2.0 * Mp * N * K / (ms * 1e-3) / 1e12
        out[str(Mp)] = {"ms": round(ms, 4), "tops": round(tops, 1),
                        "frac_of_bf16_peak": round(tops / float(peaks["bf16_tflops"]), 4)}
    out["note"] = ("y = W8A8(x) with K=4096, N=12288 through bi_linear_w8a8 (int8 x int8 -> exact int32: above "
                   "256 tokens a pass writes exact f16 copies of q and w into the workspace, then a persistent "
                   "TMA-fed tcgen05.mma kind::f16 kernel accumulates fp32 TMEM chunks of 1024 K into int32 "
                   "totals; the time includes the copy pass); peak = measured cuBLAS dense bf16, since "
                   "sm_103a's tcgen05 has no int8 kind")
    return out


def blockq_measure(bi, torch, dev, stream, peaks, Ms=(1, 8, 16)):
    """The block-scaled variant (q6-style weight blocks of 256, int8 activation
    blocks of 32, fixed fp32 order) on layer 0's gate/up shape (N = 24576,
    K = 4096) through bi_linear_q6, timed alone: stored weight bytes (codes,
    sub-scales, super-block scales) per second.  Four quantised copies of the
    weights rotate, so each call reads its weights from HBM, not L2."""
    import gen
    N, K, copies = 24576, 4096, 4
    w = torch.from_numpy(gen.weight_f32(gen.STACK36.seed, 0, 0, N, K)).to(dev)
    Ws = []
    for c in range(copies):
        ql = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        qh = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
        sc = torch.empty((N, K // 16), dtype=torch.int8, device=dev)
        d = torch.empty((N, K // 256), dtype=torch.float32, device=dev)
        bi.bi_quantize_weight_q6(w, ql, qh, sc, d)
        Ws.append((ql, qh, sc, d))
    del w
    wbytes = N * K // 2 + N * K // 4 + N * K // 16 + 4 * N * K // 256
    out = {}
    for M in Ms:
        x = torch.from_numpy(gen.activations(gen.STACK36, M, K).view(np.int16)).to(dev)
        q = torch.empty((M, K), dtype=torch.int8, device=dev)
        d_a = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        reps = 40
        with torch.cuda.stream(stream):
            bi.bi_quantize_act_blocks(x, q, d_a)
            for i in range(2 * copies):
                bi.bi_linear_q6(q, d_a, *Ws[i % copies], y)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(reps):
                bi.bi_linear_q6(q, d_a, *Ws[i % copies], y)
            e1.record(stream)
        stream.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        gbs = wbytes / (us * 1e-6) / 1e9
        out[str(M)] = {"us": round(us, 2), "weight_gbs": round(gbs, 1),
                       "frac_of_hbm_copy": round(gbs / float(peaks["hbm_gbs"]), 4)}
    out["note"] = ("y fp32 = block-scaled linear, N=24576, K=4096 (%d weight bytes: 6-bit codes, int8 sub-scales "
                   "per 16, fp32 scales per 256); %d rotating copies > L2" % (wbytes, copies))
    return out


def attention_measure(bi, torch, dev, stream, peaks, cases=((8, 4096, 36), (8, 32768, 4), (1, 4096, 36),
                                                            (16, 4096, 36))):
    """The split-KV verify attention of a Qwen3-8B-shaped layer (32 query heads
    over 8 kv heads of 128) through bi_attention_verify, timed alone, for
    (M queries, T0 cached positions, cache copies).  The copies (one per layer
    of a verify pass) rotate so that each call reads its cache from HBM; one
    pass over the copies is captured in a CUDA graph and replayed, so the time
    is the device's, not the Python caller's.  The path is bound by fp32
    issue: reported are microseconds per call, cache bytes per second, and
    the fused multiply-adds of the fixed-order sums (one per element of the
    scores and one per element of the weighted values: 2 D per query, head
    and visible position) per second against the SMs' fp32 rate (152 SMs x
    128 lanes x the 2.07 GHz clock)."""
    import gen
    Hq, Hkv, D = 32, 8, 128
    scale = 1.0 / math.sqrt(D)
    fma_peak = 152 * 128 * 2.07e9
    out = {}
    for M, T0, copies in cases:
        S = T0 + M
        q, k, v = gen.attn_qkv(gen.ATTENTION_SEED, M, Hq, Hkv, D, S)
        q_t = torch.from_numpy(q.view(np.int16)).to(dev)
        k0 = torch.from_numpy(k.view(np.int16)).to(dev)
        v0 = torch.from_numpy(v.view(np.int16)).to(dev)
        caches = [(k0.clone(), v0.clone()) for _ in range(copies)]
        del k0, v0
        o = torch.empty((M, Hq, D), dtype=torch.int16, device=dev)
        n = bi.bi_attention_workspace_size(M, Hq, D, T0)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            for i in range(copies):
                bi.bi_attention_verify(q_t, *caches[i], T0, scale, o, ws)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(copies):
                bi.bi_attention_verify(q_t, *caches[i], T0, scale, o, ws, stream=stream)
        replays = max(3, 360 // copies)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        us = e0.elapsed_time(e1) / (replays * copies) * 1e3
        kv_bytes = 2 * S * Hkv * D * 2
        fma = 2 * D * Hq * sum(T0 + m + 1 for m in range(M))
        out["M%d_T%d" % (M, T0)] = {
            "us": round(us, 2), "kv_gbs": round(kv_bytes / (us * 1e-6) / 1e9, 1),
            "frac_of_hbm_copy": round(kv_bytes / (us * 1e-6) / 1e9 / float(peaks["hbm_gbs"]), 4),
            "fma_tera_per_s": round(fma / (us * 1e-6) / 1e12, 2),
            "frac_of_fp32_fma_rate": round(fma / (us * 1e-6) / fma_peak, 4),
            "kv_bytes": kv_bytes, "fma": fma, "copies": copies}
        del caches, g
    out["note"] = ("Hq=32, Hkv=8, D=128, bf16 q/k/v ~ N(0,1); query m sees positions 0..T0+m; 256-position chunks "
                   "merged in order; rotating cache copies > L2; CUDA graph of one pass over the copies")
    return out


def own_ceilings(bi, torch, dev, stream, read_bytes=4 << 30, copy_bytes=2 << 30, reps=5):
    """The device's read-only and copy ceilings measured with the library's own
    probes (16-byte streaming loads, a grid of four 512-thread CTAs per SM),
    best of `reps`; copy counts read + written bytes like the driver's figure."""
    buf = torch.zeros(read_bytes, dtype=torch.uint8, device=dev)
    out = torch.zeros(1, dtype=torch.int64, device=dev)
    best_r = 0.0
    with torch.cuda.stream(stream):
        for i in range(reps + 1):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bi.bi_probe_read(buf, out, stream=stream)
            e1.record(stream)
            e1.synchronize()
            if i:
                best_r = max(best_r, read_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del buf
    src = torch.zeros(copy_bytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    best_c = 0.0
    with torch.cuda.stream(stream):
        for i in range(reps + 1):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bi.bi_probe_copy(src, dst, stream=stream)
            e1.record(stream)
            e1.synchronize()
            if i:
                best_c = max(best_c, 2 * copy_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del src, dst
    return {"read_gbs": round(best_r, 1), "copy_gbs": round(best_c, 1), "read_bytes": read_bytes,
            "copy_bytes": copy_bytes,
            "note": "bi_probe_read / bi_probe_copy, best of %d; copy counts read + written bytes" % reps}


def source_sha(path):
    """Hash of a kernel's source and the headers it is built from."""
    h = hashlib.sha256()
    d = os.path.dirname(path)
    for name in [os.path.basename(path), "ptx.cuh", "stream_mma.cuh", "row_ops.cuh", "kernels.cuh"]:
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def reduce_max(x, world, device):
    """The largest x over all ranks (x itself on one rank): the job's time is
    its slowest rank's."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(bytes_per_rank, world, ms):
    """Whole-job GB/s: every rank streams bytes_per_rank in ms (the max over ranks)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import invariant_quantized_linear_gb300 as bi

    M = args.m
    assert 1 <= M <= 16
    if args.attn_only:
        peaks, _ = read_peaks()
        if rank == 0:
            stream = torch.cuda.Stream(device=dev)
            kw = {}
            if args.attn_cases:
                kw["cases"] = tuple(tuple(int(x) for x in c.split(":")) for c in args.attn_cases.split(","))
            print(json.dumps({"attention": attention_measure(bi, torch, dev, stream, peaks, **kw)}), flush=True)
        return
    t0 = time.time()
    st = Stack(bi, torch, args.layers, dev)
    setup_s = time.time() - t0
    flags = bi.BI_FLAG_PDL
    stream = torch.cuda.Stream(device=dev)
    if args.blockq_only:
        peaks, _ = read_peaks()
        if rank == 0:
            print(json.dumps({"block_scaled": blockq_measure(bi, torch, dev, stream, peaks)}), flush=True)
        return
    if args.prefill_only:
        peaks, _ = read_peaks()
        if rank == 0:
            print(json.dumps({"prefill": prefill_measure(bi, torch, st, stream, peaks, Ms=(args.prefill_only,))}),
                  flush=True)
        return
    if args.per_config_only:
        peaks, _ = read_peaks()
        if rank == 0:
            print(json.dumps({"per_config": per_config_measure(bi, torch, st, stream, peaks)}), flush=True)
        return
    if args.linear_only:
        peaks, _ = read_peaks()
        name, m = args.linear_only.split(":")
        if rank == 0:
            print(json.dumps({"linear": {name: {m: linear_measure(bi, torch, st, stream, peaks, name, int(m))}}}),
                  flush=True)
        return

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    progs = {}
    prog_ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=dev)

    def enqueue_step(m):
        st.reset(m)
        if args.mode == "program":
            if m not in progs:
                progs[m] = st.build_program(m)
            bi.bi_program_run(progs[m], m, prog_ws)
        else:
            st.step_calls(m, flags)

    def graph_for(m):
        with torch.cuda.stream(stream):
            enqueue_step(m)            # warm-up outside capture (tensor maps, attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue_step(m)
        return g

    region = {}

    def time_graph(g, steps, warmup):
        for _ in range(warmup):
            g.replay()
        barrier()
        region["t0"] = time.monotonic()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
        barrier()
        region["t1"] = time.monotonic()
        return reduce_max(e0.elapsed_time(e1) / steps, world, dev)

    g = graph_for(M)
    clocks = ClockSampler(local)
    ms = time_graph(g, args.steps, args.warmup)
    clk = clocks.stop(region["t0"], region["t1"])
    gbs = job_rate(st.weight_bytes, world, ms)

    # per-M sweep (same step, fewer repetitions)
    per_m = {}
    if not args.no_sweep:
        for m in (1, 2, 3, 4, 5, 8):
            gm = g if m == M else graph_for(m)
            msm = time_graph(gm, max(5, args.steps // 2), 3)
            per_m[str(m)] = {"ms_per_step": round(msm, 4),
                             "weight_gbs": round(st.weight_bytes / (msm * 1e-3) / 1e9, 1),
                             "tokens_per_s_eq": round(m / (msm * 1e-3), 1)}

    if args.mode == "program":
        # dominant kernel: the program kernel itself, one launch per step;
        # its average duration is the step time measured above
        kernel_name = "program_kernel (bi_program_run, M<=16)"
        lin_launches = 1
        lin_ms = ms
        achieved = st.step_bytes(M) / (ms * 1e-3) / 1e9
        note = ("achieved = algorithmic bytes of the step (all weights and scales, activations read and "
                "written, outputs) / the program launch's event-timed duration")
    else:
        # dominant kernel: the step's weight-streaming linear launches alone,
        # back to back in a CUDA graph (same launch configuration as the step),
        # timed with events on the launching stream
        with torch.cuda.stream(stream):
            st.step_calls(M, flags, linears_only=True)
        stream.synchronize()
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl, stream=stream):
            st.step_calls(M, flags, linears_only=True)
        kernel_name = "skinny_kernel (bi_linear_w8a8, M<=16)"
        lin_launches = st.layers * 4
        lin_ms = time_graph(gl, max(5, args.steps // 2), 3)
        achieved = st.linear_bytes(M) / (lin_ms * 1e-3) / 1e9
        note = ("achieved = algorithmic bytes (W + s_w + q + s_a + y) of the step's %d linear launches / "
                "their event-timed duration back to back in a CUDA graph" % lin_launches)

    # end to end through the public API, as a verify loop runs it: every step
    # copies its input rows host->device from pinned memory, makes the library
    # call (bi_program_run; in calls mode one call per op), copies the argmax
    # and the verification result back, and waits for them on the host
    host_h0 = torch.from_numpy(st.h0_np.view(np.int16)).pin_memory()
    host_am = torch.empty(16, dtype=torch.int32).pin_memory()
    host_acc = torch.empty(2, dtype=torch.int32).pin_memory()
    h2d = int(host_h0[:M].numel()) * 2
    e2e_steps = max(3, args.steps // 2)
    with torch.cuda.stream(stream):
        enqueue_step(M)
    barrier()
    t_e2e = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            st.h0[:M].copy_(host_h0[:M], non_blocking=True)
            enqueue_step(M)
            host_am[:M].copy_(st.argmax[:M], non_blocking=True)
            host_acc.copy_(st.accept, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t_e2e) * 1e3 / e2e_steps
    e2e_ms = reduce_max(e2e_ms, world, dev)
    e2e_gbs = job_rate(st.weight_bytes, world, e2e_ms)

    peaks, kind = read_peaks()
    peak = float(peaks["hbm_gbs"])
    src = os.path.join(ROOT, "invariant_quantized_linear_gb300", "csrc",
                       "k_program.cu" if args.mode == "program" else "k_skinny.cu")
    traffic = None
    if NCU_TRAFFIC["source_sha256"] == source_sha(src):
        traffic = NCU_TRAFFIC["bytes_per_launch"]

    per_config = per_config_measure(bi, torch, st, stream, peaks) if not args.no_sweep else None
    prefill = prefill_measure(bi, torch, st, stream, peaks) if not args.no_sweep else None
    block_scaled = blockq_measure(bi, torch, dev, stream, peaks) if not args.no_sweep else None
    attention = attention_measure(bi, torch, dev, stream, peaks) if not args.no_sweep else None
    ceilings = own_ceilings(bi, torch, dev, stream) if not args.no_sweep else None
    cpu = cpu_baseline(bounded_s=12.0) if rank == 0 else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8", "data": "synthetic (seeded; fp32 N(0,0.02) weights -> absmax int8 -> pow2 scales; "
                                     "bf16 N(0,1) activations)",
            "config": {"workload": WORKLOAD, "M": M, "layers": args.layers, "hidden": 4096,
                       "intermediate": 12288, "vocab": 151936, "weight_bytes_per_step": st.weight_bytes,
                       "l2": "inputs larger than L2 (all weights read once per step)",
                       "activations": ("chained: residual stream through 36 layers (q slice of q/k/v as the "
                                       "attention stand-in, ReLU-gated MLP, power-of-two row rescale)"),
                       "packing": "q/k/v and gate/up weight rows packed: one call per group",
                       "verify": "greedy verification of M - 1 synthetic drafted tokens fused into the LM head",
                       "launch": ("one verify-pass program launch per step (persistent cooperative kernel, "
                                  "grid barrier between ops) after a device copy of the input rows, then a "
                                  "one-warp greedy-verify kernel, in a CUDA graph" if args.mode == "program" else
                                  "CUDA graph of the step, one launch per op, programmatic dependent launch"),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "pct_of_hbm_copy": round(100 * gbs / world / peak, 1),
            "tokens_per_s_eq": round(M * world / (ms * 1e-3), 1),
            "per_m": per_m,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": kernel_name,
                         "launch_us": round(lin_ms * 1e3 / lin_launches, 3),
                         "peak_kind": kind, "note": note},
            "e2e": {"value": round(e2e_gbs, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": 4 * M + 8, "ms_per_step": round(e2e_ms, 4),
                    "how": ("host wall clock per step: H2D of the input rows from pinned memory, the "
                            "library call through the C ABI (no graph), D2H of argmax and verification "
                            "result, host waits for the result every step")},
            "gpu_launches": st.launches_per_step(args.mode) * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "per_config": per_config,
            "prefill": prefill,
            "block_scaled": block_scaled,
            "attention": attention,
            "own_ceilings": ceilings,
            "frac_of_own_read_ceiling": round(achieved / ceilings["read_gbs"], 4) if ceilings else None,
            "setup_s": round(setup_s, 1),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ CPU oracle

def oracle_sample():
    """A bounded sample of the workload for the CPU oracle: layer 0 of the
    chained stack (all four packed linears and the fused elementwise steps),
    weights generated from the same recipe and quantised by the oracle."""
    import gen
    import oracle
    wl = gen.STACK36
    L = {}
    for gname, _ in gen.CHAIN_GROUPS:
        w = gen.chain_group_f32(wl.seed, 0, gname)
        L[gname] = oracle.requant_pow2(*oracle.quantize_weight(w))
        del w
    layer_bytes = sum(wq.size + 4 * sw.size for wq, sw in L.values())
    h0 = gen.activations(wl, Stack.MAXM, Stack.H)
    return oracle, L, h0, layer_bytes


def _oracle_layer(oracle, L, h0, M):
    oracle.chain_layer(h0[:M], L, Stack.QR)


def cpu_baseline(bounded_s=12.0, M=8):
    oracle, L, h0, layer_bytes = oracle_sample()
    t0 = time.time()
    n = 0
    while True:
        _oracle_layer(oracle, L, h0, M)
        n += 1
        if time.time() - t0 >= bounded_s:
            break
    dt = (time.time() - t0) / n
    total = time.time() - t0
    # the verify attention of one layer (M = 8 after 4096 positions) on the same cores
    import gen
    q, k, v = gen.attn_qkv(gen.ATTENTION_SEED, 8, 32, 8, 128, 4104)
    ta, na = time.time(), 0
    while na < 1 or time.time() - ta < 2.0:
        oracle.attention(q, k, v, 4096, 1.0 / math.sqrt(128))
        na += 1
    attn_us = (time.time() - ta) / na * 1e6
    # the same layer on one thread, bounded to a few seconds
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    t1, n1 = time.time(), 0
    while n1 < 1 or time.time() - t1 < 3.0:
        _oracle_layer(oracle, L, h0, M)
        n1 += 1
    one_thread = layer_bytes / ((time.time() - t1) / n1) / 1e9
    oracle.set_num_threads(cores)
    return {"value": round(layer_bytes / dt / 1e9, 3), "unit": UNIT,
            "cores": cores, "kind": "oracle", "one_thread_value": round(one_thread, 3),
            "sample": "layer 0 of the chained stack (q/k/v, o, gate/up, down with the fused quantisation, "
                      "residual and MLP steps; %d weight bytes) at M=%d, repeated %d times in %.1f s"
                      % (layer_bytes, M, n, total),
            "attention": {"us": round(attn_us, 1), "calls": na,
                          "sample": "verify attention of one Qwen3-8B-shaped layer (32/8 heads of 128), M = 8 "
                                    "after 4096 positions, oracle on the same cores"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    oracle, L, h0, layer_bytes = oracle_sample()
    M = args.m
    for _ in range(args.warmup):
        _oracle_layer(oracle, L, h0, M)
    t0 = time.time()
    for _ in range(args.steps):
        _oracle_layer(oracle, L, h0, M)
    dt = (time.time() - t0) / args.steps
    v = layer_bytes / dt / 1e9
    sample = ("one step = layer 0 of the chained stack (%d weight bytes) at M=%d on the CPU oracle"
              % (layer_bytes, M))
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": M},
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
