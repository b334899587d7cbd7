#!/usr/bin/env python3
"""Benchmark: one verify pass of a 36-layer Qwen3-8B-shaped W8A8 stack.

A step is one pass of the whole hot path over one batch of M tokens: for each
of 36 layers, per-token activation quantisation of each linear's input and the
seven linears (q, k, v, o, gate, up, down), then quantisation of the head input
and the LM head with its greedy argmax.  Weights (7,568,097,280 bytes of int8,
power-of-two scales) are generated from the seeded recipe, quantised on the
GPU, and stay resident; the step reads all of them, which is far more than the
L2 cache, so no explicit flush is needed.  Each linear gets its own synthetic
bf16 activations (layers are not chained).

`value` is weight GB/s over the step (weight codes + scales / step time) with
the step captured as a CUDA graph; `e2e` is the same metric measured through
the C-ABI entry points with the step's activations copied from pinned host
memory and the argmax copied back inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--m M] [--impl reference]

Under torchrun (N > 1) each rank runs an independent replica on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
WORKLOAD = "qwen3_8b_stack36_verify_pass"

# DRAM traffic of the weight-streaming kernel from one ncu capture (bytes read +
# written per launch, scaled to the given launch) and the hash of the kernel
# source it was taken on; reported only while the source is unchanged.
NCU_TRAFFIC = {"source_sha256": None, "bytes_per_launch": None, "launch": None}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--m", type=int, default=8, help="tokens per verify pass (1..16)")
    p.add_argument("--layers", type=int, default=36)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-sweep", action="store_true", help="skip the per-M sweep")
    p.add_argument("--mode", default="program", choices=["program", "calls"],
                   help="program: the step as one verify-pass program launch; calls: one launch per op")
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
    """Resident int8 weights of the stack and per-step activation buffers."""

    def __init__(self, bi, torch, layers: int, M: int, device):
        import gen
        self.bi, self.torch, self.M, self.dev = bi, torch, M, device
        self.layers = layers
        wl = gen.STACK36
        self.lin = gen.QWEN3_8B_LINEARS
        # Per layer, q/k/v share one input and so do gate/up: their weight
        # rows are stored back to back ("packed") and each group is one call.
        # Rows are independent, so the outputs are the same bits as separate
        # calls.
        self.groups = [("qkv", ("q", "k", "v"), 4096), ("o", ("o",), 4096), ("gu", ("gate", "up"), 4096),
                       ("down", ("down",), 12288)]
        byname = {l.name: l for l in self.lin}
        self.W = []       # per layer: dict group -> (wq, sw) with the group's rows packed
        self.chunk = 8192
        self.stage = torch.empty(self.chunk * 12288, dtype=torch.float32).pin_memory()
        stage_np = self.stage.numpy()
        for l in range(layers):
            d = {}
            for gname, members, K in self.groups:
                parts = [self._make_weight(lambda r0, r, lin=byname[m], l=l: gen.weight_f32(
                    wl.seed, l, lin.proj, lin.N, lin.K, row0=r0, rows=r, out=stage_np), byname[m].N, K)
                    for m in members]
                if len(parts) == 1:
                    d[gname] = parts[0]
                else:
                    d[gname] = (torch.cat([p[0] for p in parts]), torch.cat([p[1] for p in parts]))
                    del parts
            self.W.append(d)
        # LM head with the planted near-tie rows for the head's activation rows
        self.x_head_np = gen.activations(wl, 16, gen.LMHEAD.K, stream=7)
        xh = self.x_head_np[:8]
        self.head = self._make_weight(lambda r0, r: gen.lmhead_weight_f32(wl.seed, xh, r0, r, out=stage_np),
                                      gen.LMHEAD.N, gen.LMHEAD.K)
        del self.stage
        self.weight_bytes = sum(l.N * l.K + 4 * l.N for l in self.lin) * layers + \
            gen.LMHEAD.N * gen.LMHEAD.K + 4 * gen.LMHEAD.N
        # activations: inputs of q/k/v, o, gate/up, down per layer, and the head
        self.in_dims = [(g, K) for g, _, K in self.groups]
        self.x_np = {}
        self.x = {}
        for l in range(layers):
            for j, (nm, K) in enumerate(self.in_dims):
                a = gen.activations(wl, 16, K, stream=100 + 4 * l + j)
                self.x_np[(l, nm)] = a
                self.x[(l, nm)] = torch.from_numpy(a.view(np.int16)).to(device)
        self.x[("head",)] = torch.from_numpy(self.x_head_np.view(np.int16)).to(device)
        self.x_np[("head",)] = self.x_head_np
        self.ws = bi.new_workspace(16, 151936, 12288, device=device)
        self.q = torch.empty((16, 12288), dtype=torch.int8, device=device)
        self.s = torch.empty(16, dtype=torch.float32, device=device)
        self.y = {g: torch.empty((16, self.W[0][g][0].shape[0]), dtype=torch.int16, device=device)
                  for g, _, _ in self.groups}
        self.argmax = torch.empty(16, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def _make_weight(self, rows_fn, N, K):
        torch, bi = self.torch, self.bi
        wq = torch.empty((N, K), dtype=torch.int8, device=self.dev)
        sw = torch.empty(N, dtype=torch.float32, device=self.dev)
        for r0 in range(0, N, self.chunk):
            r = min(self.chunk, N - r0)
            rows_fn(r0, r)                      # fills the pinned staging buffer
            w = self.stage[:r * K].view(r, K).to(self.dev, non_blocking=True)
            bi.bi_quantize_weight(w, wq[r0:r0 + r], sw[r0:r0 + r])
            bi.bi_requant_pow2(wq[r0:r0 + r], sw[r0:r0 + r], wq[r0:r0 + r], sw[r0:r0 + r])
            torch.cuda.synchronize()
        return wq, sw

    def build_program(self, M):
        """The step as one verify-pass program (bi_program_*): the same ops,
        in the same order, each starting after all earlier ones."""
        bi = self.bi
        ops = []
        s = self.s[:M]
        for l in range(self.layers):
            for nm, K in self.in_dims:
                qbuf = self.q.view(-1)[:M * K].view(M, K)
                ops.append(bi.op_quantize_act(self.x[(l, nm)][:M, :K], qbuf, s, K=K))
                wq, sw = self.W[l][nm]
                ops.append(bi.op_linear(qbuf, s, wq, sw, self.y[nm][:M]))
        K = 4096
        qbuf = self.q.view(-1)[:M * K].view(M, K)
        ops.append(bi.op_quantize_act(self.x[("head",)][:M], qbuf, s, K=K))
        wq, sw = self.head
        ops.append(bi.op_lmhead(qbuf, s, wq, sw, None, self.argmax[:M]))
        prog = bi.new_program(len(ops), device=self.dev)
        bi.bi_program_build(ops, prog)
        return prog

    def launches_per_step(self, mode="calls"):
        if mode == "program":
            return 1
        return self.layers * 2 * len(self.groups) + 2

    def linear_bytes(self, M):
        """Algorithmic bytes of the step's linear launches: W + s_w + q + s_a + y."""
        tot = 0
        for l in range(self.layers):
            for nm, K in self.in_dims:
                N = self.W[l][nm][0].shape[0]
                tot += N * K + 4 * N + M * K + 4 * M + 2 * M * N
        return tot

    def step_bytes(self, M):
        """Algorithmic bytes of one step: every linear's W + s_w + q + s_a + y,
        every quantisation's x read and q + s_a written, the head's W + s_w +
        q + s_a and argmax."""
        tot = self.linear_bytes(M)
        for l in range(self.layers):
            for nm, K in self.in_dims:
                tot += 2 * M * K + M * K + 4 * M
        N, K = self.head[0].shape
        tot += 2 * M * K + M * K + 4 * M
        tot += N * K + 4 * N + M * K + 4 * M + 4 * M
        return tot

    def step(self, M, flags, linears_only=False):
        """Enqueue one verify pass on the current stream (or, with
        linears_only, just its linear launches back to back)."""
        bi, q, s = self.bi, self.q[:M], self.s[:M]
        for l in range(self.layers):
            for nm, K in self.in_dims:
                qbuf = self.q.view(-1)[:M * K].view(M, K)
                if not linears_only:
                    bi.bi_quantize_act(self.x[(l, nm)][:M, :K], qbuf, s, K=K, flags=flags)
                wq, sw = self.W[l][nm]
                bi.bi_linear_w8a8(qbuf, s, wq, sw, self.y[nm][:M], self.ws, flags=flags)
        if linears_only:
            return
        K = 4096
        qbuf = self.q.view(-1)[:M * K].view(M, K)
        bi.bi_quantize_act(self.x[("head",)][:M], qbuf, s, K=K, flags=flags)
        wq, sw = self.head
        bi.bi_lmhead_argmax(qbuf, s, wq, sw, None, self.argmax[:M], self.ws, flags=flags)


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


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
    t0 = time.time()
    st = Stack(bi, torch, args.layers, 16, dev)
    setup_s = time.time() - t0
    flags = bi.BI_FLAG_PDL
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    progs = {}
    prog_ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=dev)

    def enqueue_step(m):
        if args.mode == "program":
            if m not in progs:
                progs[m] = st.build_program(m)
            bi.bi_program_run(progs[m], m, prog_ws)
        else:
            st.step(m, flags)

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
        ms = e0.elapsed_time(e1) / steps
        if world > 1:
            t = torch.tensor([ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    g = graph_for(M)
    clocks = ClockSampler(local)
    ms = time_graph(g, args.steps, args.warmup)
    clk = clocks.stop(region["t0"], region["t1"])
    gbs = st.weight_bytes * world / (ms * 1e-3) / 1e9

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
            st.step(M, flags, linears_only=True)
        stream.synchronize()
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl, stream=stream):
            st.step(M, flags, linears_only=True)
        kernel_name = "skinny_kernel (bi_linear_w8a8, M<=16)"
        lin_launches = st.layers * len(st.groups)
        lin_ms = time_graph(gl, max(5, args.steps // 2), 3)
        achieved = st.linear_bytes(M) / (lin_ms * 1e-3) / 1e9
        note = ("achieved = algorithmic bytes (W + s_w + q + s_a + y) of the step's %d linear launches / "
                "their event-timed duration back to back in a CUDA graph" % lin_launches)

    # end to end: activations H2D from pinned memory, graph, argmax D2H
    host_x = {k: torch.from_numpy(v.view(np.int16)).pin_memory() for k, v in st.x_np.items()}
    host_am = torch.empty(16, dtype=torch.int32).pin_memory()
    h2d = sum(int(v[:M].numel()) * 2 for v in host_x.values())
    e2e_steps = max(3, args.steps // 2)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for k, v in host_x.items():
                st.x[k][:M].copy_(v[:M], non_blocking=True)
            g.replay()
            host_am[:M].copy_(st.argmax[:M], non_blocking=True)
        e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_gbs = st.weight_bytes * world / (e2e_ms * 1e-3) / 1e9

    peaks, kind = read_peaks()
    peak = float(peaks["hbm_gbs"])
    src = os.path.join(ROOT, "invariant_quantized_linear_gb300", "csrc",
                       "k_program.cu" if args.mode == "program" else "k_skinny.cu")
    traffic = None
    if NCU_TRAFFIC["source_sha256"] == source_sha(src):
        traffic = NCU_TRAFFIC["bytes_per_launch"]

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
                       "activations": "independent synthetic input per linear group (layers not chained)",
                       "packing": "q/k/v and gate/up weight rows packed: one call per group",
                       "launch": ("one verify-pass program launch per step (persistent cooperative kernel, "
                                  "grid barrier between ops), in a CUDA graph" if args.mode == "program" else
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
                    "d2h_bytes_per_step": 4 * M, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": st.launches_per_step(args.mode) * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "setup_s": round(setup_s, 1),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ CPU oracle

def oracle_sample():
    """A bounded sample of the workload for the CPU oracle: layer 0's q
    projection (4096 x 4096) at M = 8, weights quantised by the oracle."""
    import gen
    import oracle
    wl = gen.STACK36
    lin = gen.QWEN3_8B_LINEARS[0]
    w = gen.weight_f32(wl.seed, 0, lin.proj, lin.N, lin.K)
    wq, sw = oracle.requant_pow2(*oracle.quantize_weight(w))
    x = gen.activations(wl, 8, lin.K, stream=100)
    return oracle, x, wq, sw, lin


def cpu_baseline(bounded_s=12.0, M=8):
    oracle, x, wq, sw, lin = oracle_sample()
    t0 = time.time()
    n = 0
    while True:
        q, s = oracle.quantize_act(x[:M])
        oracle.linear_w8a8(q, s, wq, sw)
        n += 1
        if time.time() - t0 >= bounded_s:
            break
    dt = (time.time() - t0) / n
    return {"value": round((lin.N * lin.K + 4 * lin.N) / dt / 1e9, 3), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "q projection of layer 0 (4096x4096 int8, pow2 scales) at M=%d, activation "
                      "quantisation + linear, repeated %d times in %.1f s" % (M, n, time.time() - t0)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    oracle, x, wq, sw, lin = oracle_sample()
    M = args.m
    for _ in range(args.warmup):
        q, s = oracle.quantize_act(x[:M])
        oracle.linear_w8a8(q, s, wq, sw)
    t0 = time.time()
    for _ in range(args.steps):
        q, s = oracle.quantize_act(x[:M])
        oracle.linear_w8a8(q, s, wq, sw)
    dt = (time.time() - t0) / args.steps
    v = (lin.N * lin.K + 4 * lin.N) / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": M},
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "one step = layer 0's 4096x4096 q projection at M=%d on the CPU oracle" % M},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
