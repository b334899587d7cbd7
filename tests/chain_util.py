"""Chained verify-pass stacks for the GPU tests: the same seeded fp32 weights
quantised twice, on the device by the library and on the host by the oracle,
and the pass itself as one program or as one call per op."""
import numpy as np
import torch

import gen
import oracle
from tests.gpu_util import DEV, oracle_weights, to_dev, weights


class ChainStack:
    """Weights of `layers` chained layers plus an LM head of V rows."""

    def __init__(self, bi, H, QR, KV, I, V, layers, seed):
        self.bi = bi
        self.H, self.QR, self.KV, self.I, self.V = H, QR, KV, I, V
        lins = gen.chain_linears(H, QR, KV, I)
        self.gpu, self.ora = [], []
        for l in range(layers):
            g, o = {}, {}
            for name, _ in gen.CHAIN_GROUPS:
                w = gen.chain_group_f32(seed, l, name, lins)
                g[name] = weights(bi, w, pow2=True)
                o[name] = oracle_weights(oracle, w, pow2=True)
                del w
            self.gpu.append(g)
            self.ora.append(o)
        w = gen.weight_f32(seed, 0, gen.LMHEAD.proj, V, H)
        self.head_gpu = weights(bi, w, pow2=True)
        self.head_ora = oracle_weights(oracle, w, pow2=True)

    def oracle_pass(self, h0: np.ndarray, record=True):
        return oracle.verify_pass(h0, self.ora, self.head_ora, self.QR, record=record)

    def buffers(self, M):
        """Device buffers of one pass: the stream h, each linear's output and
        the codes/scales each linear reads."""
        t = torch
        b = {"h": t.empty((M, self.H), dtype=t.int16, device=DEV)}
        for name, N, K in (("qkv", self.QR + 2 * self.KV, self.H), ("o", self.H, self.QR),
                           ("gu", 2 * self.I, self.H), ("down", self.H, self.I)):
            b["y_" + name] = t.full((M, N), -1, dtype=t.int16, device=DEV)
            b["q_" + name] = t.empty((M, K), dtype=t.int8, device=DEV)
            b["s_" + name] = t.empty(M, dtype=t.float32, device=DEV)
        b["q_head"] = t.empty((M, self.H), dtype=t.int8, device=DEV)
        b["s_head"] = t.empty(M, dtype=t.float32, device=DEV)
        b["argmax"] = t.full((M,), -1, dtype=t.int32, device=DEV)
        return b

    def program_ops(self, b, upto=None):
        """Ops of the pass over all layers (or the first `upto`)."""
        bi = self.bi
        ops = []
        layers = self.gpu if upto is None else self.gpu[:upto]
        for l, W in enumerate(layers):
            if l == 0:
                ops.append(bi.op_quantize_act(b["h"], b["q_qkv"], b["s_qkv"]))
            ops.append(bi.op_linear(b["q_qkv"], b["s_qkv"], *W["qkv"], b["y_qkv"]))
            ops.append(bi.op_quantize_act(b["y_qkv"], b["q_o"], b["s_o"], K=self.QR))
            ops.append(bi.op_linear(b["q_o"], b["s_o"], *W["o"], b["y_o"]))
            ops.append(bi.op_residual_quant(b["h"], b["y_o"], b["q_gu"], b["s_gu"]))
            ops.append(bi.op_linear(b["q_gu"], b["s_gu"], *W["gu"], b["y_gu"]))
            ops.append(bi.op_relu_mul_quant(b["y_gu"], self.I, b["q_down"], b["s_down"]))
            ops.append(bi.op_linear(b["q_down"], b["s_down"], *W["down"], b["y_down"]))
            last = l == len(layers) - 1
            ops.append(bi.op_residual_quant(b["h"], b["y_down"], b["q_head"] if last else b["q_qkv"],
                                            b["s_head"] if last else b["s_qkv"]))
        ops.append(bi.op_lmhead(b["q_head"], b["s_head"], *self.head_gpu, None, b["argmax"]))
        return ops

    def run_program(self, b, h0_dev, M):
        bi = self.bi
        ops = self.program_ops(b)
        prog = bi.new_program(len(ops))
        bi.bi_program_build(ops, prog)
        ws = torch.zeros(bi.bi_program_workspace_size(), dtype=torch.uint8, device=DEV)
        b["h"].copy_(h0_dev)
        bi.bi_program_run(prog, M, ws)
        torch.cuda.synchronize()
        assert bi.bi_workspace_status(ws) == bi.BI_OK
        return prog, ws

    def run_calls(self, b, h0_dev, M, flags=0, record=None):
        """The same pass as one library call per op."""
        bi = self.bi
        ws = bi.new_workspace(M, max(self.V, 2 * self.I), max(self.H, self.I))
        b["h"].copy_(h0_dev)
        bi.bi_quantize_act(b["h"], b["q_qkv"], b["s_qkv"], flags=flags)
        for l, W in enumerate(self.gpu):
            bi.bi_linear_w8a8(b["q_qkv"], b["s_qkv"], *W["qkv"], b["y_qkv"], ws, flags=flags)
            bi.bi_quantize_act(b["y_qkv"], b["q_o"], b["s_o"], K=self.QR, flags=flags)
            bi.bi_linear_w8a8(b["q_o"], b["s_o"], *W["o"], b["y_o"], ws, flags=flags)
            bi.bi_residual_quantize(b["h"], b["y_o"], b["q_gu"], b["s_gu"], flags=flags)
            if record is not None:
                record.append({"h_mid": b["h"].clone()})
            bi.bi_linear_w8a8(b["q_gu"], b["s_gu"], *W["gu"], b["y_gu"], ws, flags=flags)
            bi.bi_relu_mul_quantize(b["y_gu"], self.I, b["q_down"], b["s_down"], flags=flags)
            bi.bi_linear_w8a8(b["q_down"], b["s_down"], *W["down"], b["y_down"], ws, flags=flags)
            bi.bi_residual_quantize(b["h"], b["y_down"], b["q_qkv"], b["s_qkv"], flags=flags)
            if record is not None:
                record[-1].update({k: b["y_" + k].clone() for k in ("qkv", "o", "gu", "down")})
                record[-1]["h"] = b["h"].clone()
        am = torch.empty(M, dtype=torch.int32, device=DEV)
        bi.bi_lmhead_argmax(b["q_qkv"], b["s_qkv"], *self.head_gpu, None, am, ws, flags=flags)
        torch.cuda.synchronize()
        return am
