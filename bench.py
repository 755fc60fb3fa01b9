#!/usr/bin/env python3
"""Benchmark of the unified-precision FP8 linear layer on GB300.

One step = one pass of the whole hot path over one training layer of the
8B-shaped model (7 linears q,k,v,o,gate,up,down at M = 8192 tokens; or the
32B-shaped layer at M = 16384 with --workload train32b):

  weight sync   128x128 quantization of the 7 BF16 master weights
  forward       1x128 quantization of the 4 distinct inputs (the attention
                and MLP inputs through the fused RMSNorm quantizer), 7
                forward GEMMs
  backward      both forms (1x128 and 128x1) of the 7 output gradients from
                one read each, 7 DGrad GEMMs, 128x1 re-quantization of the 4
                inputs, 7 WGrad GEMMs
  metric        token-mult-prob-error over the step's M tokens

Other workloads (--workload): rollout (the 7 forward products at --tokens
M), sync (the weight-sync quantizations of 32 layers), metric (the plain,
masked and per-sequence mismatch metric over 4M tokens), moe and moe_train
(the expert linears of a Qwen3-30B-A3B-shaped MoE layer, forward or a whole
training step), kvcache (FP8 KV-cache recalibration and writes of one
layer).

Inputs are synthetic (seeded, resident in HBM before timing); every
workload's working set is larger than the 129 MB L2 or L2 is flushed between
calls (the `l2` key of `config` says which).

Printed JSON (rank 0): value = the step's GEMM FLOPs (or algorithmic bytes)
/ step time, everything in the step included; per-kernel-family rates from
CUDA events around graph replays of each family; a roofline for the family
with the largest share, with its measured DRAM traffic where an ncu capture
of the current sources exists; the end-to-end rate through the same C-ABI
calls with the step's inputs copied in from pinned host buffers and its
result copied out every step; the SM clocks sampled during the timed
region; the CPU oracle timed on a bounded sample on the host cores.

--impl reference times that CPU oracle as the reference arm (a bounded
sample of the same workload per step, see CpuSample).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 linear fwd+dgrad+wgrad TFLOP/s & % FP8 peak; quantize GB/s & % HBM"
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor ratio (4.5 / 2.25 PFLOP/s)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# Algorithmic bytes per element / token (what the method must move).
BYTES_PER_ELEM = {
    "quant_act_1x128": 2 + 1 + 4 / 128,          # BF16 in, code out, one scale per 128
    "quant_w_128x128": 2 + 1 + 4 / (128 * 128),
    "requant_128x1": 1 + 1 + 4 / 128 + 4 / 128,  # code in/out, row scales in, col scales out
    # BF16 in, 1x128 codes + scales out, 128x1 codes + scales out
    "quant_dual_1x128_128x1": 2 + 1 + 1 + 4 / 128 + 4 / 128,
    "token_mult_prob_error": 8,                  # two FP32 per token
    "token_mismatch_masked": 4 + 4 + 1 + 4,      # two FP32 and the mask in, the weight out
    "swiglu_quant_1x128": 2 + 2 + 1 + 4 / 128,   # gate and up BF16 in, code + scale out
    "rmsnorm_quant_1x128": 2 + 1 + 4 / 128,      # BF16 in, code + scale out (gain: K values per call)
}
# RMSNorm epsilon of the two model families (Llama-3.1-8B: 1e-5; the 32B-class
# dense model: 1e-6)
RMS_EPS = {"train8b": 1e-5, "train32b": 1e-6}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device) -> float:
    """Maximum of a per-rank value over all ranks (the job's time is the slowest
    rank's); identity for one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, amount_per_rank: float, ms_per_step_max: float, scale: float) -> float:
    """Whole-job throughput of N replicas: every rank does `amount_per_rank`
    per step; the step takes the slowest rank's time."""
    return world * amount_per_rank / (ms_per_step_max * 1e-3) / scale


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self

        def read():
            for l in self.proc.stdout:
                if l.strip():
                    self.lines.append(l)
        self.reader = threading.Thread(target=read, daemon=True)
        self.reader.start()
        return self

    def wait_first(self, timeout: float = 5.0):
        """Block until the sampler has produced a line (it takes a moment to
        start), so that samples cover the region that follows."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout:
            time.sleep(0.01)

    def count(self):
        return len(self.lines)

    def mark(self):
        """Only samples taken from now on enter the summary."""
        self.start = len(self.lines)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines[getattr(self, "start", 0):]:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the GPU step
# --------------------------------------------------------------------------

class LayerStep:
    """Preallocated buffers and the ordered C-ABI calls of one layer step."""

    def __init__(self, kind: str, device, seed: int = 0):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet = jet
        self.kind = kind
        self.cases = wl.training_layer(kind, seed=seed, device=device)
        self.M = self.cases[0].M
        M = self.M
        dev = device
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        # distinct inputs; the attention and MLP inputs come out of an RMSNorm
        # (its gain drawn per norm), the other two are plain activations
        self.inputs = {}
        self.eps = RMS_EPS[kind]
        for c in self.cases:
            key = wl.SHARED_INPUT[c.name]
            if key not in self.inputs:
                norm = key in ("attn_in", "mlp_in")
                g = (wl.norm_gain(c.K, seed=seed, config=wl.CONFIG_ID[kind],
                                  tensor_id=600 + len(self.inputs), device=dev) if norm else None)
                self.inputs[key] = {"x": c.x, "K": c.K, "g": g,
                                    "q": e((M, c.K), u8), "s": e((c.K // 128, M), f32),
                                    "qT": e((c.K, M), u8), "sT": e((M // 128, c.K), f32)}
            c.key = key
        self.lin = []
        for c in self.cases:
            N, K = c.N, c.K
            self.lin.append({
                "case": c, "w": c.w, "dy": c.dy,
                "qw": e((N, K), u8), "sw": e((N // 128, K // 128), f32),
                "y": e((M, N), bf),
                "qdy": e((M, N), u8), "sdy": e((N // 128, M), f32),
                "dx": e((M, K), bf),
                "qdyT": e((N, M), u8), "sdyT": e((M // 128, N), f32),
                "dw": e((N, K), bf),
            })
        self.logp_train, self.logp_rollout = (t.to(dev) for t in wl.logprobs(M, seed=seed))
        self.metric_out = e((1,), f32)
        nb = max(jet.workspace_bytes("token_mult_prob_error", M), 16)
        self.metric_ws = e((nb,), u8)
        self.flops = sum(3 * 2 * M * c.N * c.K for c in self.cases)
        # algorithmic work per kernel family per step
        self.work = {"gemm_fp8_fwd": sum(2 * M * c.N * c.K for c in self.cases),
                     "gemm_fp8_dgrad": sum(2 * M * c.N * c.K for c in self.cases),
                     "gemm_fp8_wgrad": sum(2 * M * c.N * c.K for c in self.cases),
                     "quant_w_128x128": sum(c.N * c.K for c in self.cases) * BYTES_PER_ELEM["quant_w_128x128"],
                     "quant_act_1x128": sum(M * v["K"] for v in self.inputs.values() if v["g"] is None)
                                        * BYTES_PER_ELEM["quant_act_1x128"],
                     "rmsnorm_quant_1x128": sum(M * v["K"] * BYTES_PER_ELEM["rmsnorm_quant_1x128"]
                                                + 2 * v["K"] for v in self.inputs.values()
                                                if v["g"] is not None),
                     "requant_128x1": sum(M * v["K"] for v in self.inputs.values())
                                      * BYTES_PER_ELEM["requant_128x1"],
                     "quant_dual_1x128_128x1": sum(M * c.N for c in self.cases)
                                               * BYTES_PER_ELEM["quant_dual_1x128_128x1"],
                     "token_mult_prob_error": M * BYTES_PER_ELEM["token_mult_prob_error"]}
        # per linear: weight quant, fwd, dY's fused 1x128 + 128x1 quantization,
        # dgrad, wgrad; per distinct input: quant (forward), requant (backward,
        # from the saved FP8 form); the metric: two passes
        self.launches_per_step = len(self.lin) * 5 + len(self.inputs) * 2 + 2
        self.primary = ("TFLOP/s", self.flops)
        self.config = {"workload": f"{kind}_layer_M{M}", "tokens": M,
                       "linears": [(c.name, c.N, c.K) for c in self.cases],
                       "gemm_tflop_per_step": round(self.flops / 1e12, 4),
                       "l2": "no flush: per-step working set > 129 MB L2"}

    def calls(self):
        """The step as (family, thunk, shape label) in launch order."""
        j = self.jet
        out = []
        for L in self.lin:
            out.append(("quant_w_128x128", lambda L=L: j.jet_quant_w_128x128(L["w"], L["qw"], L["sw"]),
                        L["case"].name))
        for key, v in self.inputs.items():
            if v["g"] is not None:
                out.append(("rmsnorm_quant_1x128", lambda v=v: j.jet_rmsnorm_quant_1x128(
                    v["x"], v["g"], self.eps, v["q"], v["s"]), key))
            else:
                out.append(("quant_act_1x128", lambda v=v: j.jet_quant_act_1x128(v["x"], v["q"], v["s"]),
                            key))
        for L in self.lin:
            v = self.inputs[L["case"].key]
            out.append(("gemm_fp8_fwd", lambda L=L, v=v: j.jet_gemm_fp8_fwd(v["q"], v["s"], L["qw"], L["sw"], L["y"]),
                        L["case"].name))
        for L in self.lin:
            out.append(("quant_dual_1x128_128x1", lambda L=L: j.jet_quant_dual_1x128_128x1(
                L["dy"], L["qdy"], L["sdy"], L["qdyT"], L["sdyT"]), "dy_" + L["case"].name))
            out.append(("gemm_fp8_dgrad", lambda L=L: j.jet_gemm_fp8_dgrad(L["qdy"], L["sdy"], L["qw"], L["sw"], L["dx"]),
                        L["case"].name))
        for v in self.inputs.values():
            out.append(("requant_128x1", lambda v=v: j.jet_requant_128x1(v["q"], v["s"], v["qT"], v["sT"]),
                        "x%d" % v["K"]))
        for L in self.lin:
            v = self.inputs[L["case"].key]
            out.append(("gemm_fp8_wgrad", lambda L=L, v=v: j.jet_gemm_fp8_wgrad(L["qdyT"], L["sdyT"], v["qT"], v["sT"], L["dw"]),
                        L["case"].name))
        out.append(("token_mult_prob_error", lambda: j.jet_token_mult_prob_error(
            self.logp_train, self.logp_rollout, self.metric_out, self.metric_ws), "n%d" % self.M))
        return out

    def host_io(self, outputs=False):
        """Pinned host copies of the step's inputs (X, the BF16 master weights,
        dY and both log-probability vectors) and a buffer for its result, the
        mismatch metric; Y, dX and dW stay on the device, where the next
        layer, the previous layer and the optimizer read them, unless
        `outputs` (then they are copied back too)."""
        import torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        if not hasattr(self, "h_in"):
            self.h_in = [(pin(v["x"]), v["x"]) for v in self.inputs.values()]
            self.h_in += [(pin(L["w"]), L["w"]) for L in self.lin]
            self.h_in += [(pin(L["dy"]), L["dy"]) for L in self.lin]
            self.h_in += [(pin(self.logp_train), self.logp_train),
                          (pin(self.logp_rollout), self.logp_rollout)]
        outs = [self.metric_out]
        if outputs:
            outs += [L[k] for L in self.lin for k in ("y", "dx", "dw")]
        self.h_out = [(torch.empty(t.shape, dtype=t.dtype, pin_memory=True), t) for t in outs]
        nbytes = lambda pairs: sum(h.numel() * h.element_size() for h, _ in pairs)
        return nbytes(self.h_in), nbytes(self.h_out)


def fork_calls(streams, fns):
    """One call that runs independent thunks on their own streams, forked from
    and joined back into the current stream (captured as such in a graph)."""
    import torch

    def run():
        cur = torch.cuda.current_stream()
        for st, f in zip(streams, fns):
            st.wait_stream(cur)
            with torch.cuda.stream(st):
                f()
        for st in streams[:len(fns)]:
            cur.wait_stream(st)
    return run


class RolloutStep:
    """Forward only (rollout): the 4 distinct inputs quantized 1x128 (the
    attention and MLP inputs through the fused RMSNorm quantizer) and the 7
    forward GEMMs of the 8B layer at M tokens; the weights are quantized once
    beforehand (per weight sync) and not timed.  The products of one input
    (q, k, v; gate, up) are independent and run on their own streams, forked
    from and joined back into the step's stream, as an inference engine
    issues them: at decode sizes each product's launch, pipeline fill and
    split reduction then overlap the others' weight streams."""

    def __init__(self, M: int, device, seed: int = 0):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet, self.M = jet, M
        self.cases = wl.training_layer("train8b", seed=seed, device=device, M=M, with_grad=False)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.inputs, self.lin = {}, []
        self.eps = RMS_EPS["train8b"]
        for c in self.cases:
            key = wl.SHARED_INPUT[c.name]
            if key not in self.inputs:
                norm = key in ("attn_in", "mlp_in")
                g = (wl.norm_gain(c.K, seed=seed, config=wl.CONFIG_ID["rollout"],
                                  tensor_id=600 + len(self.inputs), device=device) if norm else None)
                self.inputs[key] = {"x": c.x, "K": c.K, "g": g, "q": e((M, c.K), torch.uint8),
                                    "s": e((c.K // 128, M), torch.float32)}
            c.key = key
            qw, sw = jet.quant_w_128x128(c.w)
            # split-contraction partials (M <= 128), allocated once, outside the timing
            nws = jet.workspace_bytes("gemm_fp8_fwd", M, c.N, c.K)
            self.lin.append({"case": c, "qw": qw, "sw": sw,
                             "y": e((M, c.N), torch.bfloat16),
                             "ws": e((nws,), torch.uint8) if nws else None})
        torch.cuda.synchronize()
        self.streams = [torch.cuda.Stream(device=device) for _ in range(3)]
        self.flops = sum(2 * M * c.N * c.K for c in self.cases)
        gemm_bytes = sum(M * c.K + c.N * c.K + 4 * (M * c.K // 128 + c.N * c.K // 16384)
                         + 2 * M * c.N for c in self.cases)
        self.work = {"gemm_fp8_fwd": self.flops, "gemm_fp8_fwd_bytes": gemm_bytes,
                     "quant_act_1x128": sum(M * v["K"] for v in self.inputs.values() if v["g"] is None)
                     * BYTES_PER_ELEM["quant_act_1x128"],
                     "rmsnorm_quant_1x128": sum(M * v["K"] * BYTES_PER_ELEM["rmsnorm_quant_1x128"]
                                                + 2 * v["K"] for v in self.inputs.values()
                                                if v["g"] is not None)}
        # a split GEMM is two launches: the partial tiles and their reduction
        self.launches_per_step = (len(self.lin) + len(self.inputs)
                                  + sum(L["ws"] is not None for L in self.lin))
        self.primary = ("TFLOP/s", self.flops)
        self.config = {"workload": f"rollout8b_M{M}", "tokens": M,
                       "linears": [(c.name, c.N, c.K) for c in self.cases],
                       "gemm_tflop_per_step": round(self.flops / 1e12, 6),
                       "concurrency": "q, k, v on three streams and gate, up on two",
                       "l2": "weights (218 M codes) > 129 MB L2; activations may stay in L2"}

    def calls(self):
        j, out = self.jet, []
        for key, v in self.inputs.items():
            if v["g"] is not None:
                out.append(("rmsnorm_quant_1x128", lambda v=v: j.jet_rmsnorm_quant_1x128(
                    v["x"], v["g"], self.eps, v["q"], v["s"]), key))
            else:
                out.append(("quant_act_1x128", lambda v=v: j.jet_quant_act_1x128(v["x"], v["q"], v["s"]),
                            key))
        # one call per input: its products forked onto the side streams
        groups = {}
        for L in self.lin:
            groups.setdefault(L["case"].key, []).append(L)
        for key, lins in groups.items():
            v = self.inputs[key]
            fns = [lambda L=L, v=v: j.jet_gemm_fp8_fwd(v["q"], v["s"], L["qw"], L["sw"], L["y"],
                                                      ws=L["ws"]) for L in lins]
            name = "+".join(L["case"].name for L in lins)
            out.append(("gemm_fp8_fwd", fns[0] if len(fns) == 1 else fork_calls(self.streams, fns),
                        name))
        return out

    def host_io(self):
        import torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        self.h_in = [(pin(v["x"]), v["x"]) for v in self.inputs.values()]
        self.h_out = [(torch.empty(L["y"].shape, dtype=L["y"].dtype, pin_memory=True), L["y"])
                      for L in self.lin]
        nbytes = lambda pairs: sum(h.numel() * h.element_size() for h, _ in pairs)
        return nbytes(self.h_in), nbytes(self.h_out)


class SyncStep:
    """Weight sync: 128x128 quantization of 32 layers of the 8B layer's 7
    weights (6.98e9 parameters) and 1x128 quantization of a 16384 x 14336
    Student-t(3) activation matrix."""

    LAYERS = 32

    def __init__(self, device, seed: int = 0):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet, self.M = jet, 16384
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.w = []
        for layer in range(self.LAYERS):
            for i, (name, N, K) in enumerate(wl.LLAMA8B_LINEARS):
                w = wl.weights(N, K, seed=seed, config=5, tensor_id=1000 + 10 * layer + i,
                               device=device)
                self.w.append({"name": f"L{layer}.{name}", "w": w,
                               "q": e((N, K), torch.uint8),
                               "s": e((N // 128, K // 128), torch.float32)})
        self.x = wl.heavy_activations(16384, 14336, seed=seed, device=device)
        self.xq = e((16384, 14336), torch.uint8)
        self.xs = e((14336 // 128, 16384), torch.float32)
        params = sum(t["w"].numel() for t in self.w)
        self.work = {"quant_w_128x128": params * BYTES_PER_ELEM["quant_w_128x128"],
                     "quant_act_1x128": self.x.numel() * BYTES_PER_ELEM["quant_act_1x128"]}
        self.bytes = sum(self.work.values())
        self.flops = 0
        self.launches_per_step = len(self.w) + 1
        self.streams = [torch.cuda.Stream(device=device) for _ in range(3)]
        self.primary = ("GB/s", self.bytes)
        self.config = {"workload": "sync8b_32layers", "parameters": params,
                       "concurrency": "weights three at a time on their own streams",
                       "activation": [16384, 14336],
                       "l2": "no flush: 21 GB of weights and codes per step"}

    def calls(self):
        # the weights are independent: three at a time on their own streams
        j = self.jet
        out = []
        for i in range(0, len(self.w), len(self.streams)):
            ts = self.w[i:i + len(self.streams)]
            fns = [lambda t=t: j.jet_quant_w_128x128(t["w"], t["q"], t["s"]) for t in ts]
            out.append(("quant_w_128x128", fork_calls(self.streams, fns),
                        "+".join(t["name"] for t in ts)))
        out.append(("quant_act_1x128", lambda: j.jet_quant_act_1x128(self.x, self.xq, self.xs),
                    "x16384x14336"))
        return out


class MoeStep:
    """Forward of the expert linears of one Qwen3-30B-A3B-shaped MoE layer
    (4096 tokens, top-8 of 128 experts, 32768 routed rows): 1x128
    quantization of the routed gate_up input, the grouped gate_up product
    (N = 1536, K = 2048 per expert), SwiGLU of its two halves fused with the
    1x128 quantization of the result, the grouped down product (N = 2048,
    K = 768).  The routing (row offsets per expert) and the experts' FP8
    weights are prepared beforehand and not timed."""

    def __init__(self, device, seed: int = 0):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet = jet
        off, lins = wl.moe_layer(seed=seed, device=device)
        self.off = off
        self.M = M = int(off[-1].item())
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.lin = []
        flops = nbytes = 0
        counts = (off[1:] - off[:-1]).cpu()
        used = int((counts > 0).sum())
        for name, x, w in lins:
            E, N, K = w.shape
            qw = e((E, N, K), torch.uint8)
            sw = e((E, N // 128, K // 128), torch.float32)
            for i in range(E):
                jet.jet_quant_w_128x128(w[i], qw[i], sw[i])
            self.lin.append({"name": name, "x": x, "K": K, "N": N, "qw": qw, "sw": sw,
                             "q": e((M, K), torch.uint8), "s": e((K // 128, M), torch.float32),
                             "y": e((M, N), torch.bfloat16)})
            flops += 2 * M * N * K
            nbytes += M * K + 4 * M * K // 128 + used * (N * K + 4 * N * K // 16384) + 2 * M * N
        gu, dn = self.lin
        assert gu["N"] == 2 * dn["K"]
        self.F = F = dn["K"]
        self.lin[1]["x"] = None   # the down input is the SwiGLU of the gate_up output
        torch.cuda.synchronize()
        self.flops = flops
        self.work = {"gemm_fp8_fwd_grouped": flops, "gemm_fp8_fwd_grouped_bytes": nbytes,
                     "quant_act_1x128": M * gu["K"] * BYTES_PER_ELEM["quant_act_1x128"],
                     "swiglu_quant_1x128": M * F * BYTES_PER_ELEM["swiglu_quant_1x128"]}
        self.launches_per_step = 4
        self.primary = ("TFLOP/s", flops)
        tiles = int(((counts + 127) // 128).sum())
        self.config = {"workload": f"moe_qwen3_30b_a3b_T{wl.MOE_TOKENS}",
                       "tokens": wl.MOE_TOKENS, "experts": wl.MOE_EXPERTS, "topk": wl.MOE_TOPK,
                       "routed_rows": M, "linears": [(L["name"], L["N"], L["K"]) for L in self.lin],
                       "rows_per_expert": [int(counts.min()), int(counts.max())],
                       "row_tiles": tiles, "dense_row_tiles": (M + 127) // 128,
                       "gemm_tflop_per_step": round(flops / 1e12, 4),
                       "l2": "no flush: per-step working set (~0.9 GB) > 129 MB L2"}

    def calls(self):
        j = self.jet
        gu, dn, F = self.lin[0], self.lin[1], self.F
        return [
            ("quant_act_1x128", lambda: j.jet_quant_act_1x128(gu["x"], gu["q"], gu["s"]), "x_gate_up"),
            ("gemm_fp8_fwd_grouped", lambda: j.jet_gemm_fp8_fwd_grouped(
                gu["q"], gu["s"], gu["qw"], gu["sw"], self.off, gu["y"]), "gate_up"),
            ("swiglu_quant_1x128", lambda: j.jet_swiglu_quant_1x128(
                gu["y"][:, :F], gu["y"][:, F:], dn["q"], dn["s"]), "h"),
            ("gemm_fp8_fwd_grouped", lambda: j.jet_gemm_fp8_fwd_grouped(
                dn["q"], dn["s"], dn["qw"], dn["sw"], self.off, dn["y"]), "down"),
        ]

    def host_io(self):
        import torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        gu, dn = self.lin
        self.h_in = [(pin(gu["x"]), gu["x"]), (pin(self.off), self.off)]
        self.h_out = [(torch.empty(dn["y"].shape, dtype=dn["y"].dtype, pin_memory=True), dn["y"])]
        nbytes = lambda pairs: sum(h.numel() * h.element_size() for h, _ in pairs)
        return nbytes(self.h_in), nbytes(self.h_out)


class MoeTrainStep:
    """One training step of the expert linears of the Qwen3-30B-A3B-shaped MoE
    layer (4096 tokens, top-8 of 128 experts), in the padded layout that the
    expert WGrad needs (each expert's rows padded with zero rows to whole
    128-token groups: 41984 rows for 32768 routed ones):
      weight sync   128x128 quantization of both stacked expert weights
      forward       1x128 quantization of X, grouped gate_up, SwiGLU fused
                    with the 1x128 quantization, grouped down
      backward      both forms of dY_down, grouped DGrad and WGrad of down
                    (the SwiGLU output re-quantized 128x1); both forms of
                    dY_gate_up, grouped DGrad and WGrad of gate_up (X
                    re-quantized 128x1)
    dY_gate_up stands for the SwiGLU backward's output (not on this path) and
    is a synthetic input, like dY_down.  `value` counts the FLOPs of the
    routed rows only (padding rows are work the layout costs)."""

    def __init__(self, device, seed: int = 0):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet = jet
        off, lins = wl.moe_layer(seed=seed, device="cpu")
        pad = wl.moe_pad_offsets(off)
        M, Mp = int(off[-1]), int(pad[-1])
        self.M = M
        (_, x_gu, w_gu), (_, _, w_dn) = lins
        E, Ng, Kg = w_gu.shape
        _, Nd, Kd = w_dn.shape
        assert Ng == 2 * Kd
        self.F = F = Kd
        cfg = wl.CONFIG_ID["moe"]
        sc = lambda t: wl.moe_scatter_padded(t, off, pad).to(device)
        self.x = sc(x_gu)
        self.dy_dn = sc(wl.grad_output(M, Nd, seed=seed, config=cfg, tensor_id=210))
        self.dy_gu = sc(wl.grad_output(M, Ng, seed=seed, config=cfg, tensor_id=211))
        self.w_gu, self.w_dn = w_gu.to(device), w_dn.to(device)
        self.pad = pad.to(device)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        b = self.buf = {
            "qw_gu": e((E, Ng, Kg), u8), "sw_gu": e((E, Ng // 128, Kg // 128), f32),
            "qw_dn": e((E, Nd, Kd), u8), "sw_dn": e((E, Nd // 128, Kd // 128), f32),
            "qx": e((Mp, Kg), u8), "sx": e((Kg // 128, Mp), f32),
            "qxT": e((Kg, Mp), u8), "sxT": e((Mp // 128, Kg), f32),
            "y_gu": e((Mp, Ng), bf), "qh": e((Mp, F), u8), "sh": e((F // 128, Mp), f32),
            "qhT": e((F, Mp), u8), "shT": e((Mp // 128, F), f32), "y_dn": e((Mp, Nd), bf),
            "qdd": e((Mp, Nd), u8), "sdd": e((Nd // 128, Mp), f32),
            "qddT": e((Nd, Mp), u8), "sddT": e((Mp // 128, Nd), f32),
            "qdg": e((Mp, Ng), u8), "sdg": e((Ng // 128, Mp), f32),
            "qdgT": e((Ng, Mp), u8), "sdgT": e((Mp // 128, Ng), f32),
            "dh": e((Mp, F), bf), "dx": e((Mp, Kg), bf),
            "dw_dn": e((E, Nd, Kd), bf), "dw_gu": e((E, Ng, Kg), bf)}
        torch.cuda.synchronize()
        counts = (off[1:] - off[:-1])
        used = int((counts > 0).sum())
        fl_gu, fl_dn = 2 * M * Ng * Kg, 2 * M * Nd * Kd
        self.flops = 3 * (fl_gu + fl_dn)
        wbytes = lambda n, k: used * (n * k + 4 * n * k // 16384)
        act = lambda rows, k: rows * k + 4 * rows * k // 128
        self.work = {
            "quant_w_128x128": E * (Ng * Kg + Nd * Kd) * BYTES_PER_ELEM["quant_w_128x128"],
            "quant_act_1x128": Mp * Kg * BYTES_PER_ELEM["quant_act_1x128"],
            "swiglu_quant_1x128": Mp * F * BYTES_PER_ELEM["swiglu_quant_1x128"],
            "quant_dual_1x128_128x1": Mp * (Nd + Ng) * BYTES_PER_ELEM["quant_dual_1x128_128x1"],
            "requant_128x1": Mp * (F + Kg) * BYTES_PER_ELEM["requant_128x1"],
            "gemm_fp8_fwd_grouped": fl_gu + fl_dn,
            "gemm_fp8_fwd_grouped_bytes": act(Mp, Kg) + wbytes(Ng, Kg) + 2 * Mp * Ng
                                          + act(Mp, F) + wbytes(Nd, Kd) + 2 * Mp * Nd,
            "gemm_fp8_dgrad_grouped": fl_gu + fl_dn,
            "gemm_fp8_dgrad_grouped_bytes": act(Mp, Nd) + wbytes(Nd, Kd) + 2 * Mp * Kd
                                            + act(Mp, Ng) + wbytes(Ng, Kg) + 2 * Mp * Kg,
            "gemm_fp8_wgrad_grouped": fl_gu + fl_dn,
            "gemm_fp8_wgrad_grouped_bytes": act(Mp, Nd) + act(Mp, Kd) + 2 * E * Nd * Kd
                                            + act(Mp, Ng) + act(Mp, Kg) + 2 * E * Ng * Kg}
        self.launches_per_step = 14
        self.primary = ("TFLOP/s", self.flops)
        self.config = {"workload": f"moe_train_qwen3_30b_a3b_T{wl.MOE_TOKENS}",
                       "tokens": wl.MOE_TOKENS, "experts": E, "topk": wl.MOE_TOPK,
                       "routed_rows": M, "padded_rows": Mp,
                       "linears": [("gate_up", Ng, Kg), ("down", Nd, Kd)],
                       "gemm_tflop_per_step": round(self.flops / 1e12, 4),
                       "l2": "no flush: per-step working set (~2 GB) > 129 MB L2"}

    def calls(self):
        j, b, F = self.jet, self.buf, self.F
        E, Ng, Kg = self.w_gu.shape
        _, Nd, Kd = self.w_dn.shape
        return [
            ("quant_w_128x128", lambda: j.jet_quant_w_128x128(
                self.w_gu.view(E * Ng, Kg), b["qw_gu"].view(E * Ng, Kg),
                b["sw_gu"].view(E * Ng // 128, Kg // 128)), "w_gate_up"),
            ("quant_w_128x128", lambda: j.jet_quant_w_128x128(
                self.w_dn.view(E * Nd, Kd), b["qw_dn"].view(E * Nd, Kd),
                b["sw_dn"].view(E * Nd // 128, Kd // 128)), "w_down"),
            ("quant_act_1x128", lambda: j.jet_quant_act_1x128(self.x, b["qx"], b["sx"]), "x"),
            ("gemm_fp8_fwd_grouped", lambda: j.jet_gemm_fp8_fwd_grouped(
                b["qx"], b["sx"], b["qw_gu"], b["sw_gu"], self.pad, b["y_gu"]), "gate_up"),
            ("swiglu_quant_1x128", lambda: j.jet_swiglu_quant_1x128(
                b["y_gu"][:, :F], b["y_gu"][:, F:], b["qh"], b["sh"]), "h"),
            ("gemm_fp8_fwd_grouped", lambda: j.jet_gemm_fp8_fwd_grouped(
                b["qh"], b["sh"], b["qw_dn"], b["sw_dn"], self.pad, b["y_dn"]), "down"),
            ("quant_dual_1x128_128x1", lambda: j.jet_quant_dual_1x128_128x1(
                self.dy_dn, b["qdd"], b["sdd"], b["qddT"], b["sddT"]), "dy_down"),
            ("gemm_fp8_dgrad_grouped", lambda: j.jet_gemm_fp8_dgrad_grouped(
                b["qdd"], b["sdd"], b["qw_dn"], b["sw_dn"], self.pad, b["dh"]), "down"),
            ("requant_128x1", lambda: j.jet_requant_128x1(b["qh"], b["sh"], b["qhT"], b["shT"]), "h"),
            ("gemm_fp8_wgrad_grouped", lambda: j.jet_gemm_fp8_wgrad_grouped(
                b["qddT"], b["sddT"], b["qhT"], b["shT"], self.pad, b["dw_dn"]), "down"),
            ("quant_dual_1x128_128x1", lambda: j.jet_quant_dual_1x128_128x1(
                self.dy_gu, b["qdg"], b["sdg"], b["qdgT"], b["sdgT"]), "dy_gate_up"),
            ("gemm_fp8_dgrad_grouped", lambda: j.jet_gemm_fp8_dgrad_grouped(
                b["qdg"], b["sdg"], b["qw_gu"], b["sw_gu"], self.pad, b["dx"]), "gate_up"),
            ("requant_128x1", lambda: j.jet_requant_128x1(b["qx"], b["sx"], b["qxT"], b["sxT"]), "x"),
            ("gemm_fp8_wgrad_grouped", lambda: j.jet_gemm_fp8_wgrad_grouped(
                b["qdgT"], b["sdgT"], b["qxT"], b["sxT"], self.pad, b["dw_gu"]), "gate_up"),
        ]

    def host_io(self):
        import torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        ins = [self.x, self.dy_dn, self.dy_gu, self.w_gu, self.w_dn, self.pad]
        self.h_in = [(pin(t), t) for t in ins]
        outs = [self.buf[k] for k in ("y_dn", "dx", "dw_gu", "dw_dn")]
        self.h_out = [(torch.empty(t.shape, dtype=t.dtype, pin_memory=True), t) for t in outs]
        nbytes = lambda pairs: sum(h.numel() * h.element_size() for h, _ in pairs)
        return nbytes(self.h_in), nbytes(self.h_out)


class KvCacheStep:
    """FP8 KV cache of one layer of the 8B model (8 KV heads x 128 channels)
    after a model update: recalibrate the K and V scales on a 65536-token
    prefill, then write its keys and values into a 131072-slot cache at
    scattered slots."""

    def __init__(self, device, seed: int = 0, T: int = 65536, H: int = 8, D: int = 128):
        import torch
        import fp8_block_quantized_gb300 as jet

        self.jet, self.M = jet, T
        g = torch.Generator(device="cpu").manual_seed(seed + 7000)
        mk = lambda: (torch.randn((T, H, D), generator=g)
                      * torch.exp2(torch.rand((1, H, 1), generator=g) * 6 - 3)).to(torch.bfloat16)
        self.k, self.v = mk().to(device), mk().to(device)
        S = 2 * T
        self.slots = torch.randperm(S, generator=g)[:T].to(device)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.sk, self.sv = e((H,), torch.float32), e((H,), torch.float32)
        self.ck, self.cv = e((S, H, D), torch.uint8), e((S, H, D), torch.uint8)
        n = T * H * D
        self.work = {"kv_calibrate": 2 * n * 2.0, "kv_cache_write": 2 * (n * 3.0 + 8 * T)}
        self.bytes = sum(self.work.values())
        self.flops = 0
        self.launches_per_step = 6   # a calibration is two kernels
        self.primary = ("GB/s", self.bytes)
        self.streams = [torch.cuda.Stream(device=device) for _ in range(2)]
        self.config = {"workload": f"kvcache8b_T{T}", "tokens": T, "kv_heads": H, "head_dim": D,
                       "cache_slots": S, "concurrency": "K and V on two streams",
                       "l2": "no flush: 268 MB of K/V read per step > 129 MB L2"}

    def calls(self):
        j = self.jet
        cal = [lambda: j.jet_kv_calibrate(self.k, self.sk), lambda: j.jet_kv_calibrate(self.v, self.sv)]
        wr = [lambda: j.jet_kv_cache_write(self.k, self.sk, self.slots, self.ck),
              lambda: j.jet_kv_cache_write(self.v, self.sv, self.slots, self.cv)]
        return [("kv_calibrate", fork_calls(self.streams, cal), "k+v"),
                ("kv_cache_write", fork_calls(self.streams, wr), "k+v")]

    def host_io(self):
        import torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        self.h_in = [(pin(t), t) for t in (self.k, self.v, self.slots)]
        self.h_out = [(torch.empty(t.shape, dtype=t.dtype, pin_memory=True), t)
                      for t in (self.sk, self.sv, self.ck, self.cv)]
        nbytes = lambda pairs: sum(h.numel() * h.element_size() for h, _ in pairs)
        return nbytes(self.h_in), nbytes(self.h_out)


class MetricStep:
    """token-mult-prob-error over n = 4,194,304 tokens, the masked variant
    with per-token importance weights (75% of the tokens in the mask), and the
    per-sequence variant over 2048 sequences of log-normal lengths."""

    def __init__(self, device, seed: int = 0, n: int = 4_194_304):
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        import fp8_block_quantized_gb300 as jet

        self.jet, self.M = jet, n
        self.a, self.b = (t.to(device) for t in wl.logprobs(n, seed=seed))
        self.out = torch.empty((1,), dtype=torch.float32, device=device)
        self.ws = torch.empty((max(jet.workspace_bytes("token_mult_prob_error", n), 16),),
                              dtype=torch.uint8, device=device)
        g = torch.Generator().manual_seed(seed + 5000)
        self.mask = (torch.rand(n, generator=g) < 0.75).to(torch.uint8).to(device)
        self.w = torch.empty((n,), dtype=torch.float32, device=device)
        self.mout = torch.empty((1,), dtype=torch.float32, device=device)
        self.mcount = torch.empty((1,), dtype=torch.int64, device=device)
        self.mws = torch.empty((max(jet.workspace_bytes("token_mismatch_masked", n), 16),),
                               dtype=torch.uint8, device=device)
        # per sequence: 2048 sequences of log-normal lengths over the same tokens
        rng = torch.Generator().manual_seed(seed + 6000)
        lens = torch.exp(torch.randn(2048, generator=rng, dtype=torch.float64) * 0.8 + 7.3)
        lens = (lens * (n / lens.sum())).floor().clamp(min=1).to(torch.int64)
        lens[-1] += n - int(lens.sum())
        self.seq_off = torch.zeros((2049,), dtype=torch.int64)
        self.seq_off[1:] = torch.cumsum(lens, 0)
        self.seq_off = self.seq_off.to(device)
        self.S = 2048
        self.sout = torch.empty((self.S,), dtype=torch.float32, device=device)
        self.scount = torch.empty((self.S,), dtype=torch.int64, device=device)
        self.sw = torch.empty((n,), dtype=torch.float32, device=device)
        # an L2-sized scratch written before each call so that its inputs are
        # read from HBM every step
        self.flush = torch.empty((256 << 20,), dtype=torch.uint8, device=device)
        self.work = {"token_mult_prob_error": n * BYTES_PER_ELEM["token_mult_prob_error"],
                     "token_mismatch_masked": n * BYTES_PER_ELEM["token_mismatch_masked"],
                     "token_mismatch_per_sequence": n * BYTES_PER_ELEM["token_mismatch_masked"]}
        self.bytes = sum(self.work.values())
        self.flops = 0
        self.launches_per_step = 5
        self.primary = ("GB/s", self.bytes)
        self.config = {"workload": f"metric_n{n}", "tokens": n, "masked_fraction": 0.75,
                       "sequences": self.S,
                       "l2": "flushed: 256 MB written before each call, outside the kernels' events"}

    def calls(self):
        j = self.jet
        return [("l2_flush", lambda: self.flush.fill_(1), "flush"),
                ("token_mult_prob_error", lambda: j.jet_token_mult_prob_error(
                    self.a, self.b, self.out, self.ws), "n"),
                ("l2_flush", lambda: self.flush.fill_(1), "flush"),
                ("token_mismatch_masked", lambda: j.jet_token_mismatch_masked(
                    self.a, self.b, self.mask, 0.0, self.w, self.mout, self.mcount, self.mws), "n"),
                ("l2_flush", lambda: self.flush.fill_(1), "flush"),
                ("token_mismatch_per_sequence", lambda: j.jet_token_mismatch_per_sequence(
                    self.a, self.b, self.mask, self.seq_off, 0.0, self.sw, self.sout,
                    self.scount), "S2048")]


def make_step(args, device, rank, workload=None):
    workload = workload or args.workload
    if workload in ("train8b", "train32b"):
        return LayerStep(workload, device, seed=args.seed + rank)
    if workload == "rollout":
        return RolloutStep(args.tokens, device, seed=args.seed + rank)
    if workload == "sync":
        return SyncStep(device, seed=args.seed + rank)
    if workload == "moe":
        return MoeStep(device, seed=args.seed + rank)
    if workload == "moe_train":
        return MoeTrainStep(device, seed=args.seed + rank)
    if workload == "kvcache":
        return KvCacheStep(device, seed=args.seed + rank)
    return MetricStep(device, seed=args.seed + rank)


def make_graphs(calls, steps, torch, detail):
    """The step captured as CUDA graphs: (one-step graph, {family: graph of
    that family's calls of one step, in step order}, K-step graph with a
    timing event around every call (only with `detail`), its events), or None
    when this PyTorch cannot record events as graph nodes."""
    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)
        mk()
    except TypeError:
        return None
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=side):
        for _, f, _ in calls:
            f()
    # A step that flushes L2 between its calls keeps the flush in front of
    # every call of the other families' graphs too; its time is subtracted.
    flush = [c[1] for c in calls if c[0] == "l2_flush"][:1]
    g_fam = {}
    for fam in dict.fromkeys(c[0] for c in calls):
        g_fam[fam] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fam[fam], stream=side):
            for c in calls:
                if c[0] == fam:
                    if fam != "l2_flush":
                        for f in flush:
                            f()
                    c[1]()
    g_detail, ev = None, None
    if detail:
        g_detail = torch.cuda.CUDAGraph()
        ev = [[(mk(), mk()) for _ in calls] for _ in range(steps)]
        with torch.cuda.graph(g_detail, stream=side):
            cur = torch.cuda.current_stream()
            for k in range(steps):
                for (_, f, _), (a, b) in zip(calls, ev[k]):
                    a.record(cur)
                    f()
                    b.record(cur)
    torch.cuda.current_stream().wait_stream(side)
    return g_step, g_fam, g_detail, ev


def bind_to_gpu_numa_node(torch, device):
    """Restrict this process to the host CPUs that sysfs lists as local to
    the GPU (so that pinned buffers are first touched, hence placed, in that
    node's memory).  Returns the CPU list, or None if sysfs has none."""
    try:
        p = torch.cuda.get_device_properties(device)
        bdf = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bdf}/local_cpulist") as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        if not cpus or len(cpus) >= (os.cpu_count() or 1):
            return None  # nothing to restrict
        os.sched_setaffinity(0, cpus)
        return text
    except (AttributeError, OSError, ValueError):
        return None


def gpu_numa_node(torch, device):
    """The GPU's NUMA node as sysfs lists it, or None."""
    try:
        p = torch.cuda.get_device_properties(device)
        bdf = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bdf}/numa_node") as f:
            return int(f.read().strip())
    except (AttributeError, OSError, ValueError):
        return None


def host_link_gbs(torch, device, nbytes=1 << 30):
    """Plain pinned-host <-> device copy rates (GB/s), one direction at a time:
    what bounds the end-to-end leg."""
    h = torch.empty((nbytes,), dtype=torch.uint8, pin_memory=True)
    d = torch.empty((nbytes,), dtype=torch.uint8, device=device)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        out[name] = round(3 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    del h, d
    return out


def run_e2e(args, step_a, step_b, world, device, unit, amount, scale, torch, barrier,
            outputs=False):
    """End-to-end rate through the C-ABI calls with pinned host buffers
    (`outputs`: a layer step also copies Y, dX and dW back)."""
    insts = [step_a, step_b]
    host_cpus = bind_to_gpu_numa_node(torch, device)
    link = host_link_gbs(torch, device)
    h2d = d2h = 0
    for st in insts:
        h2d, d2h = st.host_io(outputs=True) if outputs else st.host_io()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    calls = [st.calls() for st in insts]

    def enqueue(k, ev):
        i = k % 2
        st = insts[i]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev[k - 2]["cmp"])    # the inputs of this set are consumed
            for h, d in st.h_in:
                d.copy_(h, non_blocking=True)
            ev[k]["in"].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev[k]["in"])
            if k >= 2:
                s_cmp.wait_event(ev[k - 2]["out"])   # the results of this set are copied out
            for _, f, _ in calls[i]:
                f()
            ev[k]["cmp"].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev[k]["cmp"])
            for h, d in st.h_out:
                h.copy_(d, non_blocking=True)
            ev[k]["out"].record(s_out)

    mk = lambda: {n: torch.cuda.Event() for n in ("in", "cmp", "out")}
    warm = [mk() for _ in range(2)]
    for k in range(2):
        enqueue(k, warm)
    barrier()
    n = max(4, min(args.steps, 10))
    ev = [mk() for _ in range(n)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(n):
        enqueue(k, ev)
    e1.record(s_out)
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1) / n, world, device)
    return {"value": round(job_rate(world, amount, e_ms, scale), 2), "unit": unit,
            "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "host_copy_gbs": round((h2d + d2h) / (e_ms * 1e-3) / 1e9, 1),
            "host_link_gbs": link, "host_cpus": host_cpus,
            "gpu_numa_node": gpu_numa_node(torch, device),
            "max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS"),
            "steps": n, "pipelining": "2 buffer sets; copy-in, compute and copy-out streams"}


def peak_for_region(region_ms: float, pk: dict, pk_kind: str):
    """Dense FP8 peak (TFLOP/s) for a kernel family timed over `region_ms`:
    the burst cuBLAS BF16 figure x 2 when the family's timed region is
    shorter than a second (a kernel timed alone), the sustained figure
    (seconds under the power cap) otherwise.  Returns (peak, note)."""
    if region_ms < 1000.0:
        bf16, which = float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"])), "burst"
    else:
        bf16 = float(pk.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]))
        which = "sustained"
    note = (f"dense FP8 = {FP8_OVER_BF16:g} x {pk_kind} {which} cuBLAS BF16 "
            f"({which}: the family's timed region is {region_ms:.0f} ms)")
    return FP8_OVER_BF16 * bf16, note


def measure(args, workload, device, rank, world, torch, jet, barrier):
    """Time one workload: the whole step (CUDA-graph replays), each kernel
    family, the end-to-end leg; returns the JSON fields of its line."""
    step = make_step(args, device, rank, workload)
    calls = step.calls()
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        for _, f, _ in calls:
            f()
    code, word = jet.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} ({word:#x}) after warm-up")

    # ---- timed region.  The step's launches are captured once into a CUDA
    # graph: host-side enqueue work (argument checks, tensor-map encoding,
    # ctypes) then stays out of the timing, which matters for decode-sized
    # steps whose kernels last a few microseconds.  `value` = K back-to-back
    # replays of the one-step graph between two events.  Each kernel family's
    # time = K replays of a graph holding that family's calls of one step (in
    # step order, back to back) between two events: an event recorded between
    # every pair of calls would itself add microseconds per call.  With
    # --detail, a third graph of K unrolled steps with an event-record node
    # around every call gives the per-call split (those include the nodes'
    # own overhead).
    fam_ms = {}
    detail_ms = {}
    graphs = make_graphs(calls, args.steps, torch, args.detail) if not args.no_graph else None
    if graphs is not None:
        g_step, g_fam, g_detail, ev = graphs
        launch_mode = "cuda_graph"
    else:
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in calls] for _ in range(args.steps)]
        launch_mode = "stream"
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(int(device.index or 0)) as clk:
        clk.wait_first()
        if graphs is not None:
            g_step.replay()          # one untimed replay: graph upload
            for g in g_fam.values():
                g.replay()
            barrier()
            clk.mark()
            t0.record(stream)
            for k in range(args.steps):
                g_step.replay()
            t1.record(stream)
            barrier()
            # A timed region shorter than a few sampling periods is followed
            # by untimed replays of the same step, so that the clock samples
            # describe the GPU under this load.
            n0, tw = clk.count(), time.perf_counter()
            while clk.count() - n0 < 3 and time.perf_counter() - tw < 2.0:
                for k in range(args.steps):
                    g_step.replay()
                barrier()
            for fam, g in g_fam.items():
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for k in range(args.steps):
                    g.replay()
                b.record(stream)
                b.synchronize()
                fam_ms[fam] = a.elapsed_time(b)
            if "l2_flush" in fam_ms:
                per_flush = fam_ms["l2_flush"] / sum(c[0] == "l2_flush" for c in calls)
                for fam in fam_ms:
                    if fam != "l2_flush":
                        fam_ms[fam] -= per_flush * sum(c[0] == fam for c in calls)
            if g_detail is not None:
                g_detail.replay()
            barrier()
        else:
            clk.mark()
            t0.record(stream)
            for k in range(args.steps):
                for (fam, f, _), (a, b) in zip(calls, ev[k]):
                    a.record(stream)
                    f()
                    b.record(stream)
            t1.record(stream)
            barrier()
    total_ms = t0.elapsed_time(t1)
    if ev is not None:
        by_call = {}
        for k in range(args.steps):
            for (fam, _, label), (a, b) in zip(calls, ev[k]):
                ms = a.elapsed_time(b)
                by_call[fam] = by_call.get(fam, 0.0) + ms
                detail_ms[(fam, label)] = detail_ms.get((fam, label), 0.0) + ms
        if graphs is None:
            fam_ms = by_call
    code, word = jet.device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} ({word:#x}) after timing")
    total_ms = max_over_ranks(total_ms, world, device)
    # the L2 flush between metric steps is excluded from the step time
    flush_ms = fam_ms.pop("l2_flush", 0.0)
    if flush_ms:
        total_ms -= max_over_ranks(flush_ms, world, device)
        detail_ms = {k: v for k, v in detail_ms.items() if k[0] != "l2_flush"}
    ms_per_step = total_ms / args.steps
    unit, amount = step.primary
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    value = job_rate(world, amount, ms_per_step, scale)
    del graphs
    clocks = clk.summary()

    # ---- end to end: pinned host inputs in, results out, through the same
    # calls.  Every step copies all of its inputs in from pinned host memory
    # and its result back; the copies are pipelined the way a caller would
    # run them: two sets of device buffers, inputs of step k+1 copied in (one
    # stream) while step k computes (a second) and step k-1's results are
    # copied out (a third), with events ordering each buffer's reuse.  Layer
    # steps also report a second variant that copies Y, dX and dW back too.
    e2e = e2e_out = None
    if not args.no_e2e and hasattr(step, "host_io"):
        step_b = make_step(args, device, rank, workload)
        e2e = run_e2e(args, step, step_b, world, device, unit, amount, scale, torch, barrier)
        if isinstance(step, LayerStep):
            e2e_out = run_e2e(args, step, step_b, world, device, unit, amount, scale, torch,
                              barrier, outputs=True)
        del step_b

    pk, pk_kind = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    kernels = {}
    launches = {}
    for fam, _, _ in calls:
        launches[fam] = launches.get(fam, 0) + 1
    for fam, ms in fam_ms.items():
        avg_ms = ms / args.steps
        w = step.work[fam]
        if fam.startswith("gemm"):
            fp8, _ = peak_for_region(ms, pk, pk_kind)
            rate = w / (avg_ms * 1e-3) / 1e12
            kernels[fam] = {"ms_per_step": round(avg_ms, 4), "launches_per_step": launches[fam],
                            "TFLOP/s": round(rate, 1), "frac_fp8_peak": round(rate / fp8, 4),
                            "fp8_peak": round(fp8, 1)}
            if fam + "_bytes" in step.work:
                grate = step.work[fam + "_bytes"] / (avg_ms * 1e-3) / 1e9
                kernels[fam].update({"GB/s": round(grate, 1), "frac_hbm": round(grate / hbm, 4)})
        else:
            rate = w / (avg_ms * 1e-3) / 1e9
            kernels[fam] = {"ms_per_step": round(avg_ms, 4), "launches_per_step": launches[fam],
                            "GB/s": round(rate, 1), "frac_hbm": round(rate / hbm, 4)}
    dom = max(fam_ms, key=fam_ms.get)
    dom_ms_launch = fam_ms[dom] / (args.steps * launches[dom])
    dom_work_launch = step.work[dom] / launches[dom]
    fp8_dom, fp8_note = peak_for_region(fam_ms[dom], pk, pk_kind)
    # a GEMM whose arithmetic intensity is below the ridge point (dense FP8 /
    # HBM) is bounded by streaming its operands: report it against HBM
    hbm_bound_gemm = (dom.startswith("gemm") and dom + "_bytes" in step.work
                      and step.work[dom] / step.work[dom + "_bytes"] < fp8_dom * 1e3 / hbm)
    if hbm_bound_gemm:
        ach = step.work[dom + "_bytes"] / launches[dom] / (dom_ms_launch * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(ach / hbm, 4),
                "peak_note": f"{pk_kind} copy bandwidth; algorithmic bytes = codes + scales + BF16 out"}
    elif dom.startswith("gemm"):
        ach = dom_work_launch / (dom_ms_launch * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_dom, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_dom, 4), "peak_note": fp8_note}
    else:
        ach = dom_work_launch / (dom_ms_launch * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "peak_note": f"{pk_kind} copy bandwidth"}
    roof["traffic"] = measured_traffic(dom, step.config["workload"])
    quant_fams = [f for f in fam_ms if not f.startswith("gemm") and f != "token_mult_prob_error"]
    q_bytes = sum(step.work[f] for f in quant_fams)
    q_ms = sum(fam_ms[f] for f in quant_fams) / args.steps
    gemm_fams = [f for f in fam_ms if f.startswith("gemm")]
    gemm_ms = sum(fam_ms[f] for f in gemm_fams) / args.steps

    line = {
        "value": round(value, 2), "unit": unit, "ms_per_step": round(ms_per_step, 4),
        "config": dict(step.config, parallelism="replicas" if world > 1 else "single",
                       launch=launch_mode),
        "kernels": kernels,
        "roofline": roof,
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if gemm_ms > 0:
        g = step.flops / (gemm_ms * 1e-3) / 1e12
        fp8_g, _ = peak_for_region(gemm_ms * args.steps, pk, pk_kind)
        line["gemm_only"] = {"TFLOP/s": round(g, 1), "frac_fp8_peak": round(g / fp8_g, 4)}
    if q_ms > 0:
        qr = q_bytes / (q_ms * 1e-3) / 1e9
        line["quantize"] = {"GB/s": round(qr, 1), "frac_hbm": round(qr / hbm, 4)}
    if e2e is not None:
        line["e2e"] = e2e
    if e2e_out is not None:
        line["e2e_with_outputs"] = e2e_out
    if args.detail:
        line["detail_ms_per_step"] = {f"{fam}/{label}": round(ms / args.steps, 4)
                                      for (fam, label), ms in detail_ms.items()}
    del step, calls
    return line


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    import fp8_block_quantized_gb300 as jet
    jet.load()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    body = measure(args, args.workload, device, rank, world, torch, jet, barrier)
    # The default workload (the 8B-shaped layer) is followed by the 32B-shaped
    # layer in the same run, so that one line carries both training shapes.
    also = None
    if args.workload == "train8b" and not args.no_train32b:
        torch.cuda.empty_cache()
        also = measure(args, "train32b", device, rank, world, torch, jet, barrier)

    if rank == 0:
        line = {"metric": METRIC, "value": body.pop("value"), "unit": body.pop("unit"),
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": body.pop("ms_per_step"), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic"}
        line.update(body)
        if also is not None:
            line["train32b"] = also
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, seconds=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def source_hash(files) -> str:
    """sha256 (first 16 hex digits) over the given csrc files, in order."""
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "fp8_block_quantized_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel sources (the kernel's file and the headers it includes);
    otherwise null."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(workload, {}).get(kernel)
        if not ent:
            return None
        if source_hash(ent["sources"]) != ent["sources_sha256_16"]:
            return None
        return ent["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError, TypeError):
        return None


# --------------------------------------------------------------------------
# CPU oracle: baseline and reference arm
# --------------------------------------------------------------------------

def workload_name(args) -> str:
    """The `config.workload` string of each workload (both arms use it)."""
    from fp8_block_quantized_gb300 import workloads as wl
    return {"train8b": "train8b_layer_M8192", "train32b": "train32b_layer_M16384",
            "rollout": f"rollout8b_M{args.tokens}", "sync": "sync8b_32layers",
            "metric": "metric_n4194304", "moe": f"moe_qwen3_30b_a3b_T{wl.MOE_TOKENS}",
            "moe_train": f"moe_train_qwen3_30b_a3b_T{wl.MOE_TOKENS}",
            "kvcache": "kvcache8b_T65536"}[args.workload]


class CpuSample:
    """A bounded sample of a workload for the CPU oracle: `step(nthreads)`
    runs the oracle's pass over it, `amount` is its work in the workload's
    unit (FLOPs or bytes, the GPU arm's algorithmic count), `desc` says
    what the sample is."""

    def __init__(self, workload: str, seed: int = 0):
        import numpy as np
        import torch
        from fp8_block_quantized_gb300 import workloads as wl
        self.unit = "TFLOP/s"
        b = wl.bf16_bits
        if workload in ("train8b", "train32b", "rollout"):
            kind = "train8b" if workload == "rollout" else workload
            name, N, K = wl.layer_linears(kind)[0]
            cfg, T = wl.CONFIG_ID[workload], 128
            self.x = b(wl.activations(T, K, seed=seed, config=cfg, tensor_id=0))
            self.g = b(wl.norm_gain(K, seed=seed, config=cfg, tensor_id=600))
            self.eps = RMS_EPS[kind]
            self.w = b(wl.weights(N, K, seed=seed, config=cfg, tensor_id=100))
            if workload == "rollout":
                import oracle
                self.qw, self.sw = oracle.quant_w_128x128(self.w)
                self.run = self._rollout
                self.amount = 2 * T * N * K
                self.desc = (f"{name} projection at {T} tokens: RMSNorm fused with the 1x128 "
                             f"quantization of X and the binary64 forward product (weights "
                             f"quantized beforehand)")
            else:
                self.dy = b(wl.grad_output(T, N, seed=seed, config=cfg, tensor_id=200))
                self.run = self._train
                self.amount = 3 * 2 * T * N * K
                self.desc = (f"{name} projection chain (N={N}, K={K}) at {T} tokens: 128x128 "
                             f"weight quantization, RMSNorm + 1x128 of X, 1x128 of dY, 128x1 "
                             f"requant of both, binary64 forward/dgrad/wgrad")
        elif workload == "sync":
            self.unit = "GB/s"
            self.w = b(wl.weights(4096, 4096, seed=seed, config=5, tensor_id=1000))
            self.x = b(wl.heavy_activations(128, 14336, seed=seed))
            self.run = self._sync
            self.amount = (4096 * 4096 * BYTES_PER_ELEM["quant_w_128x128"]
                           + 128 * 14336 * BYTES_PER_ELEM["quant_act_1x128"])
            self.desc = "one 4096 x 4096 weight (128x128) and 128 x 14336 activations (1x128)"
        elif workload == "metric":
            self.unit = "GB/s"
            n = 262144
            a, c = wl.logprobs(n, seed=seed)
            self.a, self.c = a.numpy(), c.numpy()
            g = torch.Generator().manual_seed(seed + 5000)
            self.mask = (torch.rand(n, generator=g) < 0.75).to(torch.uint8).numpy()
            self.run = self._metric
            self.amount = n * (BYTES_PER_ELEM["token_mult_prob_error"]
                               + BYTES_PER_ELEM["token_mismatch_masked"])
            self.desc = f"n = {n} tokens: the plain and the masked metric (binary64)"
        elif workload in ("moe", "moe_train"):
            import oracle
            E, T = 4, 128                      # experts, tokens per expert (whole groups)
            (gn, Ng, Kg), (dn, Nd, Kd) = wl.MOE_LINEARS
            cfg = wl.CONFIG_ID["moe"]
            self.off = np.arange(0, (E + 1) * T, T, dtype=np.int64)
            M = E * T
            self.x = b(wl.activations(M, Kg, seed=seed, config=cfg, tensor_id=0))
            wg = wl.weights(E * Ng, Kg, seed=seed, config=cfg, tensor_id=100)
            wd = wl.weights(E * Nd, Kd, seed=seed, config=cfg, tensor_id=101)
            self.wg = b(wg).reshape(E, Ng, Kg)
            self.wd = b(wd).reshape(E, Nd, Kd)
            self.F = Kd
            fl = 2 * M * (Ng * Kg + Nd * Kd)
            if workload == "moe":
                qs = [oracle.quant_w_128x128(self.wg[e]) for e in range(E)]
                self.qwg, self.swg = np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])
                qs = [oracle.quant_w_128x128(self.wd[e]) for e in range(E)]
                self.qwd, self.swd = np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])
                self.run = self._moe
                self.amount = fl
                self.desc = (f"{E} experts x {T} tokens: 1x128 quantization, grouped gate_up, "
                             f"SwiGLU + 1x128, grouped down (binary64 products)")
            else:
                self.dyd = b(wl.grad_output(M, Nd, seed=seed, config=cfg, tensor_id=210))
                self.dyg = b(wl.grad_output(M, Ng, seed=seed, config=cfg, tensor_id=211))
                self.run = self._moe_train
                self.amount = 3 * fl
                self.desc = (f"{E} experts x {T} tokens: weight quantization, forward, grouped "
                             f"DGrad and WGrad of gate_up and down (binary64 products)")
        elif workload == "kvcache":
            self.unit = "GB/s"
            T, H, D = 4096, 8, 128
            g = torch.Generator().manual_seed(seed + 7000)
            mk = lambda: (torch.randn((T, H, D), generator=g)
                          * torch.exp2(torch.rand((1, H, 1), generator=g) * 6 - 3)).to(torch.bfloat16)
            self.k, self.v = b(mk()), b(mk())
            self.slots = torch.randperm(2 * T, generator=g)[:T].numpy()
            self.cache = np.zeros((2 * T, H, D), np.uint8)
            self.run = self._kv
            n = T * H * D
            self.amount = 2 * n * 2.0 + 2 * (n * 3.0 + 8 * T)
            self.desc = f"{T} tokens x {H} heads x {D}: calibration and cache write of K and V"
        else:
            raise ValueError(workload)

    def _train(self, nt):
        import oracle
        qw, sw = oracle.quant_w_128x128(self.w, nthreads=nt)
        qx, sx = oracle.rmsnorm_quant_1x128(self.x, self.g, self.eps, nthreads=nt)
        oracle.gemm_fwd(qx, sx, qw, sw, nthreads=nt)
        qdy, sdy = oracle.quant_act_1x128(self.dy, nthreads=nt)
        oracle.gemm_dgrad(qdy, sdy, qw, sw, nthreads=nt)
        qxT, sxT = oracle.requant_128x1(qx, sx, nthreads=nt)
        qdyT, sdyT = oracle.requant_128x1(qdy, sdy, nthreads=nt)
        oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT, nthreads=nt)

    def _rollout(self, nt):
        import oracle
        qx, sx = oracle.rmsnorm_quant_1x128(self.x, self.g, self.eps, nthreads=nt)
        oracle.gemm_fwd(qx, sx, self.qw, self.sw, nthreads=nt)

    def _sync(self, nt):
        import oracle
        oracle.quant_w_128x128(self.w, nthreads=nt)
        oracle.quant_act_1x128(self.x, nthreads=nt)

    def _metric(self, nt):
        import oracle
        oracle.token_mult_prob_error(self.a, self.c)
        oracle.token_mismatch_masked(self.a, self.c, self.mask)

    def _moe_forward(self, qwg, swg, qwd, swd, nt):
        import numpy as np
        import oracle
        from fp8_block_quantized_gb300.workloads import bf16_bits as wl_bf16
        qx, sx = oracle.quant_act_1x128(self.x, nthreads=nt)
        y = oracle.gemm_fwd_grouped(qx, sx, qwg, swg, self.off, nthreads=nt)
        import torch
        yb = wl_bf16(torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16))
        F = self.F
        qh, sh = oracle.swiglu_quant_1x128(np.ascontiguousarray(yb[:, :F]),
                                           np.ascontiguousarray(yb[:, F:]), nthreads=nt)
        oracle.gemm_fwd_grouped(qh, sh, qwd, swd, self.off, nthreads=nt)
        return qx, sx, qh, sh

    def _moe(self, nt):
        self._moe_forward(self.qwg, self.swg, self.qwd, self.swd, nt)

    def _moe_train(self, nt):
        import numpy as np
        import oracle
        E = self.wg.shape[0]
        qs = [oracle.quant_w_128x128(self.wg[e], nthreads=nt) for e in range(E)]
        qwg, swg = np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])
        qs = [oracle.quant_w_128x128(self.wd[e], nthreads=nt) for e in range(E)]
        qwd, swd = np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])
        qx, sx, qh, sh = self._moe_forward(qwg, swg, qwd, swd, nt)
        for dy, qw, sw, qa, sa in ((self.dyd, qwd, swd, qh, sh), (self.dyg, qwg, swg, qx, sx)):
            qdy, sdy = oracle.quant_act_1x128(dy, nthreads=nt)
            oracle.gemm_dgrad_grouped(qdy, sdy, qw, sw, self.off, nthreads=nt)
            qdyT, sdyT = oracle.requant_128x1(qdy, sdy, nthreads=nt)
            qaT, saT = oracle.requant_128x1(qa, sa, nthreads=nt)
            oracle.gemm_wgrad_grouped(qdyT, sdyT, qaT, saT, self.off, nthreads=nt)

    def _kv(self, nt):
        import oracle
        for x in (self.k, self.v):
            s = oracle.kv_calibrate(x)
            oracle.kv_cache_write(x, s, self.slots, self.cache)

    def step(self, nthreads):
        self.run(nthreads)

    def rate(self, reps, seconds):
        return reps * self.amount / seconds / (1e12 if self.unit == "TFLOP/s" else 1e9)


def usable_cores() -> int:
    """Host cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0)) or 1
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload: str, seconds: float = 12.0):
    import oracle
    oracle.build()
    nthreads = usable_cores()
    smp = CpuSample(workload)
    reps, t0 = 0, time.perf_counter()
    while True:
        smp.step(nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 200:
            break
    return {"value": round(smp.rate(reps, el), 6), "unit": smp.unit, "cores": nthreads,
            "kind": "oracle", "seconds": round(el, 2), "reps": reps,
            "sample": f"{smp.desc}; {reps} passes"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    nthreads = usable_cores()
    smp = CpuSample(args.workload, seed=args.seed)
    for _ in range(args.warmup):
        smp.step(nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.step(nthreads)
    el = time.perf_counter() - t0
    value = smp.rate(args.steps, el)
    sample_desc = f"{smp.desc}, one pass per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": smp.unit,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_name(args), "sample": sample_desc},
            "cpu_baseline": {"value": round(value, 6), "unit": smp.unit, "cores": nthreads,
                             "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": round(value, 6), "unit": smp.unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("jet", "reference"), default="jet")
    ap.add_argument("--workload", choices=("train8b", "train32b", "rollout", "sync", "metric", "moe",
                                           "moe_train", "kvcache"),
                    default="train8b",
                    help="train8b (default, the benchmark's workload), train32b, or the "
                         "rollout / weight-sync / metric / MoE expert forward / MoE expert "
                         "training / FP8 KV-cache configurations")
    ap.add_argument("--tokens", type=int, default=2048, help="M for --workload rollout")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every call from the host inside the timed region "
                         "instead of replaying a captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train32b", action="store_true",
                    help="with the default train8b workload, skip the 32B-shaped layer that "
                         "is otherwise measured after it and reported under `train32b`")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--detail", action="store_true",
                    help="also report per-launch-site kernel times")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
