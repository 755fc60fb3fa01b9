"""Seeded synthetic inputs for the FP8 linear-layer workloads.

This module only draws random tensors; it holds none of the quantization or
GEMM arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
All draws use ``torch.Generator`` seeded with ``seed + 1000 * config + tensor_id``
and are rounded to BF16 (round-to-nearest-even) at the end.

Workloads (the shapes are those of the Llama-3.1-8B and a 32B-class layer; the
pages run RL on such models, see "Jet-RL ..." (gist.science), "Experimentelle
Ergebnisse", and the 163.com article, section 四):

* ``single``  - one linear, M=256 tokens, K=N=512.  X ~ N(0,1) with 4 random
  channels x50 and one all-zero 1x128 group; W ~ N(0, 0.02); dY ~ N(0, 1e-3).
* ``rollout`` - forward GEMMs of the 8B shapes at M in {1,16,64,256,2048};
  X ~ N(0,1) with round(0.001*K) (>= 1) outlier channels x50.
* ``train8b`` / ``train32b`` - the 7 linears of one 8B-shaped layer at M=8192
  or 32B-shaped layer at M=16384; X as ``rollout``; dY ~ N(0, 1e-3) with a
  Bernoulli(0.01) mask of entries replaced by 1e-3 * t(3).
* ``sync``    - 128x128 quantization of 32 layers of 8B weights ~ N(0, 0.02)
  and 1x128 quantization of a 16384 x 14336 t(3) activation matrix.
* ``metric``  - n = 4,194,304 tokens, logp_rollout = log U(1e-4, 1),
  logp_train = logp_rollout + N(0, 0.02), float32.
* ``moe``     - the expert linears of one mixture-of-experts layer shaped like
  Qwen3-30B-A3B (hidden 2048, 128 experts, expert FFN width 768, top-8
  routing): 4096 tokens routed to 8 distinct experts each, drawn with
  probabilities softmax(N(0,1)) over the experts (a skewed load with ragged,
  sometimes empty, experts); X as ``rollout``, W ~ N(0, 0.02) per expert.
  The FP8 MoE experiment is on the 163.com / nmedialink pages ("在专家混合
  模型中的突破"); the layer shape is the public model configuration.

"N(0, s)": s is the standard deviation.  Student-t(3) is drawn as
Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3) with independent standard normals.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# (name, N = out_features, K = in_features); k and v are separate GEMMs.
LLAMA8B_LINEARS = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
DENSE32B_LINEARS = (
    ("q", 8192, 5120),
    ("k", 1024, 5120),
    ("v", 1024, 5120),
    ("o", 5120, 8192),
    ("gate", 25600, 5120),
    ("up", 25600, 5120),
    ("down", 5120, 25600),
)
# Linears of one layer that read the same input activation.
SHARED_INPUT = {"q": "attn_in", "k": "attn_in", "v": "attn_in", "o": "attn_out",
                "gate": "mlp_in", "up": "mlp_in", "down": "mlp_act"}
ROLLOUT_M = (1, 16, 64, 256, 2048)
CONFIG_ID = {"single": 1, "rollout": 2, "train8b": 3, "train32b": 4, "sync": 5,
             "metric": 5, "moe": 6}
# (name, N, K) of one expert of the Qwen3-30B-A3B-shaped MoE layer; gate and
# up of an expert are one [2 * 768, 2048] product.
MOE_EXPERTS, MOE_TOPK, MOE_TOKENS = 128, 8, 4096
MOE_LINEARS = (("gate_up", 1536, 2048), ("down", 2048, 768))


def _gen(seed: int, config: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 1000 * int(config) + int(tensor_id))
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def student_t3(shape, g, device) -> torch.Tensor:
    z = _randn(shape, g, device)
    chi = _randn(shape, g, device).square_()
    chi += _randn(shape, g, device).square_()
    chi += _randn(shape, g, device).square_()
    return z / torch.sqrt(chi / 3.0)


def activations(M: int, K: int, *, seed=0, config=2, tensor_id=0, device="cpu",
                n_outlier=None, zero_group=False) -> torch.Tensor:
    """X ~ N(0,1) [M,K] with outlier channels x50 (and optionally one zero 1x128 group)."""
    g = _gen(seed, config, tensor_id, device)
    x = _randn((M, K), g, device)
    if n_outlier is None:
        n_outlier = max(1, round(0.001 * K))
    if n_outlier:
        cols = torch.randperm(K, generator=g, device=device)[:n_outlier]
        x[:, cols] *= 50.0
    if zero_group and M > 0:
        r = int(torch.randint(0, M, (1,), generator=g, device=device))
        kb = int(torch.randint(0, K // 128, (1,), generator=g, device=device))
        x[r, kb * 128:(kb + 1) * 128] = 0.0
    return x.to(torch.bfloat16)


def weights(N: int, K: int, *, seed=0, config=2, tensor_id=100, device="cpu",
            std=0.02) -> torch.Tensor:
    g = _gen(seed, config, tensor_id, device)
    return (_randn((N, K), g, device) * std).to(torch.bfloat16)


def grad_output(M: int, N: int, *, seed=0, config=3, tensor_id=200, device="cpu",
                std=1e-3, heavy_frac=0.01) -> torch.Tensor:
    """dY ~ N(0, std) with a Bernoulli(heavy_frac) mask of entries std * t(3)."""
    g = _gen(seed, config, tensor_id, device)
    dy = _randn((M, N), g, device) * std
    if heavy_frac > 0:
        mask = torch.rand((M, N), generator=g, device=device) < heavy_frac
        t = student_t3((M, N), g, device) * std
        dy = torch.where(mask, t, dy)
    return dy.to(torch.bfloat16)


def norm_gain(K: int, *, seed=0, config=3, tensor_id=600, device="cpu",
              std=0.1) -> torch.Tensor:
    """RMSNorm gain g [K] = 1 + N(0, std) in BF16 (a learned norm weight near 1;
    the pages give no value)."""
    g = _gen(seed, config, tensor_id, device)
    return (1.0 + std * _randn((K,), g, device)).to(torch.bfloat16)


def heavy_activations(M: int, K: int, *, seed=0, config=5, tensor_id=300,
                      device="cpu") -> torch.Tensor:
    g = _gen(seed, config, tensor_id, device)
    return student_t3((M, K), g, device).to(torch.bfloat16)


def logprobs(n: int, *, seed=0, config=5, tensor_id=400, device="cpu", sigma=0.02):
    """(logp_train, logp_rollout) float32 [n]."""
    g = _gen(seed, config, tensor_id, device)
    u = torch.rand((n,), generator=g, device=device, dtype=torch.float64)
    b = torch.log(1e-4 + (1.0 - 1e-4) * u).to(torch.float32)
    a = (b.double() + sigma * torch.randn((n,), generator=g, device=device,
                                          dtype=torch.float64)).to(torch.float32)
    return a, b


@dataclass
class LinearCase:
    """One linear of a layer: X [M,K], W [N,K], dY [M,N] (BF16)."""
    name: str
    M: int
    N: int
    K: int
    x: torch.Tensor
    w: torch.Tensor
    dy: torch.Tensor | None


def single_linear(seed=0, device="cpu", M=256, N=512, K=512) -> LinearCase:
    """The single-linear case: 4 outlier channels, one all-zero group."""
    x = activations(M, K, seed=seed, config=1, tensor_id=0, device=device,
                    n_outlier=4, zero_group=True)
    w = weights(N, K, seed=seed, config=1, tensor_id=100, device=device)
    dy = grad_output(M, N, seed=seed, config=1, tensor_id=200, device=device,
                     heavy_frac=0.0)
    return LinearCase("single", M, N, K, x, w, dy)


def layer_linears(kind: str = "train8b"):
    return LLAMA8B_LINEARS if kind in ("train8b", "rollout", "sync") else DENSE32B_LINEARS


def training_layer(kind="train8b", seed=0, device="cpu", M=None, with_grad=True):
    """All 7 linears of one layer; linears sharing an input share the tensor."""
    cfg = CONFIG_ID[kind]
    if M is None:
        M = 8192 if kind == "train8b" else 16384
    lins = layer_linears(kind)
    inputs = {}
    cases = []
    for i, (name, N, K) in enumerate(lins):
        key = SHARED_INPUT[name]
        if key not in inputs:
            inputs[key] = activations(M, K, seed=seed, config=cfg,
                                      tensor_id=len(inputs), device=device)
        w = weights(N, K, seed=seed, config=cfg, tensor_id=100 + i, device=device)
        dy = (grad_output(M, N, seed=seed, config=cfg, tensor_id=200 + i,
                          device=device) if with_grad else None)
        cases.append(LinearCase(name, M, N, K, inputs[key], w, dy))
    return cases


def moe_offsets(tokens: int, experts: int, topk: int, *, seed=0, config=6, tensor_id=500,
                device="cpu") -> torch.Tensor:
    """int64 [experts + 1]: first row of each expert's tokens once the
    tokens * topk routed copies are sorted by expert.  Each token picks topk
    distinct experts with probabilities softmax(N(0,1)) drawn once per layer."""
    g = _gen(seed, config, tensor_id, "cpu")
    popularity = torch.softmax(torch.randn((experts,), generator=g, dtype=torch.float64), 0)
    pick = torch.multinomial(popularity.expand(tokens, experts), topk, replacement=False,
                             generator=g)
    counts = torch.bincount(pick.flatten(), minlength=experts)
    off = torch.zeros((experts + 1,), dtype=torch.int64)
    off[1:] = torch.cumsum(counts, 0)
    return off.to(device)


def moe_layer(seed=0, device="cpu", tokens=MOE_TOKENS, experts=MOE_EXPERTS, topk=MOE_TOPK,
              linears=MOE_LINEARS):
    """(offsets, [(name, x [M, K], w [E, N, K])]) of one MoE layer; M = tokens * topk."""
    cfg = CONFIG_ID["moe"]
    off = moe_offsets(tokens, experts, topk, seed=seed, config=cfg, device=device)
    M = int(off[-1])
    out = []
    for i, (name, N, K) in enumerate(linears):
        x = activations(M, K, seed=seed, config=cfg, tensor_id=i, device=device)
        w = weights(experts * N, K, seed=seed, config=cfg, tensor_id=100 + i,
                    device=device).view(experts, N, K)
        out.append((name, x, w))
    return off, out


def moe_pad_offsets(off: torch.Tensor, group: int = 128) -> torch.Tensor:
    """Offsets of the same experts with each expert's rows padded up to a
    whole number of `group`-token groups (the layout the expert WGrad needs)."""
    counts = (off[1:] - off[:-1] + group - 1) // group * group
    pad = torch.zeros_like(off)
    pad[1:] = torch.cumsum(counts, 0)
    return pad


def moe_scatter_padded(t: torch.Tensor, off: torch.Tensor, pad: torch.Tensor) -> torch.Tensor:
    """Rows of each expert moved from `off` to its padded start in `pad`; the
    padding rows are zero."""
    out = torch.zeros((int(pad[-1]),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    for e in range(off.numel() - 1):
        a, b, p = int(off[e]), int(off[e + 1]), int(pad[e])
        out[p:p + b - a] = t[a:b]
    return out


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a BF16 tensor's bit patterns (host copy)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
