"""Seeded synthetic inputs for one MoE layer.

This module only draws numbers; it contains none of the layer's arithmetic.
Both the CUDA path and the CPU oracle receive the same host tensors, so the
oracle sees exactly the bf16/fp32 bits the GPU sees.

Recipe (per tensor a separate ``torch.Generator`` seeded with
``seed * 1_000_003 + tensor_id``; ids x=1, logits=2, W1=3, W3=4, W2=5, dy=6):

* ``x``      [T, d]        N(0, 1) drawn in fp32, rounded to bf16 (RNE)
* ``logits`` [T, E]        N(0, 1) fp32; for ``zipf`` workloads plus the
                           per-expert bias fl32(2 * ln(r^-1.2 / H_{E,1.2}))
                           with rank r = e + 1, added in fp32
* ``W1, W3`` [E+S, f, d]   N(0, 0.02) (fp32 draw * 0.02), rounded to bf16,
                           drawn expert by expert; nn.Linear [out, in] layout
* ``W2``     [E+S, d, f]   as W1
* ``dy``     [T, d]        N(0, 1), rounded to bf16 (upstream gradient)

Shared-expert weights are stored after the E routed experts.
"""
from dataclasses import dataclass
import math

import torch

from .configs import MoEConfig

TENSOR_ID = {"x": 1, "logits": 2, "W1": 3, "W3": 4, "W2": 5, "dy": 6}


def _gen(seed: int, name: str) -> torch.Generator:
    return torch.Generator().manual_seed(seed * 1_000_003 + TENSOR_ID[name])


def _normal(shape, g, std=1.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def zipf_bias(E: int, s: float = 1.2, scale: float = 2.0) -> torch.Tensor:
    """Per-expert logit bias scale*ln(Zipf(s) weight of rank e+1), fp32."""
    h = math.fsum(r ** -s for r in range(1, E + 1))
    return torch.tensor([scale * math.log((e + 1) ** -s / h) for e in range(E)],
                        dtype=torch.float64).to(torch.float32)


def make_logits(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    z = _normal((cfg.T, cfg.E), _gen(seed, "logits"))
    if cfg.zipf:
        z = z + zipf_bias(cfg.E)[None, :]
    return z.contiguous()


def make_x(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    return _normal((cfg.T, cfg.d), _gen(seed, "x")).to(torch.bfloat16)


def make_dy(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    return _normal((cfg.T, cfg.d), _gen(seed, "dy")).to(torch.bfloat16)


def make_weight(cfg: MoEConfig, name: str, seed: int = 0, std: float = 0.02) -> torch.Tensor:
    nexp = cfg.E + cfg.S
    rows, cols = (cfg.d, cfg.f) if name == "W2" else (cfg.f, cfg.d)
    out = torch.empty(nexp, rows, cols, dtype=torch.bfloat16)
    g = _gen(seed, name)
    for e in range(nexp):
        out[e] = _normal((rows, cols), g, std).to(torch.bfloat16)
    return out


@dataclass
class LayerInputs:
    cfg: MoEConfig
    x: torch.Tensor
    logits: torch.Tensor
    W1: torch.Tensor
    W3: torch.Tensor
    W2: torch.Tensor
    dy: torch.Tensor


def make_layer_inputs(cfg: MoEConfig, seed: int = 0) -> LayerInputs:
    """All host tensors of one layer, fwd and bwd."""
    return LayerInputs(cfg, make_x(cfg, seed), make_logits(cfg, seed),
                       make_weight(cfg, "W1", seed), make_weight(cfg, "W3", seed),
                       make_weight(cfg, "W2", seed), make_dy(cfg, seed))
