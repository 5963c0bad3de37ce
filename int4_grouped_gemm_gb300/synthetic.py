"""Seeded synthetic inputs for the sparse MoE layer.

This module only draws random numbers in a fixed order and holds none of the
layer's arithmetic (no quantisation, routing or expert math).  Both the CUDA
path and the CPU oracle are fed from it, so that they see the same inputs.

Workload shapes follow the MoE description on the pages (a router scoring 256
experts and picking 8, plus an always-on shared expert; "Lily: Perplexity's
Custom Inference Engine for Apple Silicon", section "The architecture that
forces the issue: MoE plus Gated DeltaNet"), with hidden 2048 and expert
intermediate 512, int4 group 64 (group 32 for the tiny case).

Recipe (the pages are silent on it):
  * one ``torch.Generator`` per (config, layer), seeded with ``seed`` (layer 0)
    or ``seed * 1000 + layer``;
  * draw order: router weights [E, H] ~ N(0, 0.02) fp32, then the per-expert
    router bias (config dependent), then for e = 0..E (index E is the shared
    expert) the gate [I, H], up [I, H] and down [H, I] matrices ~ N(0, 0.02),
    then the activations x [T, H] ~ N(0, 1) rounded to bf16;
  * bias "normal": N(0, 1) per expert; bias "zipf": a seeded permutation
    assigns popularity ranks r = 1..E, ranks 1..E-32 get ln(r^-1.2 / Z), the
    last 32 ranks get -30 so that they are never picked.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    group: int
    seed: int
    has_shared: bool = True
    bias: str = "none"          # "none" | "normal" | "zipf"
    layers: int = 1
    steps: int = 0              # decode steps (chained through all layers)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=16, H=256, E=16, k=2, I=128, group=32, seed=0),
    "prefill512": MoEConfig("prefill512", T=512, H=2048, E=256, k=8, I=512, group=64, seed=1),
    "prefill4096": MoEConfig("prefill4096", T=4096, H=2048, E=256, k=8, I=512, group=64, seed=2,
                             bias="normal"),
    "decode40": MoEConfig("decode40", T=1, H=2048, E=256, k=8, I=512, group=64, seed=3,
                          layers=40, steps=256),
    "skew16384": MoEConfig("skew16384", T=16384, H=2048, E=256, k=8, I=512, group=64, seed=4,
                           bias="zipf"),
}


def layer_seed(cfg: MoEConfig, layer: int) -> int:
    return cfg.seed if layer == 0 else cfg.seed * 1000 + layer


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _router_bias(cfg: MoEConfig, g, device) -> Optional[torch.Tensor]:
    if cfg.bias == "none":
        return None
    if cfg.bias == "normal":
        return torch.randn(cfg.E, generator=g, device=device, dtype=torch.float32)
    if cfg.bias == "zipf":
        n_cold = 32
        perm = torch.randperm(cfg.E, generator=g, device=device)
        n_hot = cfg.E - n_cold
        ranks = torch.arange(1, n_hot + 1, dtype=torch.float64)
        p = ranks ** -1.2
        p = p / p.sum()
        by_rank = torch.full((cfg.E,), -30.0, dtype=torch.float64)
        by_rank[:n_hot] = torch.log(p)
        bias = torch.empty(cfg.E, dtype=torch.float64)
        bias[perm.cpu()] = by_rank
        return bias.to(torch.float32).to(device)
    raise ValueError(cfg.bias)


@dataclass
class LayerInputs:
    cfg: MoEConfig
    router_w: torch.Tensor                 # [E, H] fp32
    router_bias: Optional[torch.Tensor]    # [E] fp32 or None
    w_gate: torch.Tensor                   # [E+1, I, H] fp32 (index E = shared)
    w_up: torch.Tensor                     # [E+1, I, H] fp32
    w_down: torch.Tensor                   # [E+1, H, I] fp32
    x: Optional[torch.Tensor] = None       # [T, H] bf16
    extra: dict = field(default_factory=dict)


def make_layer(cfg: MoEConfig, layer: int = 0, device="cpu", T: Optional[int] = None,
               with_x: bool = True) -> LayerInputs:
    """Draw one layer's fp32 weights (before int4 packing) and its bf16 input."""
    g = _gen(device, layer_seed(cfg, layer))
    E, H, I = cfg.E, cfg.H, cfg.I
    nexp = E + (1 if cfg.has_shared else 0)
    router_w = torch.randn(E, H, generator=g, device=device, dtype=torch.float32) * 0.02
    bias = _router_bias(cfg, g, device)
    w_gate = torch.empty(nexp, I, H, device=device, dtype=torch.float32)
    w_up = torch.empty(nexp, I, H, device=device, dtype=torch.float32)
    w_down = torch.empty(nexp, H, I, device=device, dtype=torch.float32)
    for e in range(nexp):
        w_gate[e].normal_(0.0, 0.02, generator=g)
        w_up[e].normal_(0.0, 0.02, generator=g)
        w_down[e].normal_(0.0, 0.02, generator=g)
    x = None
    if with_x:
        x = make_x(cfg, g, device, T if T is not None else cfg.T)
    return LayerInputs(cfg, router_w, bias, w_gate, w_up, w_down, x)


def make_x(cfg: MoEConfig, g, device, T: int) -> torch.Tensor:
    return torch.randn(T, cfg.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_tokens(H: int, n: int, seed: int, device="cpu") -> torch.Tensor:
    """Fresh bf16 N(0,1) tokens [n, H] from their own seeded stream."""
    g = _gen(device, seed)
    return torch.randn(n, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_logits(T: int, E: int, seed: int, kind: str = "normal") -> torch.Tensor:
    """Synthetic fp32 router logits [T, E] for routing-only checks.

    kind "normal": N(0, 1); "ties": values drawn from a 4-level grid so that
    many exact ties occur; "equal": every logit 0.
    """
    g = _gen("cpu", seed)
    if kind == "normal":
        return torch.randn(T, E, generator=g, dtype=torch.float32)
    if kind == "ties":
        return torch.randint(0, 4, (T, E), generator=g).to(torch.float32) * 0.25
    if kind == "equal":
        return torch.zeros(T, E, dtype=torch.float32)
    raise ValueError(kind)


def make_weight_matrix(rows: int, K: int, seed: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    g = _gen(device, seed)
    return torch.randn(rows, K, generator=g, device=device, dtype=torch.float32) * std


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """Reinterpret a bf16 tensor as int16 bit patterns (no arithmetic)."""
    return t.contiguous().view(torch.int16)



@dataclass(frozen=True)
class AttnConfig:
    """Decode attention of one token (the second workload): Hq query heads
    sharing Hkv key-value heads, head dimension D, L cached positions (the
    cache holds L_cap)."""
    name: str
    Hq: int
    Hkv: int
    D: int
    L: int
    seed: int
    L_cap: int = 0        # 0: L
    k_scale: float = 1.0  # standard deviation of the keys

    @property
    def cap(self) -> int:
        return self.L_cap or self.L


# 16 query heads sharing 2 key-value heads ("Lily: ...", section "The
# architecture that forces the issue: MoE plus Gated DeltaNet"); head
# dimension 128 (the pages give none); 32K context, where the pages quote
# the packing's gain ("Inside Lily ...", "Key Optimizations at a Glance")
ATTN_CONFIGS = {
    "gqa32k": AttnConfig("gqa32k", Hq=16, Hkv=2, D=128, L=32768, seed=11),
    "gqa4k": AttnConfig("gqa4k", Hq=16, Hkv=2, D=128, L=4096, seed=12),
    "gqa128k": AttnConfig("gqa128k", Hq=16, Hkv=2, D=128, L=131072, seed=13),
}


def make_attention(cfg: AttnConfig, device="cpu"):
    """Seeded q [Hq, D], k, v [Hkv, L_cap, D] in bf16: q and v N(0, 1), k
    N(0, k_scale^2); draw order q, k, v."""
    g = _gen(device, cfg.seed)
    q = torch.randn(cfg.Hq, cfg.D, generator=g, device=device).to(torch.bfloat16)
    k = (torch.randn(cfg.Hkv, cfg.cap, cfg.D, generator=g, device=device) * cfg.k_scale).to(torch.bfloat16)
    v = torch.randn(cfg.Hkv, cfg.cap, cfg.D, generator=g, device=device).to(torch.bfloat16)
    return q, k, v
