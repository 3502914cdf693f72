"""Seeded synthetic inputs for one MoE-layer forward.

This module holds the workload shapes and the random draws that feed both the
CUDA path and the fp64 oracle.  It contains none of the layer's arithmetic:
no softmax, no top-k, no counting, no matrix products.  Everything here is a
random draw, a cast, or a fixed additive bias that shapes the routing
distribution of a workload.

Shapes follow the model tables of "Training a 1T-Params MoE on EU public
infrastructure" (Model section: hidden 6,144, 384 routed experts, top-8,
expert hidden 1,792, 65,536-token sequences) and the small 7B-A1B class of
"Scalable Pretraining of Large MoE LMs on Aurora Super Computer" (§3.1).

Draw order per call, all from one ``torch.Generator`` seeded with ``seed`` on
``device``: logits noise [T,E] fp32, then (skew only) a permutation of the
experts, then x [T,d], then for e = 0..E-1 the gate matrix [d,f], then for
each e the up matrix [d,f], then for each e the down matrix [f,d].  Every
normal is an fp32 draw; bf16 tensors are made by one round-to-nearest-even
cast after scaling.  Values depend on (config, seed, device type): the CPU
and CUDA generators are different algorithms.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    d: int          # hidden size
    E: int          # routed experts
    k: int          # experts per token
    f: int          # expert hidden size
    routing: str    # "normal" | "zipf" | "fur"
    renormalize: bool = True

    @property
    def P(self) -> int:
        """Routed (token, slot) pairs."""
        return self.T * self.k

    def as_dict(self):
        return asdict(self)


CONFIGS = {
    # tiny MoE layer: small enough for the oracle to run in full in milliseconds
    "tiny": MoEConfig("tiny", T=256, d=128, E=8, k=2, f=64, routing="normal"),
    # 7B-A1B-class layer
    "small": MoEConfig("small", T=8192, d=2048, E=64, k=8, f=1024, routing="normal"),
    # one layer of the 951.9B model, 16,384 tokens
    "t1": MoEConfig("t1", T=16384, d=6144, E=384, k=8, f=1792, routing="normal"),
    # same layer, router biased by a Zipf law over the experts
    "skew": MoEConfig("skew", T=16384, d=6144, E=384, k=8, f=1792, routing="zipf"),
    # the t1 routing shape (16,384 tokens, 384 experts, top-8: ~341 rows per
    # expert) on narrow experts: the profiling case of the per-tile behaviour
    # of the t1 GEMMs with a few GB on the device
    "t1_narrow": MoEConfig("t1_narrow", T=16384, d=1024, E=384, k=8, f=512, routing="normal"),
    # one 64k-token sequence with forced-uniform routing
    "long": MoEConfig("long", T=65536, d=6144, E=384, k=8, f=1792, routing="fur"),
}

# Zipf exponent of the skewed workload and the additive lift of the
# forced-uniform workload (far above the largest N(0,1) draw of 2.5e7 samples).
ZIPF_S = 1.2
FUR_LIFT = 16.0


def custom(name="custom", T=64, d=64, E=4, k=2, f=64, routing="normal", renormalize=True) -> MoEConfig:
    return MoEConfig(name, T=T, d=d, E=E, k=k, f=f, routing=routing, renormalize=renormalize)


def get(name_or_cfg) -> MoEConfig:
    if isinstance(name_or_cfg, MoEConfig):
        return name_or_cfg
    return CONFIGS[name_or_cfg]


def fur_assignment(T: int, E: int, k: int) -> torch.Tensor:
    """Expert of pair (t, j) under forced-uniform routing: (t*k + j) mod E.

    Every expert receives floor(T*k/E) or ceil(T*k/E) pairs and no token
    repeats an expert while k <= E.
    """
    p = torch.arange(T * k, dtype=torch.int64)
    return (p % E).view(T, k)


def zipf_bias(perm: torch.Tensor, s: float = ZIPF_S) -> torch.Tensor:
    """Per-expert logit bias -s*ln(rank), rank = perm + 1 (a permutation of 1..E)."""
    rank = perm.to(torch.float64) + 1.0
    return (-s * torch.log(rank)).to(torch.float32)


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def generate(cfg, seed: int = 0, device="cpu", weights: bool = True, x: bool = True) -> dict:
    """All inputs of one layer forward for ``cfg``.

    Returns x bf16 [T,d], logits fp32 [T,E] and (when ``weights``) w_gate,
    w_up bf16 [E,d,f] and w_down bf16 [E,f,d], all on ``device``.
    Weights are N(0, 1) scaled by 1/sqrt(fan_in) (fan_in = d for gate/up,
    f for down); x and the logits noise are N(0, 1).
    """
    cfg = get(cfg)
    dev = torch.device(device)
    g = _gen(seed, dev)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    logits = torch.randn(T, E, generator=g, device=dev, dtype=torch.float32)
    if cfg.routing == "zipf":
        perm = torch.randperm(E, generator=g, device=dev)
        logits = logits + zipf_bias(perm.cpu()).to(dev)[None, :]
    elif cfg.routing == "fur":
        assign = fur_assignment(T, E, k).to(dev)
        lift = torch.zeros(T, E, device=dev, dtype=torch.float32)
        lift.scatter_(1, assign, FUR_LIFT)
        logits = logits + lift
    elif cfg.routing != "normal":
        raise ValueError(f"unknown routing {cfg.routing!r}")
    out = {"cfg": cfg, "seed": seed, "logits": logits.contiguous()}
    if not x:
        return out
    out["x"] = torch.randn(T, d, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    if weights:
        sg = 1.0 / math.sqrt(d)
        sd = 1.0 / math.sqrt(f)
        w_gate = torch.empty(E, d, f, device=dev, dtype=torch.bfloat16)
        w_up = torch.empty(E, d, f, device=dev, dtype=torch.bfloat16)
        w_down = torch.empty(E, f, d, device=dev, dtype=torch.bfloat16)
        for e in range(E):
            w_gate[e] = (torch.randn(d, f, generator=g, device=dev) * sg).to(torch.bfloat16)
        for e in range(E):
            w_up[e] = (torch.randn(d, f, generator=g, device=dev) * sg).to(torch.bfloat16)
        for e in range(E):
            w_down[e] = (torch.randn(f, d, generator=g, device=dev) * sd).to(torch.bfloat16)
        out.update(w_gate=w_gate, w_up=w_up, w_down=w_down)
    return out


def generate_router(cfg, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router weights w_router [d, E] bf16, N(0, 1)/sqrt(d), from their own
    generator (seeded with seed + 1,000,003) so they do not shift the draws
    of ``generate``.  With x ~ N(0, 1) the router logits are about N(0, 1),
    like the workloads' logits."""
    cfg = get(cfg)
    g = _gen(seed + 1_000_003, torch.device(device))
    return (torch.randn(cfg.d, cfg.E, generator=g, device=device) / math.sqrt(cfg.d)).to(torch.bfloat16)


def generate_logits(cfg, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router logits alone, with the same values ``generate`` returns."""
    return generate(cfg, seed, device, weights=False, x=False)["logits"]
