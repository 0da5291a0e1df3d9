"""Seeded synthetic inputs for the MoE layer (shared by the CUDA path's tests,
the benchmark and the oracle comparisons).

Distributions (standard deviations):
  x      ~ N(0, 1)                      (n, H)
  W_gate ~ N(0, 0.02)                   (H, E)
  W13[e] ~ N(0, 1/sqrt(H))              (H, 2I); columns [0, I) gate, [I, 2I) up
  W2[e]  ~ N(0, 1/sqrt(I))              (I, H)
  bias   (skewed workload only)         (E,) float32, see `skew_bias`

Values are drawn in float32 with torch's generator on the target device and
then cast to the workload dtype; the cast values are the inputs.  Every tensor
(and every expert slice) has its own sub-seed derived from the workload seed,
the tensor name and the expert index, so a tensor can be regenerated alone.

This module computes none of the layer's arithmetic (no routing, no GEMM).
"""
from __future__ import annotations

import hashlib
import math

import torch

from .configs import MoEConfig, SKEW_BETA, SKEW_COLD, SKEW_ZIPF_S

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(cfg: MoEConfig) -> torch.dtype:
    return _TORCH_DTYPE[cfg.dtype]


def sub_seed(seed: int, name: str, index: int = -1) -> int:
    h = hashlib.sha256(f"{seed}/{name}/{index}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, name: str, index: int = -1) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, name, index))
    return g


def _randn(shape, std, dtype, device, seed, name, index=-1):
    g = _gen(device, seed, name, index)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_x(cfg: MoEConfig, device, seed: int | None = None, n: int | None = None):
    s = cfg.seed if seed is None else seed
    rows = cfg.n if n is None else n
    return _randn((rows, cfg.H), 1.0, torch_dtype(cfg), device, s, "x")


def make_w_gate(cfg: MoEConfig, device):
    return _randn((cfg.H, cfg.E), 0.02, torch_dtype(cfg), device, cfg.seed, "w_gate")


def make_w13(cfg: MoEConfig, device):
    dt = torch_dtype(cfg)
    w = torch.empty((cfg.E, cfg.H, 2 * cfg.I), dtype=dt, device=device)
    std = 1.0 / math.sqrt(cfg.H)
    for e in range(cfg.E):
        w[e].copy_(_randn((cfg.H, 2 * cfg.I), std, dt, device, cfg.seed, "w13", e))
    return w


def make_w2(cfg: MoEConfig, device):
    dt = torch_dtype(cfg)
    w = torch.empty((cfg.E, cfg.I, cfg.H), dtype=dt, device=device)
    std = 1.0 / math.sqrt(cfg.I)
    for e in range(cfg.E):
        w[e].copy_(_randn((cfg.I, cfg.H), std, dt, device, cfg.seed, "w2", e))
    return w


def skew_bias(cfg: MoEConfig, beta: float = SKEW_BETA, cold: int = SKEW_COLD):
    """Per-expert logit bias with a Zipf(s)-like ranking.

    A seeded permutation assigns each expert a rank r_e in 1..E; the bias is
    b_e = -s * beta * ln(r_e), so exp(b_e) = r_e^(-s*beta).  The `cold`
    highest ranks get b_e = -inf: those experts are never chosen.  Returned on
    the CPU as float32.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(sub_seed(cfg.seed, "skew_rank"))
    rank = torch.randperm(cfg.E, generator=g) + 1           # r_e in 1..E
    b = -SKEW_ZIPF_S * beta * torch.log(rank.to(torch.float64))
    b[rank > cfg.E - cold] = -math.inf
    return b.to(torch.float32)


def make_bias(cfg: MoEConfig, device):
    if not cfg.skew:
        return None
    return skew_bias(cfg).to(device)


def make_layer(cfg: MoEConfig, device):
    """All weights of the layer: dict(w_gate, bias, w13, w2)."""
    return {
        "w_gate": make_w_gate(cfg, device),
        "bias": make_bias(cfg, device),
        "w13": make_w13(cfg, device),
        "w2": make_w2(cfg, device),
    }


def make_micro_batches(cfg: MoEConfig, device):
    """The token inputs: one tensor per micro-batch."""
    if cfg.num_mb == 1:
        return [make_x(cfg, device)]
    return [make_x(cfg, device, seed=s) for s in cfg.mb_seeds]


def to_f64_numpy(t):
    """Exact upcast of a (device) tensor to a float64 numpy array on the host."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
