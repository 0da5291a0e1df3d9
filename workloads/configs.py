"""Workload registry: the MoE-layer shapes the library is exercised on.

Every workload is one MoE expert layer of the single-card forward described in
"MoE 分布式推理基础（基于 vLLM）" §1.2 (Algorithm 2): n tokens of hidden size H,
E experts with intermediate size I, top-K routing.  The OLMoE shape
(H=2048, I=1024, E=64, K=8) is the model named in that page's preamble.

This module holds sizes and seeds only; it contains none of the layer's
arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    n: int            # tokens per micro-batch
    H: int            # hidden size
    I: int            # expert intermediate size (W13 is H x 2I, W2 is I x H)
    E: int            # number of experts
    K: int            # experts per token
    dtype: str        # "f32" or "bf16": x, weights, h, y_perm and y
    norm_topk_prob: bool
    seed: int
    skew: bool = False        # per-expert logit bias with a Zipf-like ranking
    num_mb: int = 1           # micro-batches (2 for the two-stream overlap run)
    mb_seeds: tuple = ()      # seeds of the micro-batch inputs (weights use `seed`)

    @property
    def nK(self) -> int:
        return self.n * self.K

    def expert_flops(self) -> int:
        """GEMM1 (4·nK·H·I) + GEMM2 (2·nK·I·H) per micro-batch."""
        return 6 * self.nK * self.H * self.I

    def router_flops(self) -> int:
        return 2 * self.n * self.H * self.E

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The five workloads of the layer.  Sizes and seeds are fixed; distributions
# are produced by workloads.synth.
TINY = MoEConfig("tiny_fp32", n=256, H=128, I=64, E=8, K=2, dtype="f32",
                 norm_topk_prob=True, seed=0)
OLMOE = MoEConfig("olmoe_bf16", n=4096, H=2048, I=1024, E=64, K=8, dtype="bf16",
                  norm_topk_prob=False, seed=1)
SKEW = MoEConfig("olmoe_skew_bf16", n=16384, H=2048, I=1024, E=64, K=8, dtype="bf16",
                 norm_topk_prob=False, seed=2, skew=True)
DSV3 = MoEConfig("dsv3_bf16", n=8192, H=7168, I=2048, E=256, K=8, dtype="bf16",
                 norm_topk_prob=True, seed=3)
DOMINO = MoEConfig("domino_2mb_olmoe_bf16", n=4096, H=2048, I=1024, E=64, K=8,
                   dtype="bf16", norm_topk_prob=False, seed=4, num_mb=2, mb_seeds=(4, 5))

ALL = (TINY, OLMOE, SKEW, DSV3, DOMINO)
BY_NAME = {c.name: c for c in ALL}

# Skewed routing: bias b_e = -1.1 * SKEW_BETA * ln(r_e) for a seeded rank r_e in
# 1..E, with the SKEW_COLD coldest ranks set to -inf.  SKEW_BETA was found by
# oracle/calibrate_skew.py (bisection on the per-expert count CV, target 1.5).
SKEW_ZIPF_S = 1.1
SKEW_BETA = 0.7174
SKEW_COLD = 4
