"""bench.py's host-side accounting, CPU only: the algorithmic FLOPs and bytes
the roofline fractions divide by, and the peak fallbacks."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import OLMOE, TINY  # noqa: E402


def test_olmoe_algorithmic_figures():
    """The OLMoE-shaped layer (n=4096, H=2048, I=1024, E=64, K=8, bf16): GEMM1
    4·nK·H·I = 275 GFLOP over x_perm + W13 + h = 738 MB; GEMM2 137 GFLOP
    (+ the weighting) over h + W2 + y = 470 MB; permute and combine 151 MB."""
    a = bench.algorithmic(OLMOE)
    nK, H, I, E = 4096 * 8, 2048, 1024, 64
    assert a["gemm1"]["flop"] == 4 * nK * H * I == 274877906944
    assert a["gemm1"]["bytes"] == nK * H * 2 + E * H * 2 * I * 2 + nK * I * 2 == 738197504
    assert a["gemm2"]["flop"] == 2 * nK * I * H + nK * H
    assert round(a["gemm2"]["bytes"] / 1e6) == 470
    assert round(a["permute"]["bytes"] / 1e6) == 151
    assert round(a["combine"]["bytes"] / 1e6) == 151
    assert a["router"]["flop"] == 2 * 4096 * H * E


def test_empty_experts_carry_no_weight_bytes():
    counts = [0] * 32 + [1024] * 32
    full, half = bench.algorithmic(OLMOE), bench.algorithmic(OLMOE, counts)
    w13 = 2048 * 2 * 1024 * 2
    assert full["gemm1"]["bytes"] - half["gemm1"]["bytes"] == 32 * w13
    assert full["gemm1"]["flop"] == half["gemm1"]["flop"]


def test_float32_layers_count_four_bytes():
    a = bench.algorithmic(TINY)
    n, H, K = TINY.n, TINY.H, TINY.K
    assert a["permute"]["bytes"] == n * H * 4 + n * K * H * 4 + n * K * 4


def test_fallback_peaks():
    assert bench.FALLBACK_PEAKS["hbm_gbs"] == 6800.0
    assert bench.FALLBACK_PEAKS["bf16_tflops"] == 1900.0
