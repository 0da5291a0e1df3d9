"""Find the bias scale beta of the skewed-routing workload (oracle-side script).

TEST INFRASTRUCTURE.  The skewed workload adds b_e = -1.1 * beta * ln(r_e) to
the router logits (r_e a seeded rank, the coldest ranks at -inf).  This script
bisects beta so that the oracle's per-expert hit counts on that workload's
inputs have CV = sigma(n_e)/mu(n_e) close to 1.5, the imbalance measure of
"MoE 分布式推理基础（基于 vLLM）" §1.2.  The result is stored by hand as
workloads.configs.SKEW_BETA.  Inputs are drawn on the CPU here; the device
draws differ in value but not in distribution, so the CV carries over within
a few hundredths (the tests report the CV actually reached).

    python -m oracle.calibrate_skew
"""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle as O
from workloads import SKEW
from workloads import synth


def cv_for(beta, xw, cfg):
    b = synth.skew_bias(cfg, beta=beta).numpy().astype(np.float64)
    logits = xw + b[None, :]
    e_top, _ = O.topk(logits, cfg.K, cfg.norm_topk_prob)
    counts, *_ = O.dispatch_layout(e_top, cfg.E)
    return O.count_cv(counts), counts


def main(target=1.5):
    cfg = SKEW
    x = synth.to_f64_numpy(synth.make_x(cfg, "cpu"))
    wg = synth.to_f64_numpy(synth.make_w_gate(cfg, "cpu"))
    xw = O.router_logits(x, wg)
    lo, hi = 0.0, 3.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        cv, _ = cv_for(mid, xw, cfg)
        if cv < target:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    cv, counts = cv_for(beta, xw, cfg)
    print(f"beta={beta:.4f} cv={cv:.4f} zeros={int((counts == 0).sum())} "
          f"max/mean={counts.max() / counts.mean():.2f}")


if __name__ == "__main__":
    main()
