"""Helpers shared by the GPU parity tests: run the library on seeded inputs,
and evaluate the fp64 oracle on the same inputs (copied to the host)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from workloads import synth

NEAR_TIE_GAP = 1e-6
TOL = {"bf16": 1e-2, "f32": 1e-4}

f64 = synth.to_f64_numpy


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


class Run:
    """One forward of the library on a workload, with every intermediate."""

    def __init__(self, cfg, n=None, seed=None, device="cuda:0", sm_reserve=0):
        import top_routing_dispatch_gb300 as M
        self.cfg = cfg if n is None else cfg.with_(n=n)
        cfg = self.cfg
        self.dev = torch.device(device)
        self.L = synth.make_layer(cfg, self.dev)
        self.x = synth.make_x(cfg, self.dev, seed=seed)
        self.desc = M.desc_for(cfg)
        self.layer = M.MoELayer(self.desc, self.L["w_gate"], self.L["bias"], self.L["w13"],
                                self.L["w2"])
        self.y = self.layer.forward([self.x], sm_reserve=sm_reserve)[0]
        torch.cuda.synchronize()
        self.status = int(self.layer.status.item())

    def view(self, name):
        return self.layer.view(name)

    def np(self, name):
        return f64(self.view(name)) if name not in (
            "topk_idx", "counts", "offsets", "perm", "inv_perm") else self.view(name).cpu().numpy()

    # ---- oracle side
    # weights are upcast on the device by torch (exact) and copied one expert
    # at a time, so the oracle never holds all experts in float64
    def w13_get(self, e):
        return self.L["w13"][e].to(torch.float64).cpu().numpy()

    def w2_get(self, e):
        return self.L["w2"][e].to(torch.float64).cpu().numpy()

    def oracle_logits(self, rows=None):
        x = self.x if rows is None else self.x[torch.as_tensor(rows, device=self.x.device)]
        return O.router_logits(f64(x), f64(self.L["w_gate"]), f64(self.L["bias"]))

    def oracle_layer(self, rows=None):
        """Oracle forward on all tokens or on a subset (tokens are independent
        in Algorithm 2), with near-tie tokens bound to the GPU's choice."""
        idx = None if rows is None else torch.as_tensor(rows, device=self.x.device)
        x = self.x if idx is None else self.x[idx]
        x64 = f64(x)
        logits = O.router_logits(x64, f64(self.L["w_gate"]), f64(self.L["bias"]))
        near = O.near_tie_tokens(logits, self.cfg.K, NEAR_TIE_GAP)
        gpu_idx = self.view("topk_idx").cpu().numpy()
        if rows is not None:
            gpu_idx = gpu_idx[np.asarray(rows)]
        forced = (np.where(near)[0], gpu_idx[near])
        r = O.moe_forward(x64, f64(self.L["w_gate"]), f64(self.L["bias"]), self.w13_get,
                          self.w2_get, self.cfg.K, self.cfg.norm_topk_prob, forced=forced)
        r["near"] = near
        return r


def valid_near_tie_choice(logits_row, chosen, K, gap=NEAR_TIE_GAP):
    """The chosen experts form a top-K of `logits_row` up to `gap`, in
    descending order up to `gap`."""
    s = np.sort(logits_row)[::-1]
    vals = logits_row[np.asarray(chosen)]
    return (len(set(chosen)) == K and np.all(vals >= s[K - 1] - gap)
            and np.all(np.diff(vals) <= gap))


def tie_margin(cfg):
    """The router's relative near-tie margin for this layer: tensor-core
    logits (bf16, E % 64 == 0, K <= 8, K < E) or FMA-unit logits."""
    tc = cfg.dtype == "bf16" and cfg.E % 64 == 0 and cfg.H % 64 == 0 and 1 <= cfg.K <= 8 \
        and cfg.K < cfg.E
    return 1e-4 * max(1.0, cfg.H / 2048.0) if tc else 1e-3


def logit_error_within_margin(gpu_logits, oracle_logits, margin):
    """Per token: the largest float32 logit error is below half the rescoring
    margin (margin * max(1, |largest logit|)) -- the condition under which a
    token that is not rescored cannot be ordered differently from the exact
    logits.  Returns (ok, worst ratio error / half-margin, max abs error)."""
    lo = np.asarray(oracle_logits)
    lg = np.asarray(gpu_logits)
    fin = np.isfinite(lo)
    err = np.where(fin, np.abs(lg - np.where(fin, lo, 0.0)), 0.0).max(axis=1)
    top = np.where(fin, lo, -np.inf).max(axis=1)
    half = 0.5 * margin * np.maximum(1.0, np.abs(top))
    ratio = err / half
    return bool(np.all(ratio < 1.0)), float(ratio.max()), float(err.max())
