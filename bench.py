#!/usr/bin/env python
"""Benchmark of the single-GPU MoE expert layer (router, TopK, dispatch layout,
permute, grouped SwiGLU GEMMs, combine) on the OLMoE-shaped workload
(n=4096 tokens, H=2048, I=1024, E=64, K=8, bf16), plus the two-micro-batch
two-stream schedule.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  A step is one pass of the whole layer over
one batch of synthetic tokens resident in HBM; `value` is tokens/s over all
ranks (each rank runs its own batch: weak scaling, no collective on the data
path).  L2 is flushed (a 256 MiB write) before every timed step, outside the
timed events.  --impl reference times the fp64 CPU oracle on a bounded token
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and grouped-GEMM TFLOP/s (% BF16 peak), permute/combine GB/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20          # > 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="olmoe_bf16")
    ap.add_argument("--cpu-sample", type=int, default=4096,
                    help="tokens of the workload the CPU oracle runs per measurement")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU-baseline: repeat the oracle on the sample until this much wall time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-domino", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--weights", choices=["tiled", "row"], default="tiled",
                    help="bf16 expert weights: tiled by moe_prepare_weights once, untimed "
                         "(default), or read row-major")
    ap.add_argument("--router-t", choices=["on", "off"], default="on",
                    help="bf16 layers: the router weight transposed once by moe_prepare_router "
                         "(untimed) for the near-tie rescoring, or read as stored (same results)")
    ap.add_argument("--gemm-pairs", choices=["on", "off"], default="on",
                    help="forward grouped GEMMs on CTA pairs (cta_group::2, the default) or on "
                         "single CTAs (same results)")
    ap.add_argument("--gemm-tails", choices=["auto", "on", "off"], default="auto",
                    help="fused tails of the forward pair GEMMs: chosen per launch (the default: "
                         "on at 192..384 rows per expert), always, or never (same results)")
    ap.add_argument("--extra-workloads", default="olmoe_skew_bf16,dsv3_bf16,tiny_fp32",
                    help="other single-batch workloads timed after the headline (N=1 only); "
                         "empty to skip")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), util=float(parts[4]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(load)}


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (every rank gets it); the value
    itself when running alone."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(cfg, rank):
    """Seed of a rank's token batch: rank 0 runs the workload's own inputs,
    the other replicas get their own batches (weak scaling)."""
    return cfg.seed if rank == 0 else cfg.seed + 1000 * rank


def aggregate_tokens_per_s(tokens_per_rank_step, steps, world, max_total_ms):
    """Whole-job throughput: the tokens all ranks processed over the slowest
    rank's time."""
    return world * tokens_per_rank_step * steps / (max_total_ms * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------ CPU oracle arm
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(cfg, x_rows, w_gate, bias, w13, w2, reps=1):
    """Wall seconds of the fp64 oracle on the given token rows (host arrays;
    weights as float32 host arrays, upcast per expert inside the oracle)."""
    from oracle import moe_oracle as O
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        O.moe_forward(x_rows, w_gate, bias, lambda e: w13[e], lambda e: w2[e], cfg.K,
                      cfg.norm_topk_prob)
        times.append(time.perf_counter() - t0)
    return times


def host_inputs_from_device(L, x, rows):
    import torch
    ri = torch.as_tensor(rows, device=x.device)
    f32 = lambda t: None if t is None else t.detach().to("cpu", torch.float32).numpy()
    # the row-major weights (the device run may read their tiled copies)
    return (f32(x[ri]), f32(L["w_gate"]), f32(L["bias"]), f32(L.get("w13_row", L["w13"])),
            f32(L.get("w2_row", L["w2"])))


def cpu_baseline(cfg, L, x, sample, seconds):
    """The oracle on a bounded sample, repeated until about `seconds` of wall
    time (at most 8 repetitions)."""
    rows = list(range(min(sample, cfg.n)))
    xs, wg, b, w13, w2 = host_inputs_from_device(L, x, rows)
    times = []
    while sum(times) < seconds and len(times) < 8:
        times += time_oracle(cfg, xs, wg, b, w13, w2, reps=1)
    t = sum(times)
    return {"value": len(rows) * len(times) / t, "unit": UNIT, "cores": host_cores(),
            "kind": "oracle",
            "sample": f"{len(rows)} of the {cfg.n} tokens of the {cfg.name} workload (all "
                      f"{cfg.E} experts' weights) x {len(times)} runs, fp64 numpy oracle, "
                      f"{t:.1f} s wall"}


def run_reference(args, cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from workloads import synth
    L = synth.make_layer(cfg, "cpu")
    x = synth.make_x(cfg, "cpu")
    rows = list(range(min(args.cpu_sample, cfg.n)))
    xs, wg, b, w13, w2 = host_inputs_from_device(L, x, rows)
    del L, x
    for _ in range(args.warmup):
        time_oracle(cfg, xs, wg, b, w13, w2)
    times = time_oracle(cfg, xs, wg, b, w13, w2, reps=args.steps)
    tot = sum(times)
    value = len(rows) * args.steps / tot
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, sample=len(rows)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": f"each step: the first {len(rows)} tokens of the "
                                   f"{cfg.name} workload, fp64 numpy oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)
    return 0


def workload_config(cfg, **extra):
    d = {"workload": f"{cfg.name}: MoE expert layer n={cfg.n} H={cfg.H} I={cfg.I} E={cfg.E} "
                     f"K={cfg.K} {cfg.dtype} norm_topk_prob={cfg.norm_topk_prob}",
         "n": cfg.n, "H": cfg.H, "I": cfg.I, "E": cfg.E, "K": cfg.K,
         "l2": "flushed (256 MiB write) before every timed step"}
    d.update(extra)
    return d


# ------------------------------------------------------------ GPU arm
def algorithmic(cfg, counts=None):
    """Algorithmic FLOPs and bytes per phase for one micro-batch (the figures
    the design notes define; weights of empty experts are not counted)."""
    n, H, I, E, K = cfg.n, cfg.H, cfg.I, cfg.E, cfg.K
    nK, b = n * K, (2 if cfg.dtype == "bf16" else 4)
    used = E if counts is None else int(sum(1 for c in counts if c > 0))
    return {
        "router": {"flop": 2 * n * H * E, "bytes": n * H * b + H * E * b + 2 * n * E * 4 + 2 * nK * 4},
        "layout": {"flop": 0, "bytes": 2 * nK * 4 + 2 * nK * 4 + (2 * E + 1) * 4},
        "permute": {"flop": 0, "bytes": n * H * b + nK * H * b + nK * 4},
        "permute_scatter": {"flop": 0, "bytes": n * H * b + nK * H * b + nK * 4},
        "permute_gather": {"flop": 0, "bytes": n * H * b + nK * H * b + nK * 4},
        "gemm1": {"flop": 4 * nK * H * I, "bytes": nK * H * b + used * H * 2 * I * b + nK * I * b},
        # GEMM1 with the permute fused: x once (rows are re-read from L2),
        # perm, the used experts' W13, h
        "gemm1_gather": {"flop": 4 * nK * H * I,
                         "bytes": n * H * b + nK * 4 + used * H * 2 * I * b + nK * I * b},
        # GEMM2 applies the routing weights (reads perm and topk_w) and writes
        # rows in (token, slot) order; the combine sums each token's K rows
        "gemm2": {"flop": 2 * nK * I * H + nK * H,
                  "bytes": nK * I * b + used * I * H * b + nK * H * b + 2 * nK * 4},
        "combine": {"flop": nK * H, "bytes": nK * H * b + n * H * b},
    }


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["top_routing_dispatch_gb300/csrc/gemm_tc.cu",
                "top_routing_dispatch_gb300/csrc/ptx.cuh"]


def recorded_traffic(profile, sources):
    """DRAM bytes per launch recorded in a profiles/ summary, if it was taken
    on the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", profile)
    try:
        txt = open(p).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not s or s.group(1) != source_sha(sources):
        return None
    return float(m.group(1))


class Timer:
    """CUDA-event timing on one stream, with an L2 flush and a short device
    sleep before every measured call so the host enqueues the whole call
    before the device reaches it (no host gaps inside the measurement)."""

    def __init__(self, torch, stream, dev):
        self.torch = torch
        self.stream = stream
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def prep(self, flush=True):
        with self.torch.cuda.stream(self.stream):
            if flush:
                self.flush.zero_()
            self.torch.cuda._sleep(300_000)

    def event(self):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def measure(self, fn, reps):
        ts = []
        for _ in range(reps):
            self.prep()
            e0 = self.event()
            fn()
            e1 = self.event()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return ts


# x above this size is permuted in scatter form by the forward (the library's
# choice in moe_forward_microbatches, mirrored here to label the rows)
SCATTER_PERMUTE_BYTES = 32 << 20


def scatter_permute(cfg):
    return cfg.n * cfg.H * (2 if cfg.dtype == "bf16" else 4) > SCATTER_PERMUTE_BYTES


def kernel_rows(M, desc, cfg, x, y, L, v, st, lws, stream):
    """The step as one C-ABI call per row of the layer (the rows the forward
    runs for this dtype and size)."""
    if scatter_permute(cfg):
        permute = lambda: M.moe_permute_scatter(desc, x, v["inv_perm"], v["x_perm"], st, stream)
    else:
        permute = lambda: M.moe_permute(desc, x, v["perm"], v["x_perm"], st, stream)
    rows = [
        ("router", lambda: M.moe_route_topk(desc, x, L["w_gate"], L["bias"], v["topk_idx"],
                                            v["topk_w"], v["logits"], stream)),
        ("layout", lambda: M.moe_dispatch_layout(desc, v["topk_idx"], v["counts"], v["offsets"],
                                                 v["perm"], v["inv_perm"], st, lws, stream)),
        ("permute", permute),
        ("gemm1", lambda: M.moe_expert_gemm1_swiglu(desc, v["x_perm"], L["w13"], v["offsets"],
                                                    v["h"], 0, st, stream)),
    ]
    if cfg.dtype == "bf16":  # the rows the layer runs: weighting in GEMM2, slot-sum combine
        rows += [
            ("gemm2", lambda: M.moe_expert_gemm2_weighted(desc, v["h"], L["w2"], v["offsets"],
                                                          v["perm"], v["topk_w"], v["y_perm"], 0,
                                                          st, stream)),
            ("combine", lambda: M.moe_combine_slots(desc, v["y_perm"], y, stream)),
        ]
    else:  # float32 layers: expert-ordered GEMM2, then the weighting gather-combine
        rows += [
            ("gemm2", lambda: M.moe_expert_gemm2(desc, v["h"], L["w2"], v["offsets"], v["y_perm"],
                                                 0, st, stream)),
            ("combine", lambda: M.moe_combine(desc, v["y_perm"], v["topk_w"], v["inv_perm"], y,
                                              st, stream)),
        ]
    return rows


def kernel_table(cfg, per_phase, per_phase_warm, counts, peaks, rows):
    """Per-kernel time, throughput and fraction of its own roofline."""
    alg = algorithmic(cfg, counts)
    kernels = {}
    for name, ts in per_phase.items():
        ms = statistics.mean(ts)
        a = alg[name]
        k = {"ms": ms, "gbs": a["bytes"] / (ms * 1e-3) / 1e9,
             "in_step": any(name == p for p, _ in rows)}
        k["frac_hbm"] = k["gbs"] / peaks["hbm_gbs"]
        if a["flop"]:
            k["tflops"] = a["flop"] / (ms * 1e-3) / 1e12
        if name.startswith("gemm") and cfg.dtype == "bf16":
            k["frac_bf16"] = k["tflops"] / peaks["bf16_tflops"]
        # the kernel's own roofline: the larger of its tensor time (bf16 GEMMs
        # and the bf16 router) and its HBM time, over the measured time
        on_tc = cfg.dtype == "bf16" and (name.startswith("gemm") or name == "router")
        t_tensor = a["flop"] / (peaks["bf16_tflops"] * 1e12) if on_tc else 0.0
        t_hbm = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
        k["roofline_bound"] = "tensor" if t_tensor >= t_hbm else "hbm"
        k["frac_roofline"] = max(t_tensor, t_hbm) / (ms * 1e-3)
        if name in per_phase_warm:
            k["ms_warm"] = statistics.mean(per_phase_warm[name])
        kernels[name] = k
    return kernels


def compact_kernels(kernels):
    """Per kernel: ms, the fraction of its roofline and the bound, plus the
    fraction of the bf16 peak (GEMMs) or of the HBM peak (everything else)."""
    out = {}
    for name, k in kernels.items():
        c = {"ms": round(k["ms"], 5), "bound": k["roofline_bound"],
             "frac_roofline": round(k["frac_roofline"], 4),
             "frac_hbm": round(k["frac_hbm"], 4)}
        if "frac_bf16" in k:
            c["frac_bf16"] = round(k["frac_bf16"], 4)
        out[name] = c
    return out


def tiled_weights(args, cfg):
    return args.weights == "tiled" and cfg.dtype == "bf16"


def measure_layer(args, torch, M, synth, cfg, dev, peaks, rank, steps, warmup, dist=None):
    """Times one workload's layer: `steps` forward steps (one
    moe_forward_microbatches call each, L2 flushed before each), then the same
    step as one C-ABI call per row (flushed and warm).  Returns the context the
    headline's extra measurements reuse.  With tiled weights the expert
    entry points read the moe_prepare_weights copies (prepared once, before
    any timing); L keeps the row-major weights as well (the backward's)."""
    L = synth.make_layer(cfg, dev)
    x = synth.make_x(cfg, dev, seed=rank_seed(cfg, rank))
    tiled = tiled_weights(args, cfg)
    if args.router_t == "on" and cfg.dtype == "bf16":
        L["w_gate_t"] = M.moe_prepare_router(M.desc_for(cfg), L["w_gate"])
    desc = M.desc_for(cfg, tiled=tiled, w_gate_t=L.get("w_gate_t"))
    if tiled:
        L["w13_row"], L["w2_row"] = L["w13"], L["w2"]
        L["w13"], L["w2"] = M.moe_prepare_weights(M.desc_for(cfg), L["w13_row"], L["w2_row"])
    torch.cuda.synchronize()
    layer = M.MoELayer(desc, L["w_gate"], L["bias"], L["w13"], L["w2"])
    v = {k: layer.view(k) for k in ("logits", "topk_idx", "topk_w", "counts", "offsets", "perm",
                                    "inv_perm", "x_perm", "h", "y_perm")}
    lws = torch.empty(max(M.moe_layout_workspace_size(desc), 1), dtype=torch.uint8, device=dev)
    st = layer.status
    y = torch.empty_like(x)
    stream = torch.cuda.Stream(device=dev)
    rows = kernel_rows(M, desc, cfg, x, y, L, v, st, lws, stream)
    T = Timer(torch, stream, dev)

    def phased_step(flush=True):
        T.prep(flush)
        evs = [T.event()]
        for _, fn in rows:
            fn()
            evs.append(T.event())
        return evs

    def forward_step():  # the step as a user runs it: one C-ABI call
        layer.forward([x], [y], compute=stream)

    for _ in range(warmup):
        phased_step()
        T.measure(forward_step, 1)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    fwd_ms = T.measure(forward_step, steps)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    evs = [phased_step() for _ in range(steps)]
    torch.cuda.synchronize()
    clk = clocks.stop()
    per_phase = {name: [s[i].elapsed_time(s[i + 1]) for s in evs]
                 for i, (name, _) in enumerate(rows)}
    warm = [phased_step(flush=False) for _ in range(steps)]
    torch.cuda.synchronize()
    per_phase_warm = {name: [s[i].elapsed_time(s[i + 1]) for s in warm]
                      for i, (name, _) in enumerate(rows)}
    phased_ms = [s[0].elapsed_time(s[-1]) for s in evs]
    # entry points the step does not call, timed alone on the same layout:
    # the other form of the permute (gather: x re-read K times; scatter: x
    # read once)
    xp_alt = torch.empty_like(v["x_perm"])
    if scatter_permute(cfg):
        name = "permute_gather"
        other = lambda: M.moe_permute(desc, x, v["perm"], xp_alt, st, stream)
    else:
        name = "permute_scatter"
        other = lambda: M.moe_permute_scatter(desc, x, v["inv_perm"], xp_alt, st, stream)
    T.measure(other, 3)
    per_phase[name] = T.measure(other, steps)
    status = M.moe_check_status(st, stream)
    return dict(L=L, x=x, y=y, desc=desc, layer=layer, v=v, st=st, stream=stream, T=T,
                rows=rows, fwd_ms=fwd_ms, per_phase=per_phase, per_phase_warm=per_phase_warm,
                phased_ms=phased_ms, clocks=clk, status=status)


def extra_workloads(args, torch, M, synth, dev, peaks, rank):
    """The other single-batch workloads, each in a short timed block: tokens/s,
    ms per step and every kernel's fraction of its roofline."""
    from workloads import BY_NAME
    out = {}
    for name in args.extra_workloads.split(","):
        name = name.strip()
        if not name or name == args.workload:
            continue
        cfg = BY_NAME[name]
        r = measure_layer(args, torch, M, synth, cfg, dev, peaks, rank,
                          steps=max(3, min(args.steps, 10)), warmup=3)
        counts = r["v"]["counts"].cpu().tolist()
        kern = kernel_table(cfg, r["per_phase"], r["per_phase_warm"], counts, peaks, r["rows"])
        ms = statistics.mean(r["fwd_ms"])
        out[name] = {"tokens_per_s": round(cfg.n / (ms * 1e-3), 1), "ms_per_step": round(ms, 5),
                     "permute_form": "scatter" if scatter_permute(cfg) else "gather",
                     "steps": len(r["fwd_ms"]), "device_status": r["status"],
                     "clocks": r["clocks"], "kernels": compact_kernels(kern)}
        del r
        torch.cuda.empty_cache()
    return out


def run_ours(args, cfg):
    import torch
    import top_routing_dispatch_gb300 as M
    from workloads import DOMINO, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M.moe_set_gemm_pairs(args.gemm_pairs == "on")
    M.moe_set_gemm_tails({"auto": None, "on": True, "off": False}[args.gemm_tails])
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peaks, peak_src = load_peaks()

    # timed: K steps, each one moe_forward_microbatches call (L2 flushed and
    # the whole call enqueued before each step's events); then the per-kernel
    # breakdown as one C-ABI call per row with an event between calls
    r = measure_layer(args, torch, M, synth, cfg, dev, peaks, rank, args.steps, args.warmup,
                      dist)
    L, x, y, desc, layer, v, st, stream, T = (r[k] for k in ("L", "x", "y", "desc", "layer", "v",
                                                              "st", "stream", "T"))
    total_ms = max_over_ranks(sum(r["fwd_ms"]), dist, dev)
    per_phase, per_phase_warm, rows = r["per_phase"], r["per_phase_warm"], r["rows"]

    # end to end through the public C-ABI call on pinned host buffers
    # (moe_forward_host): each step copies x in, runs the layer and copies y
    # out; the copies of one step overlap the layers of its neighbours
    x_h = x.cpu().pin_memory()
    y_hs = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    pipe = M.HostPipeline(layer, compute=stream)
    for i in range(3):
        pipe(x_h, y_hs[i % 2])
    pipe.synchronize()
    torch.cuda.synchronize()
    T.prep()
    e0 = T.event()
    pipe.copy_in.wait_event(e0)
    for i in range(args.steps):
        pipe(x_h, y_hs[i % 2])
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(pipe.copy_out)
    e1.synchronize()
    e2e_total = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    # the same copies with nothing overlapped: copy in, layer, copy out, one
    # stream, per step
    y_h = y_hs[0]
    x_d = torch.empty_like(x)

    def e2e_serial_step():
        with torch.cuda.stream(stream):
            x_d.copy_(x_h, non_blocking=True)
            layer.forward([x_d], [y], compute=stream)
            y_h.copy_(y, non_blocking=True)
    for _ in range(2):
        T.measure(e2e_serial_step, 1)
    e2e_serial_total = max_over_ranks(sum(T.measure(e2e_serial_step, args.steps)), dist, dev)

    # an entry point the step does not call, timed alone on the same layout:
    # GEMM1 with the permute fused into its A loads (x_perm never written)
    if cfg.dtype == "bf16":  # the fused-gather GEMM1 exists for bf16 layers
        h_alt = torch.empty_like(v["h"])
        fused = lambda: M.moe_expert_gemm1_swiglu_gather(desc, x, v["perm"], L["w13"],
                                                         v["offsets"], h_alt, 0, st, stream)
        T.measure(fused, 3)
        per_phase["gemm1_gather"] = T.measure(fused, max(5, args.steps // 2))

    counts = v["counts"].cpu().tolist()
    alg = algorithmic(cfg, counts)
    kernels = kernel_table(cfg, per_phase, per_phase_warm, counts, peaks, rows)
    g1 = kernels["gemm1"]
    if g1["roofline_bound"] == "tensor":
        roofline = {"bound": "tensor", "achieved": g1["tflops"], "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": g1["tflops"] / peaks["bf16_tflops"]}
    else:  # the expert weights dominate (e.g. the DeepSeek-V3-sized layer)
        roofline = {"bound": "hbm", "achieved": g1["gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": g1["gbs"] / peaks["hbm_gbs"]}
    peak_kind = "bf16 burst" if roofline["bound"] == "tensor" else "HBM copy"
    roofline.update({
        "kernel": ("grouped_gemm_tc_kernel<1> (GEMM1 + SwiGLU, "
                   + ("CTA pairs)" if args.gemm_pairs == "on" else "single CTAs)")),
        "peak_source": f"{peak_src} {peak_kind}" + (" (of measured)" if peak_src == "measured"
                                                    else " (of fallback)"),
        # DRAM bytes per launch from the ncu capture of this workload's GEMM1
        "traffic": (recorded_traffic("gemm1_olmoe_bf16.md", GEMM_SOURCES)
                    if cfg.name == "olmoe_bf16" and args.gemm_pairs == "on"
                    and args.gemm_tails != "on" else None),
        "algorithmic_flop_per_launch": alg["gemm1"]["flop"],
        "algorithmic_bytes_per_launch": alg["gemm1"]["bytes"],
        # every kernel of this workload's step (and the fused-gather GEMM1)
        "kernels": compact_kernels(kernels)})

    out = {
        "metric": METRIC, "value": aggregate_tokens_per_s(cfg.n, args.steps, world, total_ms),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded Gaussian inputs and weights, random init)",
        "config": workload_config(cfg, parallelism=f"replicas x{world} (one batch per GPU)",
                                  step="one moe_forward_microbatches call (router -> layout -> "
                                       "permute -> GEMM1+SwiGLU -> GEMM2 -> combine, one stream); "
                                       "kernels: the same rows as separate C-ABI calls"),
        "roofline": roofline,
        "kernels": kernels,
        "phased_ms_per_step": statistics.mean(r["phased_ms"]),
        "weights": ("tiled by moe_prepare_weights (once, untimed)" if tiled_weights(args, cfg)
                    else "row-major"),
        "router_weight": ("also transposed by moe_prepare_router (once, untimed)"
                          if "w_gate_t" in L else "as stored"),
        "gemm_tiles": ("CTA pairs (cta_group::2), 256 x 256; fused tails "
                       + {"auto": "chosen per launch (on at 192..384 rows per expert)",
                          "on": "always", "off": "never"}[args.gemm_tails]
                       if args.gemm_pairs == "on" else "single CTAs, 128 x 256"),
        "e2e": {"value": aggregate_tokens_per_s(cfg.n, args.steps, world, e2e_total), "unit": UNIT,
                "h2d_bytes_per_step": x_h.numel() * x_h.element_size(),
                "d2h_bytes_per_step": y_h.numel() * y_h.element_size(),
                "api": "moe_forward_host (pinned host x/y; copies overlap neighbouring steps)",
                "l2": "not flushed: each step streams the expert weights (> 129 MB L2)",
                "ms_per_step": e2e_total / args.steps},
        "e2e_serial": {"value": aggregate_tokens_per_s(cfg.n, args.steps, world, e2e_serial_total),
                       "unit": UNIT, "ms_per_step": e2e_serial_total / args.steps,
                       "note": "copy in, layer, copy out in order on one stream"},
        "gpu_launches": M.kernels_per_forward(desc) * args.steps,
        "clocks": r["clocks"],
        "device_status": r["status"],
        "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count,
    }
    if not args.no_domino:
        dom = domino(args, torch, M, synth, DOMINO, dev, peaks)
        out["domino"] = dom
        roofline["overlap"] = {k: dom[k] for k in (
            "hide_ratio_eligible", "hide_ratio_strict", "hide_ratio_eligible_runs",
            "ms_compute_only_A", "ms_dispatch_combine_only_B", "ms_serial_C", "ms_overlapped_D",
            "ms_edge_phases", "ms_eligible_phases", "bitwise_equal_to_single_stream")}
    if not args.no_backward and cfg.dtype == "bf16":
        out["backward"] = backward(args, torch, M, synth, cfg, dev, peaks, layer, L, x, v, st,
                                   stream, T)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, L, x, args.cpu_sample, args.cpu_seconds)
    if args.extra_workloads and world == 1:
        del r, L, x, y, layer, v
        torch.cuda.empty_cache()
        roofline["workloads"] = extra_workloads(args, torch, M, synth, dev, peaks, rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def backward(args, torch, M, synth, cfg, dev, peaks, layer, L, x, v, st, stream, T):
    """moe_backward on the same layer: one C-ABI call per step (combine
    backward, two dgrad GEMMs, the SwiGLU-backward GEMM, two weight-gradient
    GEMMs, router backward, dx = the router term fused with the permute
    backward), L2 flushed before each step."""
    n, H, I, E, K = cfg.n, cfg.H, cfg.I, cfg.E, cfg.K
    # the backward reads row-major weights (the forward may have run on tiles)
    w13, w2 = L.get("w13_row", L["w13"]), L.get("w2_row", L["w2"])
    desc = M.desc_for(cfg)
    nK = n * K
    f32, bf = torch.float32, torch.bfloat16
    g = torch.Generator(device=dev)
    g.manual_seed(synth.sub_seed(cfg.seed, "dy"))
    dy = torch.randn((n, H), generator=g, device=dev).to(bf)
    yp = torch.empty((nK, H), dtype=bf, device=dev)  # unweighted Y rows
    M.moe_expert_gemm2(desc, v["h"], w2, v["offsets"], yp, 0, st, stream)
    dx = torch.empty_like(x)
    dwg = torch.empty((H, E), dtype=f32, device=dev)
    dbias = torch.empty(E, dtype=f32, device=dev)
    dw13 = torch.empty((E, H, 2 * I), dtype=f32, device=dev)
    dw2 = torch.empty((E, I, H), dtype=f32, device=dev)
    ws = torch.empty(M.moe_backward_workspace_size(desc), dtype=torch.uint8, device=dev)

    def step():
        M.moe_backward(desc, x, L["w_gate"], w13, w2, dy, v["logits"],
                       v["topk_idx"], v["topk_w"], v["offsets"], v["inv_perm"], v["x_perm"],
                       v["h"], yp, dx, dwg, dbias, dw13, dw2, ws, st, stream)
    T.measure(step, 3)
    ms = statistics.mean(T.measure(step, max(5, args.steps // 2)))
    flop = 16 * nK * H * I
    return {"ms_per_step": ms, "tokens_per_s": n / (ms * 1e-3),
            "tensor_flop_per_step": flop, "tflops": flop / (ms * 1e-3) / 1e12,
            "frac_bf16": flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "note": "dgrad dh, SwiGLU-backward recompute, dgrad dX, wgrad dW2 and dW13 on "
                    "the tensor cores; router backward and the dx gather on the FMA units; "
                    "L2 flushed before each step"}


def domino(args, torch, M, synth, cfg, dev, peaks):
    """Two micro-batches on two streams: the four controls of the overlap
    check (compute only, dispatch+combine only, serial, overlapped) and the
    hide ratio, strict and over the overlap-eligible phases."""
    L = synth.make_layer(cfg, dev)
    xs = synth.make_micro_batches(cfg, dev)
    wgt = (M.moe_prepare_router(M.desc_for(cfg), L["w_gate"])
           if args.router_t == "on" and cfg.dtype == "bf16" else None)
    desc = M.desc_for(cfg, tiled=tiled_weights(args, cfg), w_gate_t=wgt)
    if tiled_weights(args, cfg):
        L["w13"], L["w2"] = M.moe_prepare_weights(M.desc_for(cfg), L["w13"], L["w2"])
    layer = M.MoELayer(desc, L["w_gate"], L["bias"], L["w13"], L["w2"], num_mb=2)
    ys = [torch.empty_like(x) for x in xs]
    sc, sd = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    T = Timer(torch, sc, dev)
    st = layer.status
    V = [{k: layer.view(k, j) for k in ("logits", "topk_idx", "topk_w", "counts", "offsets",
                                         "perm", "inv_perm", "x_perm", "h", "y_perm")}
         for j in range(2)]
    lws = [torch.empty(max(M.moe_layout_workspace_size(desc), 1), dtype=torch.uint8,
                       device=dev) for _ in range(2)]

    def front(j):
        v = V[j]
        M.moe_route_topk(desc, xs[j], L["w_gate"], L["bias"], v["topk_idx"], v["topk_w"],
                         v["logits"], sc)
        M.moe_dispatch_layout(desc, v["topk_idx"], v["counts"], v["offsets"], v["perm"],
                              v["inv_perm"], st, lws[j], sc)
        M.moe_permute(desc, xs[j], v["perm"], v["x_perm"], st, sc)

    def gemms(j):
        v = V[j]
        M.moe_expert_gemm1_swiglu(desc, v["x_perm"], L["w13"], v["offsets"], v["h"], 0, st, sc)
        M.moe_expert_gemm2_weighted(desc, v["h"], L["w2"], v["offsets"], v["perm"], v["topk_w"],
                                    v["y_perm"], 0, st, sc)

    def back(j):
        v = V[j]
        M.moe_combine_slots(desc, v["y_perm"], ys[j], sc)

    R = max(5, args.steps)
    med = lambda fn: statistics.median(T.measure(fn, R))
    layer.forward(xs, ys, compute=sc)
    torch.cuda.synchronize()
    ref = [y.clone() for y in ys]
    # the four controls and the two phase groups, measured in REPS interleaved
    # rounds; the hide ratios are taken per round and their median reported
    REPS = 5
    runs = []
    sweep = {s: [] for s in (0, 8, 16, 24, 32)}
    for _ in range(REPS):
        t_a = med(lambda: (gemms(0), gemms(1)))
        t_b = med(lambda: (front(0), front(1), back(0), back(1)))
        t_edge = med(lambda: (front(0), back(1)))
        t_elig = med(lambda: (front(1), back(0)))
        t_c = med(lambda: layer.forward(xs, ys, compute=sc))
        for s in sweep:
            sweep[s].append(med(lambda: layer.forward(xs, ys, sm_reserve=s, compute=sc,
                                                      dispatch=sd)))
        t_d = sweep[0][-1]
        runs.append(dict(A=t_a, B=t_b, C=t_c, D=t_d, edge=t_edge, elig=t_elig,
                         strict=1.0 - (t_d - t_a) / t_b,
                         elig_hide=1.0 - (t_d - t_a - t_edge) / t_elig))
    sweep_med = {s: statistics.median(ts) for s, ts in sweep.items()}
    best = min(sweep_med, key=sweep_med.get)
    layer.forward(xs, ys, sm_reserve=best, compute=sc, dispatch=sd)
    torch.cuda.synchronize()
    bitwise = all(torch.equal(a, b) for a, b in zip(ys, ref))
    mk = lambda key: statistics.median(r[key] for r in runs)
    return {
        "workload": f"{cfg.name}: 2 x n={cfg.n}, seeds {list(cfg.mb_seeds)}",
        "rounds": REPS, "reps_per_control": R,
        "ms_compute_only_A": mk("A"), "ms_dispatch_combine_only_B": mk("B"),
        "ms_serial_C": mk("C"), "ms_overlapped_D": mk("D"), "sm_reserve": 0,
        "ms_overlapped_by_sm_reserve": sweep_med, "sm_reserve_best": best,
        "ms_edge_phases": mk("edge"), "ms_eligible_phases": mk("elig"),
        "hide_ratio_strict": mk("strict"),
        "hide_ratio_eligible": mk("elig_hide"),
        "hide_ratio_eligible_runs": [round(r["elig_hide"], 4) for r in runs],
        "speedup_D_vs_C": mk("C") / mk("D"),
        "tokens_per_s_overlapped": 2 * cfg.n / (mk("D") * 1e-3),
        "bitwise_equal_to_single_stream": bitwise,
    }


def main():
    args = parse_args()
    from workloads import BY_NAME
    cfg = BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
