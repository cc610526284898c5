#!/usr/bin/env python
"""Benchmark of the Beam MoE block forward pass (router with selection bias
and group-limited top-k, dispatch, SwiGLU experts, combine) on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one full moe_forward over one batch of the decode workload
(T=64 tokens at the Beam shape: H=5120, 256 experts in 8 groups of 32, top 4
groups, top 8 experts, intermediate 2560, bf16 weights, 20 GB per layer),
replayed from a CUDA graph of that one call (the C ABI allocates nothing and
never synchronises, so it captures; a serving loop would replay it the same
way); the eager call's time is reported beside it.  Inputs are resident in HBM
when the timed region starts; L2 is flushed (a 512 MB write) before every
timed step, outside the step's events.  With
N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path has no exchange step); the value counts all ranks' tokens over
the slowest rank's time.

Besides the headline line the run measures, on rank 0: the per-stage split
(route / permute / experts / combine) through the stage entry points, the
roofline of the expert GEMMs, an end-to-end number through the C ABI with the
input and output copied between pinned host memory and the device inside
every step, the prefill workload (T=16384) as a secondary figure, and the
CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at Beam shape; decode HBM GB/s, prefill TFLOPS vs roofline"
EXPERT_BYTES = 3 * 5120 * 2560 * 2      # bf16 W_gate + W_up + W_down of one expert
FLOP_PER_TOKEN = 2 * 3 * 5120 * 2560 * 8  # expert FLOPs per token (8 routed experts)
L2_FLUSH_BYTES = 512 << 20


def traffic_per_touched_expert():
    """DRAM bytes per touched expert of the decode expert GEMMs, from the committed
    ncu figure (small-case capture, scaled by touched experts)."""
    p = os.path.join(ROOT, "profiles", "expert_gemms_decode_traffic.md")
    try:
        for line in open(p):
            if line.startswith("bytes_per_touched_expert:"):
                return int(line.split(":")[1])
    except OSError:
        pass
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sust=1400.0, src="fallback")


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"beam_moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers


class Workload:
    """Seeded inputs of one workload resident on the GPU, plus buffers."""

    def __init__(self, lib, cfg, weights, dev, stages=True, a4=None, tiled=False):
        import moe_inputs as mi
        self.cfg = cfg
        self.d = lib.dims_of(cfg)
        x, wr, b = mi.make_router_inputs(cfg)
        self.x_host = x.pin_memory()
        self.x, self.wr, self.b = x.to(dev), wr.to(dev), b.to(dev)
        self.experts = lib.Experts(*weights, a4=a4)
        if tiled:
            self.experts = self.experts.to_tiled()
        self.wdtype = self.experts.dtype
        self.ws = lib.alloc_workspace(self.d, lib.MOE_OP_FORWARD, self.wdtype, device=dev)
        T, H, k, E = cfg.T, cfg.H, cfg.top_k, cfg.E
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        if not stages:
            return
        Tk = T * k
        self.x_perm = torch.empty(Tk, H, dtype=torch.bfloat16, device=dev)
        self.offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.slot_of = torch.empty(Tk, dtype=torch.int32, device=dev)
        self.row_src = torch.empty(Tk, dtype=torch.int32, device=dev)
        self.y_partial = torch.empty(Tk, H, dtype=torch.bfloat16, device=dev)
        self.ws_route = lib.alloc_workspace(self.d, lib.MOE_OP_ROUTE, device=dev)
        self.ws_perm = lib.alloc_workspace(self.d, lib.MOE_OP_PERMUTE, device=dev)
        self.ws_exp = lib.alloc_workspace(self.d, lib.MOE_OP_EXPERTS, self.wdtype, device=dev)

    def forward(self, lib):
        lib.moe_forward(self.d, self.x, self.wr, self.b, self.experts, self.y, self.ws, self.idx,
                        self.w)


def capture_forward(lib, wl):
    """A CUDA graph of one moe_forward of the workload (same buffers)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        wl.forward(lib)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wl.forward(lib)
    torch.cuda.synchronize()
    return g


def time_steps(fn, steps, flush):
    """Per-step CUDA-event durations (ms) on the current stream, L2 flushed before each."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def stage_breakdown(lib, wl, steps, flush):
    """Route / permute / experts / combine through the stage entry points, events between."""
    names = ["route", "permute", "experts", "combine"]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    d = wl.d
    for i in range(steps):
        flush()
        e = ev[i]
        e[0].record()
        lib.moe_route(d, wl.x, wl.wr, wl.b, wl.idx, wl.w, wl.ws_route)
        e[1].record()
        lib.moe_permute(d, wl.idx, wl.x, wl.x_perm, wl.offs, wl.slot_of, wl.row_src, wl.ws_perm)
        e[2].record()
        lib.moe_experts_swiglu(d, wl.experts, wl.x_perm, wl.offs, wl.row_src, wl.w, wl.y_partial,
                               wl.ws_exp)
        e[3].record()
        lib.moe_combine(d, wl.y_partial, wl.slot_of, wl.y)
        e[4].record()
    torch.cuda.synchronize()
    out = {}
    for j, n in enumerate(names):
        out[n] = statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
    return out


def e2e_steps(lib, wl, steps, flush):
    """moe_forward with the step's input copied host->device and output device->host
    (pinned memory) inside each step's events."""
    def step():
        wl.x.copy_(wl.x_host, non_blocking=True)
        wl.forward(lib)
        wl.y_host.copy_(wl.y, non_blocking=True)
    return time_steps(step, steps, flush)


FP4_EXPERT_BYTES = 3 * (5120 * 2560 // 2 + 5120 * 2560 // 16) + 3 * 4  # codes + e4m3 scales + globals
FP8_EXPERT_BYTES = 3 * 5120 * 2560 + (2 * 2560 + 5120) * 4              # e4m3 codes + row scales
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense fp4 / bf16 tensor rate of B300


def token_major_schedule(counts, H, I, sms):
    """Load figures of the token-major expert GEMMs' static schedule (CTA b takes
    tiles b, b + grid, ...; a tile is 128 token rows of one expert against 128
    gate + 128 up or 256 down features) for expert loads `counts`: rows per
    expert, tiles and waves per GEMM, the spread of tiles over CTAs, and the
    share of MMA rows that are padding (a ragged tile costs a full one)."""
    counts = np.asarray(counts, np.int64)
    token_tiles = (counts + 127) // 128
    out = {"rows_per_expert_max": int(counts.max()), "rows_per_expert_mean": float(counts.mean()),
           "max_over_mean": float(counts.max() / counts.mean()),
           "experts_touched": int((counts > 0).sum()),
           "padded_row_frac": float(1 - counts.sum() / (128 * token_tiles.sum()))}
    for name, nf in (("gate_up", I // 128), ("down", H // 256)):
        n = int(token_tiles.sum() * nf)
        grid = max(1, min(sms, n))
        per = np.bincount(np.arange(n) % grid, minlength=grid)
        out[name] = {"tiles": n, "grid": grid, "waves": n / grid, "tiles_per_cta_max": int(per.max()),
                     "tiles_per_cta_min": int(per.min()),
                     "busy_frac": float(per.sum() / (per.max() * grid))}
    return out


def prefill_figures(lib, cfg, weights, dev, flush, peaks, steps):
    """Prefill (T=16384) or the skewed workload as a secondary figure, with
    clocks sampled over its timed steps.  Its GEMMs run inside a loop of ~10 ms
    steps, so when the samples show the power cap active (sw_power_cap) or the
    clocks below 90% of max, the peak it is compared with is the sustained one
    (cuBLAS back to back under the same cap), else the burst one; both
    fractions are printed.  The load of the expert GEMMs' tile schedule
    (token_major_schedule) comes with it."""
    pw = Workload(lib, cfg, weights, dev)
    for _ in range(2):
        pw.forward(lib)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    p_ms = statistics.mean(time_steps(lambda: pw.forward(lib), steps, flush))
    p_stage = stage_breakdown(lib, pw, 3, flush)
    clocks = sampler.stop()
    assert lib.workspace_status(pw.ws) == 0
    flop = cfg.T * FLOP_PER_TOKEN
    tflops = flop / (p_stage["experts"] / 1000.0) / 1e12
    capped = bool("sw_power_cap" in clocks.get("reasons", []) or
                  (clocks["sm_mhz"] and clocks["sm_max_mhz"] and
                   clocks["sm_mhz"] < 0.9 * clocks["sm_max_mhz"]))
    peak = peaks["bf16_sust"] if capped else peaks["bf16"]
    out = {"workload": f"{cfg.name} T={cfg.T}", "tokens_per_s": cfg.T / (p_ms / 1000.0),
           "ms_per_step": p_ms, "stages_ms": p_stage, "expert_gemm_tflops": tflops,
           "layer_tflops": flop / (p_ms / 1000.0) / 1e12,
           "peak_bf16_tflops": peak, "peak_kind": "sustained" if capped else "burst",
           "frac_of_bf16_peak": tflops / peak,
           "frac_of_burst_peak": tflops / peaks["bf16"],
           "frac_of_sustained_peak": tflops / peaks["bf16_sust"], "clocks": clocks}
    counts = np.bincount(pw.idx.cpu().numpy().ravel(), minlength=cfg.E)
    out["schedule"] = token_major_schedule(counts, cfg.H, cfg.I,
                                           torch.cuda.get_device_properties(dev).multi_processor_count)
    del pw
    torch.cuda.empty_cache()
    return out


def packed_figures(lib, mi, fmt, wts, expert_bytes, dev, flush, peaks, a4=None, tiled=False,
                   extra_T=()):
    """Packed experts (NVFP4 or FP8): decode T=64, and each T in extra_T (HBM-bound:
    packed bytes of touched experts), and prefill T=16384 (W4A16 / W8A16: the bf16
    tensor peak is its denominator; W4A4 (a4 given): the fp4 peak, the measured
    bf16 peak times the nominal fp4/bf16 ratio 13.5/2.25).  tiled: the weights in
    the tiled layout of moe_pack_nvfp4 / moe_pack_fp8."""
    out = {"layout": "tiled" if tiled else "row-major"}
    runs = [("decode", 64, 50)] + [(f"T{t}", t, 20) for t in extra_T] + [("prefill", 16384, 5)]
    for name, T, steps in runs:
        cfg = mi.CONFIGS[fmt].with_T(T)
        wl = Workload(lib, cfg, wts, dev, a4=a4, tiled=tiled)
        for _ in range(3):
            wl.forward(lib)
        torch.cuda.synchronize()
        ms = statistics.mean(time_steps(lambda: wl.forward(lib), steps, flush))
        st = stage_breakdown(lib, wl, min(steps, 20), flush)
        assert lib.workspace_status(wl.ws) == 0 and lib.workspace_status(wl.ws_exp) == 0
        touched = int(len(np.unique(wl.idx.cpu().numpy())))
        fig = {"T": T, "tokens_per_s": T / (ms / 1000.0), "ms_per_step": ms, "stages_ms": st,
               "touched_experts": touched}
        if name != "prefill":
            gbs = touched * expert_bytes / (st["experts"] / 1000.0) / 1e9
            fig.update({"expert_gemm_gbs": gbs, "frac_of_hbm_peak": gbs / peaks["hbm"],
                        "frac_of_8tbs_nominal": gbs / 8000.0})
        else:
            tf = T * FLOP_PER_TOKEN / (st["experts"] / 1000.0) / 1e12
            fig.update({"expert_gemm_tflops": tf, "frac_of_bf16_burst_peak": tf / peaks["bf16"]})
            if a4 is not None:
                fp4_peak = peaks["bf16"] * FP4_OVER_BF16
                fig.update({"peak_fp4_tflops": fp4_peak, "frac_of_fp4_peak": tf / fp4_peak,
                            "peak_fp4_source": "measured bf16 burst x nominal 13.5/2.25"})
        out[name] = fig
        del wl
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- replicas


def aggregate_replicas(ms_local: float, tokens_per_replica: int, world: int, dist=None,
                       device=None):
    """Whole-job figures of N independent replicas: the step time is the slowest
    rank's (max over ranks, one all-reduce of a scalar; no data is exchanged),
    and the value counts every rank's tokens over that time."""
    ms = ms_local
    if dist is not None and world > 1:
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_replica / (ms / 1000.0)


# ---------------------------------------------------------------- CPU oracle


def cpu_oracle_sample(wl, weights, max_seconds=25.0):
    """The oracle, as it stands, on the first tokens of the batch: routing of
    those tokens, each touched expert's SwiGLU on its rows, and the combine.
    Expert weights are copied to host one expert at a time, outside the timing."""
    import moe_inputs as mi
    import oracle
    cfg = wl.cfg
    xb = mi.bf16_bits(wl.x_host)
    wr = wl.wr.cpu().numpy()
    b = wl.b.cpu().numpy()
    wg, wu, wd = weights
    n_tok = cfg.T
    elapsed = 0.0
    t0 = time.perf_counter()
    r = oracle.route(xb[:n_tok], wr, b, cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)
    elapsed += time.perf_counter() - t0
    o = np.zeros((n_tok, cfg.top_k, cfg.H))
    done_pairs = 0
    experts = np.unique(r.idx)
    for e in experts:
        tt, kk = np.nonzero(r.idx == e)
        W = (mi.bf16_bits(wg[e]), mi.bf16_bits(wu[e]), mi.bf16_bits(wd[e]))
        t0 = time.perf_counter()
        o[tt, kk] = oracle.expert_swiglu(xb[tt], *W)
        elapsed += time.perf_counter() - t0
        done_pairs += len(tt)
        if elapsed > max_seconds:
            break
    complete = done_pairs == n_tok * cfg.top_k
    t0 = time.perf_counter()
    oracle.combine(r.w, o)
    elapsed += time.perf_counter() - t0
    tokens_equiv = n_tok * done_pairs / (n_tok * cfg.top_k)
    return {"value": tokens_equiv / elapsed, "unit": "tokens/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": (f"{'full' if complete else 'partial'} decode batch: routing of {n_tok} tokens, "
                       f"{done_pairs} (token, expert) SwiGLU evaluations over "
                       f"{len(experts) if complete else 'some'} experts, combine; "
                       f"{elapsed:.1f} s of CPU time (fp64 C oracle, OpenMP)")}


def run_reference(args, peaks):
    """The reference arm: the CPU oracle timed on the host cores, one token per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import moe_inputs as mi
    import oracle
    oracle.build()
    cfg = mi.CONFIGS["decode"]
    x, wr, b = mi.make_router_inputs(cfg)
    xb, wr, b = mi.bf16_bits(x), wr.numpy(), b.numpy()
    pool = 16  # weights drawn for 16 experts, reused round-robin: cost does not depend on values
    W = [tuple(mi.bf16_bits(m) for m in mi.make_expert(cfg, e)) for e in range(pool)]
    r = oracle.route(xb, wr, b, cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)

    def step(t):
        rr = oracle.route(xb[t:t + 1], wr, b, cfg.n_group, cfg.topk_group, cfg.top_k,
                          cfg.routed_scale)
        o = np.stack([oracle.expert_swiglu(xb[t:t + 1], *W[int(e) % pool])[0] for e in rr.idx[0]])
        oracle.combine(rr.w, o[None])

    for i in range(args.warmup):
        step(i % cfg.T)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i % cfg.T)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cores = len(os.sched_getaffinity(0))
    sample = (f"one decode token per step (its routing over 256 experts, its 8 SwiGLU experts at "
              f"H=5120/I=2560, the combine); expert weights drawn for {pool} experts and reused "
              f"round-robin, since the oracle's cost does not depend on their values")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "decode T=64, Beam MoE layer", "T": cfg.T},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    del r


# ---------------------------------------------------------------- main


def profile_config(name):
    """Workloads for --profile: the three full-size ones, and two small cases
    (32 experts, 2.5 GB of weights) that keep ncu captures to a few GB."""
    import moe_inputs as mi
    small = dict(H=5120, E=32, n_group=8, topk_group=4, top_k=8, I=2560, routed_scale=2.5)
    extra = {"prefill-small": mi.MoeConfig("prefill-small", T=4096, bias="zero", **small),
             "decode-small": mi.MoeConfig("decode-small", T=64, **small),
             "nvfp4-decode": mi.CONFIGS["nvfp4"],
             "fp8-decode": mi.CONFIGS["fp8"],
             "nvfp4-prefill": mi.CONFIGS["nvfp4"].with_T(16384),
             "nvfp4-decode-small": mi.MoeConfig("nvfp4-decode-small", T=64, weights="nvfp4", **small),
             "nvfp4-prefill-small": mi.MoeConfig("nvfp4-prefill-small", T=4096, bias="zero",
                                                 weights="nvfp4", **small)}
    if name.startswith("w4a4-"):  # the NVFP4 workloads with NVFP4 activations
        name = "nvfp4-" + name[len("w4a4-"):]
    return extra[name] if name in extra else mi.CONFIGS[name]


def run_profile(args):
    """Only W + K moe_forward calls of one workload (the command ncu captures)."""
    import group_limited_routing_bias_b300 as lib
    import moe_inputs as mi
    dev = torch.device("cuda", 0)
    cfg = profile_config(args.profile)
    weights = mi.make_expert_weights(cfg, device=dev)
    if cfg.weights == "nvfp4":
        packed = [mi.quantize_experts_nvfp4(w) for w in weights]
        weights = tuple(p[i] for i in range(3) for p in packed)
        torch.cuda.empty_cache()
    elif cfg.weights == "fp8":
        packed = [mi.quantize_experts_fp8(w) for w in weights]
        weights = tuple(p[0] for p in packed) + (None, None, None) + tuple(p[1] for p in packed)
        torch.cuda.empty_cache()
    a4 = (mi.A4_X_GLOBAL, mi.A4_H_GLOBAL) if args.profile.startswith("w4a4-") else None
    wl = Workload(lib, cfg, weights, dev, stages=False, a4=a4, tiled=args.tiled)
    for _ in range(args.warmup):
        wl.forward(lib)
    torch.cuda.synchronize()
    per = time_steps(lambda: wl.forward(lib), args.steps, lambda: None)
    assert lib.workspace_status(wl.ws) == 0
    print(json.dumps({"profile": args.profile, "T": cfg.T, "E": cfg.E, "steps": args.steps,
                      "tiled": args.tiled, "ms_per_step": statistics.mean(per)}))


def launches_per_forward(T: int, top_k: int) -> int:
    """Kernels one moe_forward launches: router (weight split, logits GEMM,
    top-k), dispatch (one fused kernel when T*k fits one 4096-entry chunk,
    else count/scan/scatter), row gather, the two expert GEMMs, combine."""
    dispatch = 1 if T * top_k <= 4096 else 3
    return 3 + dispatch + 1 + 2 + 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-nvfp4", action="store_true")
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--profile", choices=["decode", "prefill", "skewed", "prefill-small",
                                          "decode-small", "nvfp4-decode", "nvfp4-prefill",
                                          "nvfp4-decode-small", "nvfp4-prefill-small",
                                          "fp8-decode", "w4a4-decode", "w4a4-prefill",
                                          "w4a4-decode-small", "w4a4-prefill-small"], default=None,
                    help="run only warm-up + steps forwards of one workload (for ncu)")
    ap.add_argument("--tiled", action="store_true",
                    help="with --profile: expert weights in the tiled layout (moe_pack_*)")
    args = ap.parse_args()
    peaks = load_peaks()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, peaks)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    import group_limited_routing_bias_b300 as lib
    import moe_inputs as mi
    assert args.warmup >= 3, "at least 3 warm-up steps"

    cfg = mi.CONFIGS["decode"]
    weights = mi.make_expert_weights(cfg, device=dev)
    wl = Workload(lib, cfg, weights, dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush():
        flush_buf.fill_(1)

    for _ in range(args.warmup):
        wl.forward(lib)
    torch.cuda.synchronize()
    assert lib.workspace_status(wl.ws) == 0, "device status set during warm-up"
    graph = capture_forward(lib, wl)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    per_step = time_steps(graph.replay, args.steps, flush)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms, value = aggregate_replicas(statistics.mean(per_step), cfg.T, world, dist, dev)
    assert lib.workspace_status(wl.ws) == 0, "device status set during the timed steps"
    eager_ms = statistics.mean(time_steps(lambda: wl.forward(lib), args.steps, flush))

    if rank != 0:
        if dist is not None:
            barrier()
            dist.destroy_process_group()
        return

    # ---- stage split and the expert GEMMs' roofline (HBM-bound at decode)
    k2 = min(args.steps, 50)
    stages = stage_breakdown(lib, wl, k2, flush)
    idx = wl.idx.cpu().numpy()
    touched = int(len(np.unique(idx)))
    Tk = cfg.T * cfg.top_k
    act_bytes = Tk * cfg.H * 2 + 2 * Tk * cfg.I * 2 + Tk * cfg.H * 2  # x_perm, h (w+r), y_partial
    exp_bytes = touched * EXPERT_BYTES + act_bytes
    achieved = exp_bytes / (stages["experts"] / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": achieved / peaks["hbm"],
                "traffic": (tpe * touched if (tpe := traffic_per_touched_expert()) else None),
                "kernel": "expert GEMMs (gate/up + SwiGLU, down + routing weight): one "
                          "moe_experts_swiglu call, two launches",
                "peak_source": peaks["src"], "frac_of_8tbs_nominal": achieved / 8000.0,
                "algorithmic_bytes": exp_bytes, "touched_experts": touched}

    # ---- end to end through the C ABI with host buffers
    e2e_ms = statistics.mean(e2e_steps(lib, wl, min(args.steps, 100), flush))
    e2e = {"value": cfg.T / (e2e_ms / 1000.0), "unit": "tokens/s",
           "h2d_bytes_per_step": int(wl.x_host.numel() * 2),
           "d2h_bytes_per_step": int(wl.y_host.numel() * 2), "ms_per_step": e2e_ms}

    # ---- prefill, secondary figure (same weights: identical shapes and seeds)
    prefill = None
    if not args.no_prefill:
        del wl.x_perm, wl.y_partial
        prefill = prefill_figures(lib, mi.CONFIGS["prefill"], weights, dev, flush, peaks,
                                  args.prefill_steps)

    # ---- skewed load (max ~8x mean rows per expert), same shapes and weights
    skewed = None
    if not args.no_prefill:
        skewed = prefill_figures(lib, mi.CONFIGS["skewed"], weights, dev, flush, peaks,
                                 args.prefill_steps)

    # ---- packed experts (the decode weights packed to NVFP4 and to FP8), decode and prefill
    nvfp4 = fp8 = None
    if not args.no_nvfp4:
        packed = [mi.quantize_experts_nvfp4(w) for w in weights]
        fp4w = tuple(p[0] for p in packed) + tuple(p[1] for p in packed) + tuple(p[2] for p in packed)
        nvfp4 = packed_figures(lib, mi, "nvfp4", fp4w, FP4_EXPERT_BYTES, dev, flush, peaks,
                               tiled=True, extra_T=(1, 1024))
        nvfp4["w4a4"] = packed_figures(lib, mi, "nvfp4", fp4w, FP4_EXPERT_BYTES, dev, flush, peaks,
                                       a4=(mi.A4_X_GLOBAL, mi.A4_H_GLOBAL), extra_T=(1, 1024))
        del packed, fp4w
        torch.cuda.empty_cache()
        packed = [mi.quantize_experts_fp8(w) for w in weights]
        fp8w = tuple(p[0] for p in packed) + (None, None, None) + tuple(p[1] for p in packed)
        fp8 = packed_figures(lib, mi, "fp8", fp8w, FP8_EXPERT_BYTES, dev, flush, peaks, tiled=True,
                             extra_T=(1, 1024))
        del packed, fp8w
        torch.cuda.empty_cache()

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(wl, weights)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode: T=64 tokens, Beam MoE layer (H=5120, E=256 in 8 groups of "
                               "32, top-4 groups, top-8 experts, I=2560, routed scale 2.5), bf16",
                   "T": cfg.T, "l2": "flushed (512 MB write) before every timed step",
                   "launch": "CUDA graph of one moe_forward call, replayed per step",
                   "parallelism": f"replicas x{world}"},
        "ms_per_step_eager": eager_ms,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_forward(cfg.T, cfg.top_k) * args.steps, "stages_ms": stages, "prefill": prefill, "skewed": skewed, "nvfp4": nvfp4, "fp8": fp8,
    }
    print(json.dumps(line))
    if dist is not None:
        barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
