"""Derive the bias scale of the skewed workload with the oracle's router.

The skewed workload sets the selection bias to alpha * ln(p_pi(e)), p_r ~ r^-1.1
(a Zipf law over a seeded random expert permutation), and asks for the most
loaded expert to receive about 8x the mean load (T = 16384, Beam shape).  This
script bisects alpha on that target, routing with the oracle only, and prints
the load statistics; the value it finds is stored as ``moe_inputs.SKEW_ALPHA``.

    python tests/golden/derive_skew_alpha.py [--T 16384]
"""
import argparse
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import moe_inputs as mi  # noqa: E402
import oracle  # noqa: E402


def max_over_mean(alpha, x, wr, cfg):
    b = mi.zipf_bias(cfg.E, alpha, seed=0).numpy()
    r = oracle.route(x, wr, b, cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)
    load = np.bincount(r.idx.ravel(), minlength=cfg.E)
    return load.max() / load.mean(), load


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--T", type=int, default=16384)
    ap.add_argument("--target", type=float, default=8.0)
    a = ap.parse_args()
    cfg = mi.CONFIGS["skewed"].with_T(a.T)
    x, wr, _ = mi.make_router_inputs(cfg, seed=0)
    x, wr = mi.bf16_bits(x), wr.numpy()
    lo, hi = 0.0, 0.5
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        ratio, _ = max_over_mean(mid, x, wr, cfg)
        print(f"alpha={mid:.5f} max/mean={ratio:.3f}", flush=True)
        lo, hi = (mid, hi) if ratio < a.target else (lo, mid)
    alpha = round(0.5 * (lo + hi), 4)
    ratio, load = max_over_mean(alpha, x, wr, cfg)
    print(f"SKEW_ALPHA = {alpha}  max/mean = {ratio:.3f}  min load = {load.min()}  "
          f"experts with zero load = {(load == 0).sum()}")


if __name__ == "__main__":
    main()
