"""Seeded synthetic inputs for the Beam MoE block (shared by the tests, the
oracle runs and the benchmark).

This module holds no part of the block's arithmetic: it draws random tensors
with the shapes and distributions of the workloads, and (for the NVFP4
workload) packs bf16 weights into the NVFP4 storage format, which is data
preparation that happens before the layer runs.

Shapes follow the Beam pages: hidden 5,120, 256 experts in 8 groups of 32,
top 4 groups, top 8 experts, SwiGLU intermediate 2,560, routed scale 2.5
("Hugging Face releases Beam ..." third paragraph; "Reflection Releases Beam
..." section "Where Beam Saves and Where the Memory Bill Comes In").

Distributions: ``N(0, v)`` below names the *variance* v.  Token activations
x ~ N(0,1) rounded to bf16; router weight ~ N(0, 1/H) in fp32 (so logits are
~N(0,1)); selection bias ~ N(0, 0.01); W_gate, W_up ~ N(0, 1/H) and
W_down ~ N(0, 1/I) rounded to bf16.

The small tensors (x, router weight, bias) are always drawn on the CPU so the
same seed gives the same bytes on every machine; the expert weights, which
reach 20 GB at the full shape, are drawn on the requested device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int
    H: int
    E: int
    n_group: int
    topk_group: int
    top_k: int
    I: int
    routed_scale: float = 2.5
    bias: str = "normal"        # "normal" N(0, 0.01) | "zero" | "zipf"
    weights: str = "bf16"       # "bf16" | "nvfp4" | "fp8"
    zipf_alpha: float = 0.0     # scale of log(Zipf) bias for bias="zipf"

    def with_T(self, T: int) -> "MoeConfig":
        return replace(self, T=T)

    @property
    def group_size(self) -> int:
        return self.E // self.n_group


BEAM = dict(H=5120, E=256, n_group=8, topk_group=4, top_k=8, I=2560, routed_scale=2.5)

# Scale of ln(p) in the skewed workload's bias, with p_r proportional to
# r^-1.1 over a seeded random expert permutation.  It was chosen so that the
# most-loaded expert receives about 8x the mean load at T=16384 with seed 0;
# tests/golden/derive_skew_alpha.py recomputes it with the oracle's router.
SKEW_ALPHA = 0.0437

CONFIGS = {
    "tiny": MoeConfig("tiny", T=64, H=256, E=32, n_group=8, topk_group=2, top_k=4, I=128),
    "decode": MoeConfig("decode", T=64, **BEAM),
    "prefill": MoeConfig("prefill", T=16384, bias="zero", **BEAM),
    "skewed": MoeConfig("skewed", T=16384, bias="zipf", zipf_alpha=SKEW_ALPHA, **BEAM),
    "nvfp4": MoeConfig("nvfp4", T=64, weights="nvfp4", **BEAM),
    "fp8": MoeConfig("fp8", T=64, weights="fp8", **BEAM),
}
NVFP4_TOKENS = (1, 64, 1024, 16384)

# Static global scales of the W4A4 activation quantisers (the calibrated
# input scales an NVFP4 checkpoint carries): the largest magnitude each tensor's
# block scales must reach, over e4m3_max * e2m1_max = 448 * 6.  With these
# inputs x ~ N(0, 1) stays below 8 in magnitude, and h = silu(g) * u with
# g, u ~ N(0, 1) (weights ~ N(0, 1/fan_in)) below 32.
A4_X_GLOBAL = 8.0 / 2688.0
A4_H_GLOBAL = 32.0 / 2688.0


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_bias(E: int, alpha: float, seed: int, s: float = 1.1) -> torch.Tensor:
    """alpha * ln(p_pi(e)), p_r ~ r^-s normalised over r = 1..E, pi a seeded permutation."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    p = r.pow(-s)
    p = p / p.sum()
    perm = torch.randperm(E, generator=_gen(seed + 7))
    return (alpha * torch.log(p[perm])).to(torch.float32)


def make_router_inputs(cfg: MoeConfig, seed: int = 0, T: Optional[int] = None):
    """x bf16 [T,H], router weight fp32 [E,H], bias fp32 [E]; drawn on the CPU."""
    T = cfg.T if T is None else T
    x = torch.randn(T, cfg.H, generator=_gen(seed + 1)).to(torch.bfloat16)
    w_router = torch.randn(cfg.E, cfg.H, generator=_gen(seed + 2)) * (1.0 / math.sqrt(cfg.H))
    if cfg.bias == "normal":
        bias = torch.randn(cfg.E, generator=_gen(seed + 3)) * 0.1
    elif cfg.bias == "zero":
        bias = torch.zeros(cfg.E)
    elif cfg.bias == "zipf":
        bias = zipf_bias(cfg.E, cfg.zipf_alpha, seed)
    else:
        raise ValueError(cfg.bias)
    return x.contiguous(), w_router.to(torch.float32).contiguous(), bias.to(torch.float32).contiguous()


def _expert_seed(seed: int, matrix: int, e: int) -> int:
    return 1_000_003 * (seed + 1) + 4099 * matrix + e


def make_expert(cfg: MoeConfig, e: int, device="cpu", seed: int = 0):
    """bf16 (W_gate [I,H], W_up [I,H], W_down [H,I]) of expert e alone, each
    drawn from its own seeded generator on ``device``."""
    H, I = cfg.H, cfg.I
    out = []
    for j, (shape, fan_in) in enumerate((((I, H), H), ((I, H), H), ((H, I), I))):
        g = _gen(_expert_seed(seed, j, e), device)
        w = torch.randn(shape, generator=g, device=device) * (1.0 / math.sqrt(fan_in))
        out.append(w.to(torch.bfloat16))
    return tuple(out)


def make_expert_weights(cfg: MoeConfig, device="cpu", seed: int = 0):
    """bf16 W_gate [E,I,H], W_up [E,I,H], W_down [E,H,I], drawn expert by expert on ``device``
    (expert e holds the same values as ``make_expert(cfg, e, device, seed)``)."""
    E, H, I = cfg.E, cfg.H, cfg.I
    wg = torch.empty((E, I, H), dtype=torch.bfloat16, device=device)
    wu = torch.empty((E, I, H), dtype=torch.bfloat16, device=device)
    wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        wg[e], wu[e], wd[e] = make_expert(cfg, e, device, seed)
    return wg, wu, wd


# ---------------------------------------------------------------- NVFP4 packing (data preparation)

_E2M1_UP_TIES = (0.75, 1.75, 3.5)       # midpoints whose tie rounds to the even code above
_E2M1_DOWN_TIES = (0.25, 1.25, 2.5, 5.0)  # midpoints whose tie rounds to the even code below


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round to nearest E2M1 code (ties to even code), saturating at +-6; uint8 codes 0..15."""
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.uint8)
    for t in _E2M1_DOWN_TIES:
        code += (a > t).to(torch.uint8)
    for t in _E2M1_UP_TIES:
        code += (a >= t).to(torch.uint8)
    sign = (v < 0) & (code > 0)
    return code | (sign.to(torch.uint8) << 3)


def quantize_nvfp4(w: torch.Tensor):
    """Pack one weight matrix [N, K] (K contiguous) into NVFP4.

    global = amax / (448 * 6); block scale = e4m3(amax_block / (6 * global)) per 16
    elements along K; code = e2m1(w / (scale * global)).  Returns (q uint8 [N,K/2]
    with the even k in the low nibble, s uint8 [N,K/16] e4m3 bits, global fp32 scalar).
    """
    N, K = w.shape
    wf = w.to(torch.float32)
    amax = wf.abs().max()
    g = (amax / (448.0 * 6.0)).clamp_min(torch.finfo(torch.float32).tiny)
    blocks = wf.view(N, K // 16, 16)
    bmax = blocks.abs().amax(dim=-1)
    s8 = (bmax / (6.0 * g)).to(torch.float8_e4m3fn)
    s_val = s8.to(torch.float32)
    denom = (s_val * g).unsqueeze(-1)
    scaled = torch.where(denom > 0, blocks / torch.where(denom > 0, denom, torch.ones_like(denom)),
                         torch.zeros_like(blocks))
    codes = _e2m1_codes(scaled).view(N, K)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return q, s8.view(torch.uint8).contiguous(), g.to(torch.float32)


def quantize_experts_nvfp4(w: torch.Tensor):
    """Pack [E, N, K] bf16 expert weights expert by expert; returns (q [E,N,K/2], s [E,N,K/16], g fp32 [E])."""
    E, N, K = w.shape
    q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((E, N, K // 16), dtype=torch.uint8, device=w.device)
    g = torch.empty((E,), dtype=torch.float32, device=w.device)
    for e in range(E):
        q[e], s[e], g[e] = quantize_nvfp4(w[e])
    return q, s, g


# ---------------------------------------------------------------- FP8 packing (data preparation)


def quantize_fp8_rows(w: torch.Tensor):
    """One weight matrix [N, K] -> e4m3 codes uint8 [N, K] and one fp32 scale per
    row: scale = amax_row / 448, code = e4m3(w / scale) (round to nearest even)."""
    wf = w.to(torch.float32)
    amax = wf.abs().amax(dim=1).clamp_min(torch.finfo(torch.float32).tiny)
    scale = (amax / 448.0).to(torch.float32)
    q = (wf / scale[:, None]).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def quantize_experts_fp8(w: torch.Tensor):
    """[E, N, K] bf16 -> (codes uint8 [E, N, K], row scales fp32 [E, N])."""
    E, N, K = w.shape
    q = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((E, N), dtype=torch.float32, device=w.device)
    for e in range(E):
        q[e], s[e] = quantize_fp8_rows(w[e])
    return q, s


# ---------------------------------------------------------------- views


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()
