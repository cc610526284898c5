"""Parity helpers shared by the GPU tests and the benchmark: routing comparison
with near-tie accounting, and the output error norms.

Rule for routing: expert indices must match the oracle exactly, except for
tokens where the oracle's decision is a near tie: the gap between the
kept/dropped groups (topk_group-th vs next group score) or between any two
neighbours among the top_k + 1 best candidate biased scores is below 1e-5.
Such tokens are counted.  For each, the GPU's answer must still be valid: it
must equal, position by position within 1e-5 of biased score, the top_k of one
of the kept-group sets that the near ties allow (groups scoring above the
boundary are kept; among those within 1e-5 of it, every choice of the
remaining count is tried).  The reference output of such a token is then
computed with the GPU's indices (weights from the oracle's unbiased scores).
"""
from __future__ import annotations

import itertools

from dataclasses import dataclass, field

import numpy as np

TIE_EPS = 1e-5

# Router logits.  The GPU sums each logit's 3 * H exact products (bf16 x times
# the three exact bf16 parts of the fp32 router weight) on the tensor cores in
# chunks of 32 MMAs, and adds the chunks in fp32 with round-to-nearest; the
# oracle sums in fp64 and rounds once to fp32.  LOGIT_ATOL bounds
# |GPU logit - oracle logit|; it is asserted directly on the logits
# moe_route_logits returns (tests/test_gpu_parity.py: all 4.2 M logits of the
# T = 16384 workload, the K-split decode batch and a ragged tiny batch).  The
# largest difference measured on B300 is LOGIT_MEASURED (T = 16384; 1.9e-6 at
# decode); the bar is about twice that.  (Accumulating the whole K range of
# 960 MMAs in one tensor-core accumulator gave 1.2e-4: its fp32 accumulation
# does not round to nearest at every step.)
LOGIT_MEASURED = 4.3e-6
LOGIT_ATOL = 1e-5

# Routed weights w_j = r s_j / sum_i s_i with s = sigmoid(logit).  A logit
# error d moves ln s by (1 - s) d, at most d, so ln w_j moves by at most
# 2 max|d| (d ln s_j minus d ln sum s, each at most max|d|).  fp32 rounding
# adds, relative: the GPU's sigmoid (expf within 2 ulp, the add and the IEEE
# division: 3 ulp), the sum of 8 scores (7 roundings), the product and the
# division (2), and the oracle's own rounding of s and w (2); with ulp = 2^-23
# that is about 1.5e-6.  Any reading error (weights from biased scores, a
# missing 2.5, a dropped expert) moves weights by whole percents.
W_ROUND = 1.5e-6
W_RTOL = 2 * LOGIT_ATOL + W_ROUND
BF16_MAX_ERR = 2e-2      # max |err| <= 2e-2 * max |ref|
BF16_REL_FROB = 5e-3     # ||err|| <= 5e-3 * ||ref||
NVFP4_REL_FROB = 3e-2


@dataclass
class RoutingReport:
    tokens: int
    flagged: int
    flagged_differing: int
    mismatched: int                      # unflagged tokens whose indices differ
    weight_max_rel: float
    use_gpu: np.ndarray = field(repr=False)  # bool [T]: reference uses the GPU's indices
    mismatch_info: list = field(default_factory=list)  # details of up to 4 mismatched tokens

    @property
    def ok(self) -> bool:
        return self.mismatched == 0 and self.weight_max_rel <= W_RTOL


def near_tie_mask(orc, n_group, topk_group, top_k, eps=TIE_EPS) -> np.ndarray:
    T, E = orc.biased.shape
    gsz = E // n_group
    gs = -np.sort(-orc.group_score.astype(np.float64), axis=1)
    group_gap = (gs[:, topk_group - 1] - gs[:, topk_group]) if topk_group < n_group \
        else np.full(T, np.inf)
    kept_e = np.repeat(orc.group_kept.astype(bool), gsz, axis=1)
    cand = np.where(kept_e, orc.biased.astype(np.float64), -np.inf)
    top = -np.sort(-cand, axis=1)[:, :top_k + 1]
    gaps = top[:, :-1] - top[:, 1:]
    gaps = np.where(np.isfinite(gaps), gaps, np.inf)
    return np.minimum(group_gap, gaps.min(axis=1)) < eps


def allowed_selections(orc, t, n_group, topk_group, top_k, eps=TIE_EPS):
    """Every top_k selection (experts ordered by biased score, then index) that
    some eps-perturbation of the oracle's group scores could produce."""
    E = orc.biased.shape[1]
    gsz = E // n_group
    gs = orc.group_score[t].astype(np.float64)
    order = sorted(range(n_group), key=lambda j: (-gs[j], j))
    thr = gs[order[topk_group - 1]]
    forced = [j for j in range(n_group) if gs[j] > thr + eps]
    tie = [j for j in range(n_group) if abs(gs[j] - thr) <= eps]
    sb = orc.biased[t].astype(np.float64)
    out = []
    for extra in itertools.combinations(tie, topk_group - len(forced)):
        kept = set(forced) | set(extra)
        cand = [e for e in range(E) if e // gsz in kept]
        out.append((kept, sorted(cand, key=lambda e: (-sb[e], e))[:top_k]))
    return out


def gpu_choice_valid(orc, t, g, n_group, topk_group, top_k, eps=TIE_EPS) -> bool:
    E = orc.biased.shape[1]
    gsz = E // n_group
    g = [int(e) for e in g]
    if len(set(g)) != top_k or any(e < 0 or e >= E for e in g):
        return False
    sb = orc.biased[t].astype(np.float64)
    if any(sb[g[i]] < sb[g[i + 1]] - eps for i in range(top_k - 1)):
        return False  # not in descending order
    for kept, sel in allowed_selections(orc, t, n_group, topk_group, top_k, eps):
        if all(e // gsz in kept for e in g) and \
                all(abs(sb[a] - sb[b]) <= eps for a, b in zip(g, sel)):
            return True
    return False


def compare_routing(orc, gpu_idx, gpu_w, n_group, topk_group, top_k, routed_scale) -> RoutingReport:
    gpu_idx = np.asarray(gpu_idx)
    gpu_w = np.asarray(gpu_w)
    T, E = orc.biased.shape
    flagged = near_tie_mask(orc, n_group, topk_group, top_k)
    same = np.all(gpu_idx == orc.idx, axis=1)
    mismatched = int(np.sum(~same & ~flagged))
    use_gpu = ~same & flagged
    info = []

    def describe(t):
        g = gpu_idx[t]
        valid = np.all((g >= 0) & (g < E))
        gs = np.sort(orc.group_score[t].astype(np.float64))[::-1]
        return dict(t=int(t), flagged=bool(flagged[t]), oracle=orc.idx[t].tolist(), gpu=g.tolist(),
                    oracle_biased=orc.biased[t, orc.idx[t]].tolist(),
                    gpu_biased=orc.biased[t, g].tolist() if valid else None,
                    group_scores_sorted=gs.tolist())

    for t in np.nonzero(~same & ~flagged)[0][:4]:
        info.append(describe(t))
    for t in np.nonzero(use_gpu)[0]:
        if not gpu_choice_valid(orc, t, gpu_idx[t], n_group, topk_group, top_k):
            mismatched += 1
            use_gpu[t] = False
            if len(info) < 4:
                info.append(describe(t))
    # weights: against the oracle's unbiased scores for whichever indices are used
    ref_w = orc.w.astype(np.float64).copy()
    for t in np.nonzero(use_gpu)[0]:
        s = orc.scores[t, gpu_idx[t]].astype(np.float64)
        ref_w[t] = routed_scale * s / s.sum()
    good = same | use_gpu
    rel = np.abs(gpu_w.astype(np.float64) - ref_w) / np.abs(ref_w)
    wmax = float(rel[good].max()) if good.any() else 0.0
    return RoutingReport(T, int(flagged.sum()), int(use_gpu.sum()), mismatched, wmax, use_gpu, info)


def reference_routing(orc, report: RoutingReport, gpu_idx, routed_scale):
    """Indices and weights the reference output is computed with."""
    idx = orc.idx.copy()
    w = orc.w.copy()
    for t in np.nonzero(report.use_gpu)[0]:
        idx[t] = gpu_idx[t]
        s = orc.scores[t, gpu_idx[t]].astype(np.float64)
        w[t] = (routed_scale * s / s.sum()).astype(np.float32)
    return idx, w


@dataclass
class OutputErrors:
    max_abs: float
    ref_max: float
    rel_frob: float

    def ok(self, max_rel=BF16_MAX_ERR, frob=BF16_REL_FROB) -> bool:
        return self.max_abs <= max_rel * self.ref_max and self.rel_frob <= frob


def output_errors(y_gpu, y_ref) -> OutputErrors:
    a = np.asarray(y_gpu, np.float64)
    b = np.asarray(y_ref, np.float64)
    err = a - b
    return OutputErrors(float(np.abs(err).max()), float(np.abs(b).max()),
                        float(np.linalg.norm(err) / np.linalg.norm(b)))


def stratified_tokens(idx, E: int, tile_rows: int = 128, n_random: int = 32, seed: int = 0):
    """Tokens whose outputs a sampled parity check compares, at sizes where the
    oracle cannot evaluate every token.  Built from the routing the GPU used
    (idx int32 [T, k], all in [0, E)) and the dispatch's stable order (rows
    expert-major, entries t*k + j ascending inside an expert):
      - for every touched expert, the tokens of its first permuted row, of the
        first row of its last tile of tile_rows rows, and of its last row (the
        boundary rows of every expert's ragged final tile);
      - for the most-loaded expert, the first and last row of every tile;
      - n_random more tokens drawn with the seed.
    Every touched expert thus contributes to at least one compared output."""
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")  # permuted row -> entry
    counts = np.bincount(flat, minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)])
    rows = []
    for e in np.nonzero(counts)[0]:
        n, o = int(counts[e]), int(offs[e])
        rows += [o, o + (n - 1) // tile_rows * tile_rows, o + n - 1]
    heavy = int(np.argmax(counts))
    for r0 in range(0, int(counts[heavy]), tile_rows):
        rows += [offs[heavy] + r0, offs[heavy] + min(r0 + tile_rows, int(counts[heavy])) - 1]
    toks = set((order[np.asarray(rows, np.int64)] // k).tolist())
    rng = np.random.default_rng(seed)
    toks |= set(rng.choice(T, min(n_random, T), replace=False).tolist())
    out = np.array(sorted(toks), dtype=np.int64)
    assert set(np.unique(idx[out])) == set(np.unique(flat)), "a touched expert has no sampled row"
    return out


def sample_tokens(sample, idx, E: int):
    """Tokens a parity check compares: every token (sample None), the
    stratified sample over the GPU's routing (sample "stratified"), or the
    given indices."""
    T = np.asarray(idx).shape[0]
    if sample is None:
        return np.arange(T)
    if isinstance(sample, str):
        assert sample == "stratified"
        return stratified_tokens(idx, E, seed=T)
    return np.asarray(sample)


def row_errors(y_gpu, y_ref):
    """Per token row: (max|err| / max|ref|, ||err|| / ||ref||).  For batches
    whose rows differ in scale by many orders of magnitude, where the norms
    over the whole batch would only see the largest rows."""
    a = np.asarray(y_gpu, np.float64)
    b = np.asarray(y_ref, np.float64)
    err = np.abs(a - b)
    ref_max = np.abs(b).max(axis=1)
    return (err.max(axis=1) / ref_max,
            np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1))


def scale_rows(x: "torch.Tensor", big: float = 1e5, tiny: float = 1e-6, n: int = 4):
    """x bf16 [T, H] with rows 0..n-1 scaled so their largest |value| is about
    `big`, rows n..2n-1 scaled to about `tiny` (values far outside f16's
    range, and deep in its subnormals); the rest unchanged."""
    import torch
    y = x.float().clone()
    for r in range(n):
        y[r] *= big / y[r].abs().max()
        y[n + r] *= tiny / y[n + r].abs().max()
    return y.to(torch.bfloat16)
