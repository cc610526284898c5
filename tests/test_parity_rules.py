"""The near-tie rule of the GPU parity tests, checked on the CPU with
oracle routings and hand-made alternative answers."""
import numpy as np

import moe_inputs as mi
import oracle
from parity import allowed_selections, compare_routing, gpu_choice_valid


def _one_token(group_scores_tie=False):
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=11, T=256)
    return cfg, oracle.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), cfg.n_group, cfg.topk_group,
                             cfg.top_k, cfg.routed_scale, details=True)


def test_oracle_answer_is_always_valid():
    cfg, r = _one_token()
    for t in range(r.idx.shape[0]):
        assert gpu_choice_valid(r, t, r.idx[t], cfg.n_group, cfg.topk_group, cfg.top_k)


def test_wrong_answers_are_rejected():
    cfg, r = _one_token()
    t = 0
    g = r.idx[t].copy()
    # swap the order of the first two experts (a real order error)
    bad = g.copy(); bad[[0, 1]] = bad[[1, 0]]
    if r.biased[t, g[0]] - r.biased[t, g[1]] > 1e-5:
        assert not gpu_choice_valid(r, t, bad, cfg.n_group, cfg.topk_group, cfg.top_k)
    # replace the last expert with one outside the kept groups
    gsz = cfg.group_size
    outside = next(e for e in range(cfg.E) if not r.group_kept[t, e // gsz])
    bad = g.copy(); bad[-1] = outside
    assert not gpu_choice_valid(r, t, bad, cfg.n_group, cfg.topk_group, cfg.top_k)
    # a duplicate expert
    bad = g.copy(); bad[-1] = bad[0]
    assert not gpu_choice_valid(r, t, bad, cfg.n_group, cfg.topk_group, cfg.top_k)
    rep = compare_routing(r, np.where(np.arange(r.idx.shape[0])[:, None] == t, bad, r.idx), r.w,
                          cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)
    assert rep.mismatched == 1 and not rep.ok


def test_group_tie_allows_either_group():
    """Force two groups to tie at the boundary: both kept-group sets are allowed."""
    cfg, r = _one_token()
    t = 3
    gs = r.group_score[t].astype(np.float64)
    order = sorted(range(cfg.n_group), key=lambda j: (-gs[j], j))
    a, b = order[cfg.topk_group - 1], order[cfg.topk_group]
    r.group_score[t, b] = np.float32(gs[a] - 1e-7)
    alts = allowed_selections(r, t, cfg.n_group, cfg.topk_group, cfg.top_k)
    assert len(alts) == 2
    for kept, sel in alts:
        assert gpu_choice_valid(r, t, np.array(sel), cfg.n_group, cfg.topk_group, cfg.top_k)
