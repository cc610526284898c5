"""Pins for the oracle's router (CPU only).

Each test checks the oracle against something other than itself: a value
worked by hand from the routing rule, brute-force enumeration of subsets,
a library sort, or an invariant the rule implies.  The rule is stated on the
Beam pages ("Hugging Face releases Beam ...", third paragraph; "Reflection
Releases Beam ...", section "Where Beam Saves and Where the Memory Bill Comes
In"; "Beam 1.0" for the per-expert bias).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import moe_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_from_f32(a):
    a = np.ascontiguousarray(a, np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def _one_hot_case(logits, bias, H, hot, seed=0):
    """One token, one-hot at ``hot``: logit_e equals w_router[e, hot] exactly."""
    rng = np.random.default_rng(seed)
    E = len(logits)
    wr = rng.standard_normal((E, H)).astype(np.float32)
    wr[:, hot] = np.asarray(logits, np.float32)
    x = np.zeros((1, H), np.float32)
    x[0, hot] = 1.0
    return _bf16_bits_from_f32(x), wr, np.asarray(bias, np.float32)


def _parse_log(s):
    if s == "0":
        return 0.0
    neg = s.startswith("-")
    v = math.log(float(s.lstrip("-").replace("ln", "")))
    return -v if neg else v


# ------------------------------------------------------------------ golden, worked by hand


def test_hand_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "route_hand_example.json")))
    logits = [_parse_log(s) for s in g["logits"]]
    x, wr, b = _one_hot_case(logits, g["bias"], g["H"], g["hot_index"])
    r = oracle_mod.route(x, wr, b, g["n_group"], g["topk_group"], g["top_k"], g["routed_scale"],
                         details=True)
    assert r.idx[0].tolist() == g["expected_idx"]
    kept = [j for j in range(g["n_group"]) if r.group_kept[0, j]]
    assert kept == g["expected_kept_groups"]
    np.testing.assert_allclose(r.w[0], g["expected_w"], rtol=g["w_rel_tol"])
    # the one-hot token makes the logits equal to the router column exactly
    np.testing.assert_array_equal(r.logits[0], wr[:, g["hot_index"]])


# ------------------------------------------------------------------ brute force


def _brute_force(sb, s, n_group, topk_group, top_k, scale):
    """Enumerate subsets.  Group score = best pair sum in the group (fp32
    addition); kept groups = the topk_group-subset with the largest total
    score, ties to the lexicographically smallest index tuple; experts = the
    top_k-subset of the kept groups' experts with the largest total biased
    score, same tie rule; output order = biased score descending, then index."""
    E = len(sb)
    gsz = E // n_group
    gscore = []
    for j in range(n_group):
        mem = range(j * gsz, (j + 1) * gsz)
        gscore.append(max(float(np.float32(sb[a]) + np.float32(sb[c]))
                          for a, c in itertools.combinations(mem, 2)))
    best = None
    for sub in itertools.combinations(range(n_group), topk_group):
        key = (math.fsum(gscore[j] for j in sub), tuple(-j for j in sub))
        if best is None or key > best[0]:
            best = (key, sub)
    kept = best[1]
    cand = [e for e in range(E) if e // gsz in kept]
    best = None
    for sub in itertools.combinations(cand, top_k):
        key = (math.fsum(float(sb[e]) for e in sub), tuple(-e for e in sub))
        if best is None or key > best[0]:
            best = (key, sub)
    chosen = sorted(best[1], key=lambda e: (-float(sb[e]), e))
    sv = np.array([float(s[e]) for e in chosen])
    w = scale * sv / sv.sum()
    return chosen, sorted(kept), w


def _check_against_brute(oracle_mod, x, wr, b, G, kg, k, scale):
    r = oracle_mod.route(x, wr, b, G, kg, k, scale, details=True)
    for t in range(x.shape[0]):
        chosen, kept, w = _brute_force(r.biased[t], r.scores[t], G, kg, k, scale)
        assert r.idx[t].tolist() == chosen, t
        assert [j for j in range(G) if r.group_kept[t, j]] == kept, t
        np.testing.assert_allclose(r.w[t], w, rtol=1e-6)
    return r


def test_brute_force_tiny_config(oracle_mod):
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=0)
    _check_against_brute(oracle_mod, mi.bf16_bits(x), wr.numpy(), b.numpy(), cfg.n_group,
                         cfg.topk_group, cfg.top_k, cfg.routed_scale)


@pytest.mark.parametrize("E,G,kg,k", [(32, 8, 2, 4), (16, 4, 2, 3), (24, 3, 2, 5), (12, 6, 3, 4)])
def test_brute_force_tie_stress(oracle_mod, E, G, kg, k):
    """Logits and biases from tiny value sets, so equal scores are everywhere."""
    rng = np.random.default_rng(E * 100 + k)
    H = 8
    T = 48
    wr = rng.standard_normal((E, H)).astype(np.float32)
    xs, ws, bs = [], [], []
    for t in range(T):
        hot = t % H
        wr_t = wr.copy()
        wr_t[:, hot] = rng.choice([-1.0, 0.0, 0.5, 1.0], size=E).astype(np.float32)
        x, wr_t, bias = _one_hot_case(wr_t[:, hot], rng.choice([0.0, 0.25], size=E), H, hot)
        xs.append(x), ws.append(wr_t), bs.append(bias)
    # one token at a time, since each has its own router column values
    for x, w, bias in zip(xs, ws, bs):
        _check_against_brute(oracle_mod, x, w, bias, G, kg, k, 2.5)


def test_brute_force_beam_groups(oracle_mod):
    """At the Beam shape the kept groups are brute-forced over all 70 four-group
    subsets and all 496 pairs per group; the experts are checked against the
    separation property (every chosen score beats every unchosen candidate)."""
    cfg = mi.CONFIGS["decode"]
    x, wr, b = mi.make_router_inputs(cfg, seed=3, T=6)
    r = oracle_mod.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), cfg.n_group, cfg.topk_group,
                         cfg.top_k, cfg.routed_scale, details=True)
    gsz = cfg.group_size
    for t in range(6):
        sb = r.biased[t]
        gscore = [max(float(np.float32(sb[a]) + np.float32(sb[c]))
                      for a, c in itertools.combinations(range(j * gsz, (j + 1) * gsz), 2))
                  for j in range(cfg.n_group)]
        np.testing.assert_array_equal(r.group_score[t], np.float32(gscore))
        best = max(itertools.combinations(range(cfg.n_group), cfg.topk_group),
                   key=lambda sub: (math.fsum(gscore[j] for j in sub), tuple(-j for j in sub)))
        kept = [j for j in range(cfg.n_group) if r.group_kept[t, j]]
        assert kept == sorted(best)
        chosen = set(r.idx[t].tolist())
        cand = [e for e in range(cfg.E) if e // gsz in kept]
        assert chosen <= set(cand)
        lo = min(sb[e] for e in chosen)
        assert all(sb[e] <= lo for e in cand if e not in chosen)


# ------------------------------------------------------------------ library reductions


@pytest.mark.parametrize("G,kg", [(1, 1), (8, 8), (4, 4)])
def test_reduces_to_plain_topk(oracle_mod, G, kg):
    """With one group, or with every group kept, the router is plain top-k of
    the biased scores: a stable sort (numpy lexsort) gives the answer."""
    cfg = mi.CONFIGS["decode"]
    x, wr, b = mi.make_router_inputs(cfg, seed=5, T=32)
    r = oracle_mod.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), G, kg, 8, 2.5, details=True)
    for t in range(32):
        order = np.lexsort((np.arange(cfg.E), -r.biased[t].astype(np.float64)))
        assert r.idx[t].tolist() == order[:8].tolist()


def test_logits_match_library_matmul(oracle_mod):
    """Logits equal a float64 library matmul rounded once to fp32, and the
    sigmoid equals scipy's expit on them; transposed operands would fail here
    because H != E."""
    from scipy.special import expit
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=1)
    r = oracle_mod.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), cfg.n_group, cfg.topk_group,
                         cfg.top_k, cfg.routed_scale, details=True)
    ref = (x.double().numpy() @ wr.double().numpy().T).astype(np.float32)
    np.testing.assert_allclose(r.logits, ref, rtol=0, atol=1e-6)
    np.testing.assert_allclose(r.scores, expit(r.logits.astype(np.float64)).astype(np.float32),
                               rtol=2e-7)
    np.testing.assert_array_equal(r.biased, r.scores + b.numpy()[None, :])


# ------------------------------------------------------------------ invariants


def test_invariants_beam_shape(oracle_mod):
    cfg = mi.CONFIGS["decode"]
    x, wr, b = mi.make_router_inputs(cfg, seed=9, T=2048)
    r = oracle_mod.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), cfg.n_group, cfg.topk_group,
                         cfg.top_k, cfg.routed_scale, details=True)
    gsz = cfg.group_size
    assert r.group_kept.sum(1).tolist() == [cfg.topk_group] * 2048
    for t in range(2048):
        idx = r.idx[t]
        assert len(set(idx.tolist())) == cfg.top_k
        groups = set((idx // gsz).tolist())
        assert len(groups) <= cfg.topk_group
        assert all(r.group_kept[t, j] for j in groups)
        sb = r.biased[t, idx]
        assert np.all(sb[:-1] >= sb[1:])
    assert np.all(r.w > 0)
    np.testing.assert_allclose(r.w.astype(np.float64).sum(1), 2.5, atol=1e-6)


def test_excluded_not_zero_masked(oracle_mod):
    """With large negative biases every biased score is below zero; experts of
    dropped groups must still never be chosen (a zero mask would pick them)."""
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=2)
    b = np.full(cfg.E, -2.0, np.float32)
    r = _check_against_brute(oracle_mod, mi.bf16_bits(x), wr.numpy(), b, cfg.n_group,
                             cfg.topk_group, cfg.top_k, cfg.routed_scale)
    assert np.all(r.biased < 0)
    gsz = cfg.group_size
    for t in range(cfg.T):
        assert all(r.group_kept[t, e // gsz] for e in r.idx[t])


def test_all_equal_scores_pick_lowest_indices(oracle_mod):
    """Equal logits and zero bias: every group ties, so the lowest groups and
    the lowest experts win, and the weights are all routed_scale / k."""
    E, G, kg, k, H = 32, 8, 2, 4, 16
    x, wr, b = _one_hot_case([0.25] * E, [0.0] * E, H, 5)
    r = oracle_mod.route(x, wr, b, G, kg, k, 2.5, details=True)
    assert r.idx[0].tolist() == [0, 1, 2, 3]
    assert r.group_kept[0].tolist() == [1, 1, 0, 0, 0, 0, 0, 0]
    np.testing.assert_array_equal(r.w[0], np.float32(2.5 / 4))


def test_token_and_expert_relabeling(oracle_mod):
    """Permuting tokens permutes the routing; permuting groups as blocks and
    experts inside groups relabels the chosen experts (ties aside)."""
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=4)
    xb, wr, b = mi.bf16_bits(x), wr.numpy(), b.numpy()
    args = (cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)
    r0 = oracle_mod.route(xb, wr, b, *args)
    rng = np.random.default_rng(0)
    tp = rng.permutation(cfg.T)
    r1 = oracle_mod.route(np.ascontiguousarray(xb[tp]), wr, b, *args)
    np.testing.assert_array_equal(r1.idx, r0.idx[tp])
    np.testing.assert_array_equal(r1.w, r0.w[tp])
    gsz = cfg.group_size
    gperm = rng.permutation(cfg.n_group)
    inner = [rng.permutation(gsz) for _ in range(cfg.n_group)]
    # new expert label n holds old expert old_of[n]
    old_of = np.array([gperm[n // gsz] * gsz + inner[n // gsz][n % gsz] for n in range(cfg.E)])
    new_of = np.argsort(old_of)
    r2 = oracle_mod.route(xb, np.ascontiguousarray(wr[old_of]), np.ascontiguousarray(b[old_of]), *args)
    np.testing.assert_array_equal(r2.idx, new_of[r0.idx])
    np.testing.assert_array_equal(r2.w, r0.w)


def test_bad_arguments_rejected(oracle_mod):
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg)
    for G, kg, k in [(5, 2, 4), (8, 0, 4), (8, 9, 4), (8, 2, 9), (32, 2, 2)]:
        with pytest.raises(ValueError):
            oracle_mod.route(mi.bf16_bits(x), wr.numpy(), b.numpy(), G, kg, k, 2.5)
