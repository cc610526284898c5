"""GPU parity: every stage of the CUDA path, called through the C ABI, against
the CPU oracle on the same seeded inputs.

Bars: router logits within LOGIT_ATOL of the oracle's (asserted on every
logit); routing indices bit-exact except counted near ties (tests/parity.py);
weights within W_RTOL relative, derived there from the logit bound;
dispatch bit-exact against a stable sort; combine bit-exact against an fp32
sum in k order; outputs within max|err| <= 2e-2 * max|ref| and relative
Frobenius error <= 5e-3, on every token up to mid-size batches and, at
T = 16384, on a stratified sample that gives every touched expert compared
rows and includes the boundary rows of every expert's last tile.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity import (LOGIT_ATOL, W_RTOL, compare_routing, output_errors, reference_routing,
                    row_errors, stratified_tokens)
from parity import scale_rows as mi_scale_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


def bits(t):
    return mi.bf16_bits(t)


class Case:
    """Seeded inputs of one workload, on the GPU and as host bytes for the oracle."""

    def __init__(self, cfg, T=None, seed=0, weights=True):
        self.cfg = cfg if T is None else cfg.with_T(T)
        c = self.cfg
        x, wr, b = mi.make_router_inputs(c, seed=seed)
        self.x_h, self.wr_h, self.b_h = x, wr, b
        self.x, self.wr, self.b = x.to(DEV), wr.to(DEV), b.to(DEV)
        if weights:
            self.wg, self.wu, self.wd = mi.make_expert_weights(c, device=DEV, seed=seed)

    def oracle_route(self):
        c = self.cfg
        return oracle.route(bits(self.x_h), self.wr_h.numpy(), self.b_h.numpy(), c.n_group,
                            c.topk_group, c.top_k, c.routed_scale, details=True)

    def get_expert(self, e):
        return bits(self.wg[e]), bits(self.wu[e]), bits(self.wd[e])

    def experts(self, lib):
        return lib.Experts(self.wg, self.wu, self.wd)


def gpu_route(lib, case):
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_ROUTE)
    idx = torch.full((c.T, c.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((c.T, c.top_k), dtype=torch.float32, device=DEV)
    lib.moe_route(d, case.x, case.wr, case.b, idx, w, ws)
    assert lib.workspace_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()


def check_routing(case, orc, idx, w, max_flag_frac=0.05):
    c = case.cfg
    rep = compare_routing(orc, idx, w, c.n_group, c.topk_group, c.top_k, c.routed_scale)
    print(f"\n[{c.name} T={c.T}] routing: {rep}")
    assert rep.ok, (rep, rep.mismatch_info)
    assert rep.flagged <= max(2, max_flag_frac * c.T)
    return rep


# ------------------------------------------------------------------ router


@pytest.mark.parametrize("name,T", [("tiny", 64), ("tiny", 200), ("tiny", 1), ("decode", 64),
                                    ("decode", 333), ("skewed", 1024), ("prefill", 16384)])
def test_route(lib, name, T):
    case = Case(mi.CONFIGS[name], T=T, weights=False)
    idx, w = gpu_route(lib, case)
    check_routing(case, case.oracle_route(), idx, w)


@pytest.mark.parametrize("name,T", [("decode", 64), ("tiny", 333), ("prefill", 16384)])
def test_route_logits_within_bound(lib, name, T):
    """The fp32 logits the selection is made from (moe_route_logits) against the
    oracle's fp64 sums rounded to fp32, every logit: the measured difference
    is what bounds the routed weights' error (W_RTOL).  decode T=64 adds
    K-split partial sums; T=16384 runs one K range per tile.  The routing
    outputs equal moe_route's bit for bit."""
    case = Case(mi.CONFIGS[name], T=T, weights=False)
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_ROUTE)
    idx = torch.full((c.T, c.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((c.T, c.top_k), dtype=torch.float32, device=DEV)
    logits = torch.full((c.T, c.E), float("nan"), dtype=torch.float32, device=DEV)
    lib.moe_route_logits(d, case.x, case.wr, case.b, idx, w, logits, ws)
    assert lib.workspace_status(ws) == 0
    orc = case.oracle_route()
    got = logits.cpu().numpy().astype(np.float64)
    diff = np.abs(got - orc.logits.astype(np.float64))
    print(f"\n[{c.name} T={c.T}] max |logit - oracle| = {diff.max():.3e} "
          f"(mean {diff.mean():.2e}, max |logit| {np.abs(got).max():.2f}); bound {LOGIT_ATOL:.1e}, "
          f"weights bound {W_RTOL:.2e}")
    assert np.isfinite(got).all()
    assert diff.max() <= LOGIT_ATOL
    i2, w2 = gpu_route(lib, case)
    np.testing.assert_array_equal(idx.cpu().numpy(), i2)
    np.testing.assert_array_equal(w.cpu().numpy(), w2)
    check_routing(case, orc, i2, w2)


def test_route_all_ties_pick_lowest(lib):
    """Zero input: every logit is 0, every score ties; the lowest groups and
    experts win and every weight is 2.5 / 8."""
    c = mi.CONFIGS["decode"].with_T(5)
    case = Case(c, weights=False)
    case.x.zero_()
    case.b.zero_()
    idx, w = gpu_route(lib, case)
    assert (idx == np.arange(8)[None, :]).all()
    np.testing.assert_array_equal(w, np.float32(2.5 / 8))


# ------------------------------------------------------------------ permute


def stable_sort_reference(idx, E):
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")
    slot_of = np.empty_like(order)
    slot_of[order] = np.arange(len(flat))
    offsets = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))])
    return offsets.astype(np.int32), slot_of.astype(np.int32), order.astype(np.int32)


@pytest.mark.parametrize("T,E,k,skew", [(64, 256, 8, 0.0), (1, 256, 8, 0.0), (3000, 256, 8, 0.0),
                                        (16384, 256, 8, 2.0), (64, 32, 4, 0.0), (777, 32, 4, 1.0)])
def test_permute(lib, T, E, k, skew):
    rng = np.random.default_rng(T + E + k)
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    H = 256
    d = lib.make_dims(T, H, E, 8 if E == 256 else 8, 4 if E == 256 else 2, k, 128, 2.5)
    x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    Tk = T * k
    x_perm = torch.zeros(Tk, H, dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.zeros(Tk, dtype=torch.int32, device=DEV)
    row_src = torch.zeros(Tk, dtype=torch.int32, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_PERMUTE)
    lib.moe_permute(d, torch.from_numpy(idx).to(DEV), x, x_perm, offs, slot_of, row_src, ws)
    assert lib.workspace_status(ws) == 0
    o_ref, s_ref, r_ref = stable_sort_reference(idx, E)
    np.testing.assert_array_equal(offs.cpu().numpy(), o_ref)
    np.testing.assert_array_equal(slot_of.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(row_src.cpu().numpy(), r_ref)
    assert torch.equal(x_perm, x[torch.from_numpy(r_ref // k).long().to(DEV)])


def test_permute_flags_bad_indices(lib):
    T, E, k, H = 100, 32, 4, 128
    rng = np.random.default_rng(1)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[7, 2] = E
    idx[50, 0] = -3
    d = lib.make_dims(T, H, E, 8, 2, k, 128, 2.5)
    x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    x_perm = torch.zeros(T * k, H, dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.zeros(T * k, dtype=torch.int32, device=DEV)
    row_src = torch.zeros(T * k, dtype=torch.int32, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_PERMUTE)
    lib.moe_permute(d, torch.from_numpy(idx).to(DEV), x, x_perm, offs, slot_of, row_src, ws)
    assert lib.workspace_status(ws) == lib.MOE_DEV_BAD_INDEX
    so = slot_of.cpu().numpy()
    assert so[7 * k + 2] == -1 and so[50 * k] == -1
    assert offs.cpu().numpy()[-1] == T * k - 2


# ------------------------------------------------------------------ experts + combine


def forward(lib, case, sample=None):
    """Full moe_forward on the GPU; returns (y fp64 numpy, idx, w)."""
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(c.T, c.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(c.T, c.top_k, dtype=torch.float32, device=DEV)
    lib.moe_forward(d, case.x, case.wr, case.b, case.experts(lib), y, ws, idx, w)
    assert lib.workspace_status(ws) == 0
    return y.double().cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check_forward(lib, case, sample=None):
    """sample: None (every token), "stratified" (tests/parity.py's
    stratified_tokens over the GPU's routing) or explicit token indices."""
    c = case.cfg
    y, idx, w = forward(lib, case)
    orc = case.oracle_route()
    rep = check_routing(case, orc, idx, w)
    ridx, rw = reference_routing(orc, rep, idx, c.routed_scale)
    if isinstance(sample, str):
        tokens = stratified_tokens(idx, c.E, seed=c.T)
    else:
        tokens = np.arange(c.T) if sample is None else np.asarray(sample)
    y_ref = oracle.experts_forward(bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens)
    err = output_errors(y[tokens], y_ref)
    print(f"[{c.name} T={c.T}] output: {err} over {len(tokens)} tokens")
    assert err.ok(), err
    assert np.isfinite(y).all()
    return y, idx, w


@pytest.mark.parametrize("T", [64, 200, 1, 5, 333, 1500, 2048])
def test_forward_tiny(lib, T):
    """Tiny shape; from T = 256 (1024 token rows at top-4) the token-major expert
    GEMMs run (T = 333: ~42 rows per expert, every tile ragged)."""
    check_forward(lib, Case(mi.CONFIGS["tiny"], T=T))


def test_forward_tiny_skewed_token_major(lib):
    """Token-major path with a strongly skewed load (some experts with one or
    two tiles, some with many), every output compared."""
    c = mi.CONFIGS["tiny"].with_T(1800)
    case = Case(c)
    case.b_h = mi.zipf_bias(c.E, 0.15, seed=3)
    case.b = case.b_h.to(DEV)
    y, idx, _ = check_forward(lib, case)
    load = np.bincount(idx.ravel(), minlength=c.E)
    assert load.max() > 3 * load.mean()


def test_forward_tiny_skewed_weights_on_m(lib):
    """Weights-on-M path (T*k < 1024) with a strongly skewed load: experts of a
    few rows (half-height activation box), of up to one tile, and of several
    tiles; every output compared."""
    c = mi.CONFIGS["tiny"].with_T(200)
    case = Case(c)
    case.b_h = mi.zipf_bias(c.E, 0.15, seed=5)
    case.b = case.b_h.to(DEV)
    y, idx, _ = check_forward(lib, case)
    load = np.bincount(idx.ravel(), minlength=c.E)
    assert load.max() > 64 and (load[load > 0] <= 32).any()


def test_forward_decode_full(lib):
    """The decode workload in the launch configuration the benchmark times."""
    check_forward(lib, Case(mi.CONFIGS["decode"]))


@pytest.mark.parametrize("T", [256, 1024])
def test_forward_beam_mid_batch_sampled(lib, T):
    """Beam shape between decode and prefill: token-major tiles with a few to a
    few dozen rows per expert."""
    rng = np.random.default_rng(T)
    case = Case(mi.CONFIGS["decode"], T=T)
    check_forward(lib, case, sample=np.sort(rng.choice(T, 48, replace=False)))


def test_forward_prefill_sampled(lib):
    """T=16384, every touched expert's first row, last-tile boundary rows and
    last row compared (stratified sample)."""
    check_forward(lib, Case(mi.CONFIGS["prefill"]), sample="stratified")


def test_forward_skewed_sampled(lib):
    """Skewed load (max ~8x mean): the stratified sample adds the first and last
    row of every tile of the most-loaded expert."""
    case = Case(mi.CONFIGS["skewed"])
    y, idx, _ = check_forward(lib, case, sample="stratified")
    load = np.bincount(idx.ravel(), minlength=256)
    assert load.max() >= 6 * load.mean()


@pytest.mark.parametrize("T", [150, 2048])
def test_stages_match_forward(lib, T):
    """moe_route -> moe_permute -> moe_experts_swiglu -> moe_combine equals moe_forward
    bit for bit, and each y_partial row is its routed expert's output times its weight.
    At T=2048 moe_forward's gate/up GEMM gathers x rows itself while the staged
    calls read x_perm."""
    c = mi.CONFIGS["tiny"].with_T(T)
    case = Case(c)
    d = lib.dims_of(c)
    y_fwd, idx_fwd, w_fwd = forward(lib, case)
    Tk = c.T * c.top_k
    idx = torch.empty(c.T, c.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(c.T, c.top_k, dtype=torch.float32, device=DEV)
    lib.moe_route(d, case.x, case.wr, case.b, idx, w, lib.alloc_workspace(d, lib.MOE_OP_ROUTE))
    x_perm = torch.empty(Tk, c.H, dtype=torch.bfloat16, device=DEV)
    offs = torch.empty(c.E + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.empty(Tk, dtype=torch.int32, device=DEV)
    row_src = torch.empty(Tk, dtype=torch.int32, device=DEV)
    lib.moe_permute(d, idx, case.x, x_perm, offs, slot_of, row_src,
                    lib.alloc_workspace(d, lib.MOE_OP_PERMUTE))
    y_partial = torch.empty(Tk, c.H, dtype=torch.bfloat16, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_EXPERTS)
    lib.moe_experts_swiglu(d, case.experts(lib), x_perm, offs, row_src, w, y_partial, ws)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    lib.moe_combine(d, y_partial, slot_of, y)
    assert lib.workspace_status(ws) == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_fwd)
    np.testing.assert_array_equal(y.double().cpu().numpy(), y_fwd)
    # combine: fp32 sum in k order, one rounding to bf16
    yp = y_partial.float().cpu().numpy()
    so = slot_of.cpu().numpy().reshape(c.T, c.top_k)
    acc = np.zeros((c.T, c.H), np.float32)
    for j in range(c.top_k):
        acc += yp[so[:, j]]
    ref = torch.from_numpy(acc).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(y.double().cpu().numpy(), ref)
    # per-row expert outputs against the oracle's expert path
    xb = bits(case.x_h)
    ii, ww = idx.cpu().numpy(), w.cpu().numpy()
    rows_ref = np.zeros((c.T, c.top_k, c.H))
    for e in np.unique(ii):
        tt, kk = np.nonzero(ii == e)
        rows_ref[tt, kk] = oracle.expert_swiglu(xb[tt], *case.get_expert(int(e))) * ww[tt, kk][:, None]
    got = yp[so.ravel()].reshape(c.T, c.top_k, c.H)
    err = output_errors(got, rows_ref)
    assert err.ok(), err


@pytest.mark.parametrize("name,T", [("decode", 64), ("tiny", 2048)])
def test_forward_bf16_activation_range(lib, name, T):
    """Token rows with |x| up to 1e5 and rows of about 1e-6 keep bf16's range
    through the whole block (h of the large rows reaches ~1e10): every row
    within the bf16 bars relative to its own scale.  decode T=64 runs the
    weights-on-M GEMMs, tiny T=2048 the token-major ones."""
    case = Case(mi.CONFIGS[name], T=T)
    case.x_h = mi_scale_rows(case.x_h)
    case.x = case.x_h.to(DEV)
    c = case.cfg
    y, idx, w = forward(lib, case)
    orc = case.oracle_route()
    rep = check_routing(case, orc, idx, w, max_flag_frac=0.2)
    ridx, rw = reference_routing(orc, rep, idx, c.routed_scale)
    tokens = np.arange(16)
    y_ref = oracle.experts_forward(bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens)
    assert np.isfinite(y[tokens]).all()
    mx, fr = row_errors(y[tokens], y_ref)
    print(f"\n[{c.name} T={c.T}] rows |x|~1e5: rel-Frob {fr[:4]}; |x|~1e-6: {fr[4:8]}; "
          f"max |y| {np.abs(y_ref[:4]).max():.3g} / {np.abs(y_ref[4:8]).max():.3g}")
    assert (mx <= 2e-2).all() and (fr <= 5e-3).all(), (mx, fr)


def test_zero_down_weights_give_zero(lib):
    case = Case(mi.CONFIGS["tiny"])
    case.wd.zero_()
    y, _, _ = forward(lib, case)
    assert np.all(y == 0)


def test_empty_batch(lib):
    """T == 0 is a no-op that reads no pointer."""
    c = mi.CONFIGS["tiny"]
    d = lib.dims_of(c, T=0)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD)
    wg, wu, wd = mi.make_expert_weights(c, device=DEV)
    x = torch.empty(0, c.H, dtype=torch.bfloat16, device=DEV)
    y = torch.empty(0, c.H, dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros(c.E, c.H, device=DEV)
    b = torch.zeros(c.E, device=DEV)
    lib.moe_forward(d, x, wr, b, lib.Experts(wg, wu, wd), y, ws)
    assert lib.workspace_status(ws) == 0


# ------------------------------------------------------------------ general router shapes


@pytest.mark.parametrize("E,G,kg,k", [
    (256, 4, 2, 8),     # groups of 64: two slots per lane merged
    (256, 2, 1, 8),     # groups of 128
    (256, 1, 1, 8),     # one group of 256: plain top-k
    (256, 8, 8, 8),     # every group kept
    (64, 8, 3, 6),      # groups of 8
    (128, 16, 5, 16),   # 16 groups of 8, top_k 16
    (32, 16, 4, 3),     # groups of 2
])
def test_route_general_shapes(lib, E, G, kg, k):
    cfg = mi.MoeConfig(f"route-E{E}-G{G}", T=300, H=512, E=E, n_group=G, topk_group=kg, top_k=k,
                       I=128)
    case = Case(cfg, weights=False)
    idx, w = gpu_route(lib, case)
    check_routing(case, case.oracle_route(), idx, w)


@pytest.mark.parametrize("E,G,kg,k,H,I,T", [(64, 4, 2, 6, 384, 384, 700),
                                             (128, 8, 4, 8, 256, 640, 900)])
def test_forward_other_shapes(lib, E, G, kg, k, H, I, T):
    """Forward at shapes other than Beam's (H, I multiples of 128 only)."""
    cfg = mi.MoeConfig(f"shape-E{E}-H{H}-I{I}", T=T, H=H, E=E, n_group=G, topk_group=kg, top_k=k,
                       I=I)
    check_forward(lib, Case(cfg))
