"""GPU parity of the W4A4 path (NVFP4 weights and NVFP4 activations) through
the C ABI, against the oracle's W4A4 expert on the same packed weights and
the same activation global scales.

The activation quantiser decides codes in fp32 on both sides with the same
operations, so quantising x is compared bit for bit.  h is quantised from
the GPU's fp32 h, which differs from the oracle's fp32(h) in its last bits
(summation order, the SiLU's exp), so a code can differ where h sits on a
rounding boundary; the output is held to the bf16 bars (max|err| <= 2e-2
max|ref|, relative Frobenius <= 5e-3), far inside the 3e-2 allowed for NVFP4.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity import (NVFP4_REL_FROB, compare_routing, output_errors, reference_routing,
                    sample_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda"

TINY4 = mi.MoeConfig("tiny-nvfp4", T=64, H=256, E=32, n_group=8, topk_group=2, top_k=4, I=256,
                     weights="nvfp4")
A4 = (mi.A4_X_GLOBAL, mi.A4_H_GLOBAL)


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


class A4Case:
    def __init__(self, cfg, T=None, seed=0):
        self.cfg = cfg if T is None else cfg.with_T(T)
        c = self.cfg
        x, wr, b = mi.make_router_inputs(c, seed=seed)
        self.x_h, self.wr_h, self.b_h = x, wr, b
        self.x, self.wr, self.b = x.to(DEV), wr.to(DEV), b.to(DEV)
        packed = []
        for w in mi.make_expert_weights(c, device=DEV, seed=seed):
            packed.append(mi.quantize_experts_nvfp4(w))
            del w
        (self.qg, self.sg, self.gg), (self.qu, self.su, self.gu), (self.qd, self.sd, self.gd) = packed
        torch.cuda.empty_cache()

    def experts(self, lib, a4=A4):
        return lib.Experts(self.qg, self.qu, self.qd, self.sg, self.su, self.sd, self.gg, self.gu,
                           self.gd, a4=a4)

    def get_expert(self, e):
        M = oracle.Nvfp4Matrix
        return (M(self.qg[e].cpu().numpy(), self.sg[e].cpu().numpy(), float(self.gg[e])),
                M(self.qu[e].cpu().numpy(), self.su[e].cpu().numpy(), float(self.gu[e])),
                M(self.qd[e].cpu().numpy(), self.sd[e].cpu().numpy(), float(self.gd[e])))


def forward(lib, case, a4=A4):
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_NVFP4_A4)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(c.T, c.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(c.T, c.top_k, dtype=torch.float32, device=DEV)
    lib.moe_forward(d, case.x, case.wr, case.b, case.experts(lib, a4), y, ws, idx, w)
    assert lib.workspace_status(ws) == 0
    return y, idx.cpu().numpy(), w.cpu().numpy()


def check(lib, case, sample=None):
    c = case.cfg
    y, idx, w = forward(lib, case)
    orc = oracle.route(mi.bf16_bits(case.x_h), case.wr_h.numpy(), case.b_h.numpy(), c.n_group,
                       c.topk_group, c.top_k, c.routed_scale, details=True)
    rep = compare_routing(orc, idx, w, c.n_group, c.topk_group, c.top_k, c.routed_scale)
    assert rep.ok, (rep, rep.mismatch_info)
    ridx, rw = reference_routing(orc, rep, idx, c.routed_scale)
    tokens = sample_tokens(sample, idx, c.E)
    y_ref = oracle.experts_forward(mi.bf16_bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens,
                                   a4=A4)
    err = output_errors(y.double().cpu().numpy()[tokens], y_ref)
    print(f"\n[{c.name} W4A4 T={c.T}] routing {rep}; output {err} over {len(tokens)} tokens")
    assert err.rel_frob <= NVFP4_REL_FROB
    assert err.ok(), err
    return y


# ------------------------------------------------------------------ quantiser


@pytest.mark.parametrize("rows,cols,g", [(1, 16, 0.01), (37, 256, mi.A4_X_GLOBAL),
                                         (1000, 5120, mi.A4_X_GLOBAL), (333, 2560, 0.0371)])
def test_quantize_matches_oracle_bit_for_bit(lib, rows, cols, g):
    gen = torch.Generator().manual_seed(rows + cols)
    x = (torch.randn(rows, cols, generator=gen) * 2).to(torch.bfloat16)
    if rows > 2:
        x[1, :16] = 0.0                      # all-zero block: scale 0, codes 0
        x[2, 16:32] *= 1e-4                  # tiny block: subnormal or zero scale
        x[0, :cols:7] = -0.0                 # signed zeros
        x[2, 0] = 3e4                        # beyond 6 * 448 * g: saturated scale and codes
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, cols // 16, dtype=torch.uint8, device=DEV)
    lib.moe_quantize_nvfp4(x.to(DEV), g, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_nvfp4(x.float().numpy(), g)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


def test_quantize_rejects_bad_arguments(lib):
    x = torch.zeros(4, 24, dtype=torch.bfloat16, device=DEV)  # cols % 16 != 0
    q = torch.empty(4, 12, dtype=torch.uint8, device=DEV)
    s = torch.empty(4, 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_quantize_nvfp4(x, 0.01, q, s)
    assert e.value.status == 1
    x = torch.zeros(4, 32, dtype=torch.bfloat16, device=DEV)
    q = torch.empty(4, 16, dtype=torch.uint8, device=DEV)
    s = torch.empty(4, 2, dtype=torch.uint8, device=DEV)
    for g in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(lib.MoeError):
            lib.moe_quantize_nvfp4(x, g, q, s)


# ------------------------------------------------------------------ the W4A4 forward


@pytest.mark.parametrize("T", [1, 64, 200, 2048])
def test_w4a4_tiny(lib, T):
    """T=2048 gives 256 rows per expert: two token tiles per expert and a ragged tail."""
    check(lib, A4Case(TINY4, T=T))


@pytest.mark.parametrize("T,sample", [(1, None), (64, None), (1024, "stratified"),
                                      (16384, "stratified")])
def test_w4a4_beam(lib, T, sample):
    """The four batch sizes of the NVFP4 workload with NVFP4 activations; from
    T=1024 every touched expert's first row, last-tile boundary rows and last
    row are compared."""
    check(lib, A4Case(mi.CONFIGS["nvfp4"], T=T), sample)


def test_w4a4_experts_entry_point_matches_forward(lib):
    """moe_experts_swiglu in W4A4 mode (quantising the caller's bf16 x_perm)
    gives the same y as moe_forward, bit for bit."""
    c = TINY4.with_T(300)
    case = A4Case(c)
    d = lib.dims_of(c)
    y_fwd, _, _ = forward(lib, case)
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
    ws = lib.alloc_workspace(d, lib.MOE_OP_EXPERTS, lib.MOE_W_NVFP4_A4)
    lib.moe_experts_swiglu(d, case.experts(lib), x_perm, offs, row_src, w, y_partial, ws)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    lib.moe_combine(d, y_partial, slot_of, y)
    assert lib.workspace_status(ws) == 0
    assert torch.equal(y, y_fwd)


def test_w4a4_rejects_bad_globals(lib):
    case = A4Case(TINY4)
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_NVFP4_A4)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    for a4 in ((0.0, 0.01), (0.01, -1.0), (float("nan"), 0.01), (0.01, float("inf"))):
        with pytest.raises(lib.MoeError) as e:
            lib.moe_forward(d, case.x, case.wr, case.b, case.experts(lib, a4), y, ws)
        assert e.value.status == 1


def test_w4a4_tiny_skewed(lib):
    """Strongly skewed load on the W4A4 path: experts with one tile, experts with
    many, every output compared."""
    case = A4Case(TINY4, T=1800)
    case.b_h = mi.zipf_bias(TINY4.E, 0.15, seed=3)
    case.b = case.b_h.to(DEV)
    check(lib, case)
    _, idx, _ = forward(lib, case)
    load = np.bincount(idx.ravel(), minlength=TINY4.E)
    assert load.max() > 3 * load.mean()


def test_w4a4_beam_skewed_sampled(lib):
    """The skewed Beam workload (max load ~8x mean) packed to NVFP4, W4A4."""
    base = mi.CONFIGS["skewed"]
    cfg = mi.MoeConfig("skewed-w4a4", T=base.T, H=base.H, E=base.E, n_group=base.n_group,
                       topk_group=base.topk_group, top_k=base.top_k, I=base.I,
                       routed_scale=base.routed_scale, bias=base.bias, weights="nvfp4",
                       zipf_alpha=base.zipf_alpha)
    case = A4Case(cfg)
    check(lib, case, "stratified")
    _, idx, _ = forward(lib, case)
    load = np.bincount(idx.ravel(), minlength=cfg.E)
    assert load.max() >= 6 * load.mean()


def test_w4a4_other_dims(lib):
    """A non-Beam shape: 64 experts in 8 groups of 8, keep 3, top 6, H=512, I=768."""
    cfg = mi.MoeConfig("w4a4-dims", T=300, H=512, E=64, n_group=8, topk_group=3, top_k=6, I=768,
                       weights="nvfp4")
    check(lib, A4Case(cfg))


def test_w4a4_staged_drops_bad_indices(lib):
    """Out-of-range expert indices are dropped by the dispatch (status bit set);
    the W4A4 experts then run on the remaining rows only."""
    c = TINY4.with_T(96)
    case = A4Case(c)
    d = lib.dims_of(c)
    Tk = c.T * c.top_k
    idx = torch.empty(c.T, c.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(c.T, c.top_k, dtype=torch.float32, device=DEV)
    lib.moe_route(d, case.x, case.wr, case.b, idx, w, lib.alloc_workspace(d, lib.MOE_OP_ROUTE))
    bad = idx.clone()
    bad[5, 1] = c.E + 3
    bad[40, 0] = -1
    x_perm = torch.zeros(Tk, c.H, dtype=torch.bfloat16, device=DEV)
    offs = torch.empty(c.E + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.empty(Tk, dtype=torch.int32, device=DEV)
    row_src = torch.empty(Tk, dtype=torch.int32, device=DEV)
    ws_p = lib.alloc_workspace(d, lib.MOE_OP_PERMUTE)
    lib.moe_permute(d, bad, case.x, x_perm, offs, slot_of, row_src, ws_p)
    assert lib.workspace_status(ws_p) == lib.MOE_DEV_BAD_INDEX
    assert int(offs[-1]) == Tk - 2
    y_partial = torch.zeros(Tk, c.H, dtype=torch.bfloat16, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_EXPERTS, lib.MOE_W_NVFP4_A4)
    lib.moe_experts_swiglu(d, case.experts(lib), x_perm, offs, row_src, w, y_partial, ws)
    assert lib.workspace_status(ws) == 0
    # every kept row equals the oracle's W4A4 expert output times its weight
    rs = row_src.cpu().numpy()[: Tk - 2]
    ent_t, ent_k = rs // c.top_k, rs % c.top_k
    bad_np = bad.cpu().numpy()
    w_np = w.cpu().numpy()
    xb = mi.bf16_bits(case.x_h)
    o = np.zeros((Tk - 2, c.H))
    for e in np.unique(bad_np[ent_t, ent_k]):
        rows = np.nonzero(bad_np[ent_t, ent_k] == e)[0]
        o[rows] = oracle.expert_swiglu_w4a4(xb[ent_t[rows]], *case.get_expert(int(e)), *A4)
    ref = o * w_np[ent_t, ent_k][:, None]
    got = y_partial.double().cpu().numpy()[: Tk - 2]
    err = output_errors(got, ref)
    assert err.ok(), err
