"""GPU parity with NVFP4 expert weights (e2m1 codes, one e4m3 scale per 16 k,
one fp32 global per expert and matrix), through the C ABI, against the oracle
evaluated on the same packed bytes.

The GPU dequantises exactly (code * scale is exact in f16; the global scale
multiplies the fp32 accumulator), so the output error is the 16-bit rounding
of h and y_partial, as with bf16 weights: the tests hold it to the bf16 bars
(max|err| <= 2e-2 max|ref|, relative Frobenius <= 5e-3), tighter than the
3e-2 relative Frobenius allowed for this workload.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity import (NVFP4_REL_FROB, compare_routing, output_errors, reference_routing,
                    row_errors, sample_tokens, scale_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"

TINY4 = mi.MoeConfig("tiny-nvfp4", T=64, H=256, E=32, n_group=8, topk_group=2, top_k=4, I=256,
                     weights="nvfp4")


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


class Fp4Case:
    def __init__(self, cfg, T=None, seed=0, tiled=False):
        self.tiled, self._tiled_experts = tiled, None
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

    def experts(self, lib):
        ex = lib.Experts(self.qg, self.qu, self.qd, self.sg, self.su, self.sd, self.gg, self.gu,
                         self.gd)
        if not self.tiled:
            return ex
        if self._tiled_experts is None:
            self._tiled_experts = ex.to_tiled()
        return self._tiled_experts

    def get_expert(self, e):
        M = oracle.Nvfp4Matrix
        return (M(self.qg[e].cpu().numpy(), self.sg[e].cpu().numpy(), float(self.gg[e])),
                M(self.qu[e].cpu().numpy(), self.su[e].cpu().numpy(), float(self.gu[e])),
                M(self.qd[e].cpu().numpy(), self.sd[e].cpu().numpy(), float(self.gd[e])))


def forward(lib, case):
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_NVFP4)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(c.T, c.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(c.T, c.top_k, dtype=torch.float32, device=DEV)
    lib.moe_forward(d, case.x, case.wr, case.b, case.experts(lib), y, ws, idx, w)
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
    y_ref = oracle.experts_forward(mi.bf16_bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens)
    err = output_errors(y.double().cpu().numpy()[tokens], y_ref)
    print(f"\n[{c.name} T={c.T}] routing {rep}; output {err} over {len(tokens)} tokens")
    assert err.rel_frob <= NVFP4_REL_FROB
    assert err.ok(), err
    return y


@pytest.mark.parametrize("T", [64, 200, 1, 2048])
def test_nvfp4_tiny(lib, T):
    """T=1 (4 rows) takes the weights-on-M GEMMs, the others the token-major ones."""
    check(lib, Fp4Case(TINY4, T=T))


@pytest.mark.parametrize("T,sample", [(1, None), (64, None), (1024, "stratified"),
                                      (16384, "stratified")])
def test_nvfp4_beam(lib, T, sample):
    """The four batch sizes of the NVFP4 workload; from T=1024 every touched
    expert's first row, last-tile boundary rows and last row are compared."""
    check(lib, Fp4Case(mi.CONFIGS["nvfp4"], T=T), sample)


@pytest.mark.parametrize("name,T", [("nvfp4", 64), ("tiny-nvfp4", 2048)])
def test_nvfp4_bf16_activation_range(lib, name, T):
    """Both packed-weight paths keep bf16's range (f16 operands scaled by a
    power of two per token row): token rows with |x| up to 1e5 (h ~ 1e10) and
    rows of about 1e-6, every row within the bf16 bars relative to its own
    scale.  The NVFP4 workload at T=64 runs the GEMMs with the weights
    dequantised into tensor memory, the tiny shape at T=2048 the token-major
    ones."""
    case = Fp4Case(mi.CONFIGS["nvfp4"] if name == "nvfp4" else TINY4, T=T)
    case.x_h = scale_rows(case.x_h)
    case.x = case.x_h.to(DEV)
    c = case.cfg
    y, idx, w = forward(lib, case)
    orc = oracle.route(mi.bf16_bits(case.x_h), case.wr_h.numpy(), case.b_h.numpy(), c.n_group,
                       c.topk_group, c.top_k, c.routed_scale, details=True)
    rep = compare_routing(orc, idx, w, c.n_group, c.topk_group, c.top_k, c.routed_scale)
    assert rep.ok, (rep, rep.mismatch_info)
    ridx, rw = reference_routing(orc, rep, idx, c.routed_scale)
    tokens = np.arange(16)
    y_ref = oracle.experts_forward(mi.bf16_bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens)
    yg = y.double().cpu().numpy()[tokens]
    assert np.isfinite(yg).all()
    mx, fr = row_errors(yg, y_ref)
    print(f"\n[{c.name} T={c.T}] rows |x|~1e5: rel-Frob {fr[:4]}; |x|~1e-6: {fr[4:8]}")
    assert (mx <= 2e-2).all() and (fr <= 5e-3).all(), (mx, fr)


@pytest.mark.parametrize("T", [5, 64, 2048])
def test_nvfp4_tiny_tiled(lib, T):
    """Weights in the tiled layout (moe_pack_nvfp4), on both GEMM paths: parity
    with the oracle, and the row-major forward's output bit for bit."""
    case = Fp4Case(TINY4, T=T)
    y_rm = check(lib, case)
    case.tiled = True
    assert torch.equal(check(lib, case), y_rm)


@pytest.mark.parametrize("T", [1, 64, 16384])
def test_nvfp4_beam_tiled(lib, T):
    """Tiled weights give the row-major forward's output bit for bit (the
    row-major output itself is held to the oracle by test_nvfp4_beam)."""
    case = Fp4Case(mi.CONFIGS["nvfp4"], T=T)
    y_rm, idx_rm, _ = forward(lib, case)
    case.tiled = True
    y_t, idx_t, _ = forward(lib, case)
    np.testing.assert_array_equal(idx_t, idx_rm)
    assert torch.equal(y_t, y_rm)


@pytest.mark.parametrize("tiled", [False, True])
def test_nvfp4_experts_entry_point_matches_forward(lib, tiled):
    """moe_experts_swiglu with NVFP4 weights (bf16 x_perm converted inside)
    gives the same y as moe_forward, bit for bit."""
    c = TINY4.with_T(300)
    case = Fp4Case(c, tiled=tiled)
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
    ws = lib.alloc_workspace(d, lib.MOE_OP_EXPERTS, lib.MOE_W_NVFP4)
    lib.moe_experts_swiglu(d, case.experts(lib), x_perm, offs, row_src, w, y_partial, ws)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    lib.moe_combine(d, y_partial, slot_of, y)
    assert lib.workspace_status(ws) == 0
    assert torch.equal(y, y_fwd)


def test_nvfp4_rejects_unsupported_shape(lib):
    """NVFP4 needs H and I multiples of 256 (a scale box spans 256 k)."""
    c = mi.CONFIGS["tiny"]  # I = 128
    case = Fp4Case(TINY4)
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_NVFP4)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    ex = lib.Experts(case.qg[:, :128].contiguous(), case.qu[:, :128].contiguous(),
                     case.qd[:, :, :64].contiguous(), case.sg[:, :128].contiguous(),
                     case.su[:, :128].contiguous(), case.sd[:, :, :8].contiguous(), case.gg, case.gu,
                     case.gd)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_forward(d, case.x, case.wr, case.b, ex, y, ws)
    assert e.value.status == 2
