"""GPU parity with FP8 expert weights (e4m3 codes with one fp32 scale per
output row), through the C ABI, against the oracle on the same bytes.  The
GPU dequantises exactly (e4m3 is exact in f16; the row scale multiplies the
fp32 accumulator), so the bf16 bars apply."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity import (compare_routing, output_errors, reference_routing, row_errors,
                    sample_tokens, scale_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


class Fp8Case:
    def __init__(self, cfg, T=None, seed=0, tiled=False):
        self.tiled, self._tiled_experts = tiled, None
        self.cfg = cfg if T is None else cfg.with_T(T)
        c = self.cfg
        x, wr, b = mi.make_router_inputs(c, seed=seed)
        self.x_h, self.wr_h, self.b_h = x, wr, b
        self.x, self.wr, self.b = x.to(DEV), wr.to(DEV), b.to(DEV)
        packed = [mi.quantize_experts_fp8(w) for w in mi.make_expert_weights(c, device=DEV, seed=seed)]
        (self.qg, self.rg), (self.qu, self.ru), (self.qd, self.rd) = packed
        torch.cuda.empty_cache()

    def experts(self, lib):
        ex = lib.Experts(self.qg, self.qu, self.qd, None, None, None, self.rg, self.ru, self.rd)
        if not self.tiled:
            return ex
        if self._tiled_experts is None:
            self._tiled_experts = ex.to_tiled()
        return self._tiled_experts

    def get_expert(self, e):
        M = oracle.Fp8Matrix
        return (M(self.qg[e].cpu().numpy(), self.rg[e].cpu().numpy()),
                M(self.qu[e].cpu().numpy(), self.ru[e].cpu().numpy()),
                M(self.qd[e].cpu().numpy(), self.rd[e].cpu().numpy()))


def forward(lib, case):
    c = case.cfg
    d = lib.dims_of(c)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_FP8)
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
    assert err.ok(), err
    return y


@pytest.mark.parametrize("T", [64, 1, 300, 2048])
def test_fp8_tiny(lib, T):
    """T=1 (4 rows) takes the weights-on-M GEMMs, the others the token-major ones."""
    check(lib, Fp8Case(mi.CONFIGS["tiny"], T=T))


@pytest.mark.parametrize("T,sample", [(64, None), (16384, "stratified")])
def test_fp8_beam(lib, T, sample):
    check(lib, Fp8Case(mi.CONFIGS["fp8"], T=T), sample)


@pytest.mark.parametrize("name,T,sample", [("tiny", 5, None), ("tiny", 64, None),
                                            ("tiny", 2048, None), ("fp8", 64, None),
                                            ("fp8", 16384, "stratified")])
def test_fp8_tiled(lib, name, T, sample):
    """Weights in the tiled layout (moe_pack_fp8), on both GEMM paths: parity
    with the oracle, and the row-major forward's output bit for bit."""
    case = Fp8Case(mi.CONFIGS[name], T=T)
    y_rm = check(lib, case, sample)
    case.tiled = True
    assert torch.equal(forward(lib, case)[0], y_rm)


@pytest.mark.parametrize("name,T", [("fp8", 64), ("tiny", 2), ("tiny", 2048)])
def test_fp8_bf16_activation_range(lib, name, T):
    """The three FP8 GEMM paths keep bf16's range (f16 operands scaled by a
    power of two per token row): rows with |x| up to 1e5 and of about 1e-6,
    each within the bf16 bars relative to its own scale.  fp8 T=64 runs the
    tensor-memory GEMMs, tiny T=2 (I = 128) the weights-on-M ones with the
    weights dequantised in shared memory, tiny T=2048 the token-major ones."""
    case = Fp8Case(mi.CONFIGS[name], T=T)
    n = 1 if T < 8 else 4
    case.x_h = scale_rows(case.x_h, n=n)
    case.x = case.x_h.to(DEV)
    c = case.cfg
    y, idx, w = forward(lib, case)
    orc = oracle.route(mi.bf16_bits(case.x_h), case.wr_h.numpy(), case.b_h.numpy(), c.n_group,
                       c.topk_group, c.top_k, c.routed_scale, details=True)
    rep = compare_routing(orc, idx, w, c.n_group, c.topk_group, c.top_k, c.routed_scale)
    assert rep.ok, (rep, rep.mismatch_info)
    ridx, rw = reference_routing(orc, rep, idx, c.routed_scale)
    tokens = np.arange(2 * n)
    y_ref = oracle.experts_forward(mi.bf16_bits(case.x_h), ridx, rw, case.get_expert, tokens=tokens)
    yg = y.double().cpu().numpy()[tokens]
    assert np.isfinite(yg).all()
    mx, fr = row_errors(yg, y_ref)
    print(f"\n[{c.name} T={c.T}] rows |x|~1e5: rel-Frob {fr[:n]}; |x|~1e-6: {fr[n:]}")
    assert (mx <= 2e-2).all() and (fr <= 5e-3).all(), (mx, fr)
