"""GPU parity of the auxiliary-loss-free bias update (moe_bias_update) against
the oracle, bit for bit, on the GPU's own routings; and a short balancing loop
(route, update, route again) on the skewed workload that lowers the load skew."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


def test_hand_example(lib):
    d = lib.make_dims(2, 256, 32, 8, 2, 2, 128, 2.5)
    idx = torch.tensor([[0, 2], [0, 3]], dtype=torch.int32, device=DEV)
    b0 = torch.randn(32, generator=torch.Generator().manual_seed(0)).to(DEV)
    b = b0.clone()
    g = lib.moe_bias_update(d, idx, b, 0.001, 0, 100)
    ref, g_ref = oracle.bias_update(idx.cpu().numpy(), b0.cpu().numpy(), 32, 0.001, 0, 100)
    assert g == g_ref
    np.testing.assert_array_equal(b.cpu().numpy(), ref)


def test_balancing_loop_matches_oracle_and_reduces_skew(lib):
    cfg = mi.CONFIGS["skewed"].with_T(4096)
    x, wr, b = mi.make_router_inputs(cfg)
    x, wr, bias = x.to(DEV), wr.to(DEV), b.to(DEV)
    d = lib.dims_of(cfg)
    ws = lib.alloc_workspace(d, lib.MOE_OP_ROUTE)
    idx = torch.empty(cfg.T, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.top_k, dtype=torch.float32, device=DEV)
    skew = []
    steps = 40
    for step in range(steps):
        lib.moe_route(d, x, wr, bias, idx, w, ws)
        load = np.bincount(idx.cpu().numpy().ravel(), minlength=cfg.E)
        skew.append(load.max() / load.mean())
        before = bias.cpu().numpy()
        g = lib.moe_bias_update(d, idx, bias, 0.02, step, steps)
        ref, g_ref = oracle.bias_update(idx.cpu().numpy(), before, cfg.E, 0.02, step, steps)
        assert g == g_ref
        np.testing.assert_array_equal(bias.cpu().numpy(), ref)
    assert lib.workspace_status(ws) == 0
    print(f"\nmax/mean load over the loop: {skew[0]:.2f} -> {skew[-1]:.2f}")
    assert skew[-1] < 0.5 * skew[0]
