"""Checks of the seeded input generators and the NVFP4 packing used as data
preparation for the NVFP4 workload (CPU only)."""
import numpy as np
import torch

import moe_inputs as mi


def test_router_inputs_are_seeded_and_shaped():
    cfg = mi.CONFIGS["tiny"]
    a = mi.make_router_inputs(cfg, seed=0)
    b = mi.make_router_inputs(cfg, seed=0)
    c = mi.make_router_inputs(cfg, seed=1)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert not torch.equal(a[0], c[0])
    x, wr, bias = a
    assert x.dtype == torch.bfloat16 and x.shape == (cfg.T, cfg.H)
    assert wr.dtype == torch.float32 and wr.shape == (cfg.E, cfg.H)
    assert bias.shape == (cfg.E,)


def test_distributions():
    cfg = mi.CONFIGS["decode"]
    x, wr, bias = mi.make_router_inputs(cfg, seed=0, T=256)
    assert abs(float(x.float().std()) - 1.0) < 0.01
    assert abs(float(wr.std()) * np.sqrt(cfg.H) - 1.0) < 0.01
    assert abs(float(bias.std()) - 0.1) < 0.03


def test_e2m1_rounding_ties_to_even_and_saturates():
    v = torch.tensor([0.0, 0.24, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.1, 7.0, 100.0,
                      -0.75, -5.0, -0.1])
    codes = mi._e2m1_codes(v).tolist()
    #            0  .24 .25 .26 .75 1.25 1.75 2.5 3.5 5  5.1 7  100  -.75 -5  -.1
    assert codes == [0, 0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 7, 10, 14, 0]


def test_nvfp4_pack_roundtrip_of_representable_matrix():
    """A matrix whose entries are exactly e2m1 * e4m3 * global packs without loss."""
    e2m1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6])
    rng = torch.Generator().manual_seed(0)
    N, K = 4, 64
    vals = e2m1[torch.randint(0, 8, (N, K), generator=rng)]
    vals = vals * torch.where(torch.rand(N, K, generator=rng) < 0.5, -1.0, 1.0)
    vals[:, ::16] = 6.0  # each block reaches the e2m1 maximum, so its scale is exact
    scale = torch.tensor([1.0, 2.0, 0.5, 0.25]).repeat(N, 1).repeat_interleave(16, dim=1)
    w = (vals * scale * 0.01).to(torch.bfloat16)
    q, s, g = mi.quantize_nvfp4(w)
    codes = torch.stack([q & 15, q >> 4], dim=-1).view(N, K)
    mag = e2m1[(codes & 7).long()] * torch.where((codes & 8) > 0, -1.0, 1.0)
    sv = s.view(torch.float8_e4m3fn).to(torch.float32).repeat_interleave(16, dim=1)
    back = mag * sv * g
    torch.testing.assert_close(back, w.to(torch.float32), rtol=1e-2, atol=0)


def test_expert_weights_are_per_expert_seeded():
    cfg = mi.CONFIGS["tiny"]
    wg, wu, wd = mi.make_expert_weights(cfg, seed=2)
    g5, u5, d5 = mi.make_expert(cfg, 5, seed=2)
    assert torch.equal(wg[5], g5) and torch.equal(wu[5], u5) and torch.equal(wd[5], d5)
    assert not torch.equal(wg[5], wg[6])
    assert abs(float(wd.float().std()) * np.sqrt(cfg.I) - 1.0) < 0.02
