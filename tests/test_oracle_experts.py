"""Pins for the oracle's expert path and NVFP4 decoding (CPU only).

The expert is a SwiGLU MLP ("Hugging Face releases Beam ...", third
paragraph: each expert a SwiGLU MLP with intermediate size 2,560); the
block's output is the routed-weight sum of its 8 experts with no shared
expert ("Reflection Releases Beam ...", section "Where Beam Saves and Where
the Memory Bill Comes In").  NVFP4 decoding follows the OCP MX v1.0 tables.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import moe_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a):
    """fp32 values exact in bf16 -> uint16 bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def silu(z):
    return z * expit(z)


def test_one_hot_weights_closed_form(oracle_mod):
    """W_gate, W_up and W_down are selection matrices (H=8, I=4, so a
    transposed operand cannot line up): o_j = silu(x[p(r(j))]) * x[q(r(j))]."""
    H, I = 8, 4
    p = [5, 0, 7, 2]
    q = [1, 1, 6, 3]
    rr = [3, 0, 2, 1, 1, 0, 3, 2]
    wg = np.zeros((I, H), np.float32)
    wu = np.zeros((I, H), np.float32)
    wd = np.zeros((H, I), np.float32)
    for i in range(I):
        wg[i, p[i]] = 1.0
        wu[i, q[i]] = 1.0
    for j in range(H):
        wd[j, rr[j]] = 1.0
    x = np.array([[1.0, -2.0, 0.5, 3.0, -0.25, 2.0, -1.5, 0.75],
                  [0.0, 1.0, -1.0, 4.0, 1.0, -3.0, 2.0, -0.5]], np.float32)
    o = oracle_mod.expert_swiglu(bits(x), bits(wg), bits(wu), bits(wd))
    for t in range(2):
        a = [silu(float(x[t, p[i]])) * float(x[t, q[i]]) for i in range(I)]
        np.testing.assert_allclose(o[t], [a[rr[j]] for j in range(H)], rtol=1e-14, atol=0)


def test_gate_and_up_are_not_interchangeable(oracle_mod):
    """W_gate = 2*Id, W_up = Id, W_down = Id: o = silu(2x) * x, not silu(x) * 2x."""
    H = I = 4
    x = np.array([[1.0, -1.0, 0.5, 2.0]], np.float32)
    eye = np.eye(4, dtype=np.float32)
    o = oracle_mod.expert_swiglu(bits(x), bits(2 * eye), bits(eye), bits(eye))
    np.testing.assert_allclose(o[0], silu(2 * x[0].astype(np.float64)) * x[0], rtol=1e-14)


def test_matches_library_matmul(oracle_mod):
    """Random expert at the tiny shape against numpy float64 matmuls and scipy's expit."""
    cfg = mi.CONFIGS["tiny"]
    wg, wu, wd = mi.make_expert_weights(cfg, seed=3)
    x, _, _ = mi.make_router_inputs(cfg, seed=3, T=10)
    o = oracle_mod.expert_swiglu(mi.bf16_bits(x), mi.bf16_bits(wg[5]), mi.bf16_bits(wu[5]),
                                 mi.bf16_bits(wd[5]))
    xd = x.double().numpy()
    g = xd @ wg[5].double().numpy().T
    u = xd @ wu[5].double().numpy().T
    ref = (silu(g) * u) @ wd[5].double().numpy().T
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)


def _tiny_block(seed=0):
    cfg = mi.CONFIGS["tiny"]
    x, wr, b = mi.make_router_inputs(cfg, seed=seed)
    wg, wu, wd = mi.make_expert_weights(cfg, seed=seed)
    W = [(mi.bf16_bits(wg[e]), mi.bf16_bits(wu[e]), mi.bf16_bits(wd[e])) for e in range(cfg.E)]
    return cfg, mi.bf16_bits(x), wr.numpy(), b.numpy(), W


def test_combine_is_weighted_sum_in_k_order(oracle_mod):
    w = np.array([[0.5, 0.25, 2.0]], np.float32)
    o = np.arange(12, dtype=np.float64).reshape(1, 3, 4)
    y = oracle_mod.combine(w, o)
    np.testing.assert_array_equal(y[0], 0.5 * o[0, 0] + 0.25 * o[0, 1] + 2.0 * o[0, 2])


def test_identical_experts_give_scaled_mlp(oracle_mod):
    """Every expert the same: the weights sum to 2.5, so y = 2.5 * MLP(x)."""
    cfg, x, wr, b, W = _tiny_block(1)
    y, r = oracle_mod.moe_forward(x, wr, b, lambda e: W[0], cfg.n_group, cfg.topk_group,
                                  cfg.top_k, cfg.routed_scale)
    mlp = oracle_mod.expert_swiglu(x, *W[0])
    np.testing.assert_allclose(y, 2.5 * mlp, rtol=2e-6, atol=1e-9)


def test_zero_down_expert_contributes_nothing(oracle_mod):
    cfg, x, wr, b, W = _tiny_block(2)
    y, r = oracle_mod.moe_forward(x, wr, b, lambda e: W[e], cfg.n_group, cfg.topk_group,
                                  cfg.top_k, cfg.routed_scale)
    hot = int(r.idx[0, 0])
    W0 = list(W)
    W0[hot] = (W[hot][0], W[hot][1], np.zeros_like(W[hot][2]))
    y0, _ = oracle_mod.moe_forward(x, wr, b, lambda e: W0[e], cfg.n_group, cfg.topk_group,
                                   cfg.top_k, cfg.routed_scale)
    # recompute with that expert's slot dropped from the weighted sum
    o = np.zeros((cfg.T, cfg.top_k, cfg.H))
    for t in range(cfg.T):
        for k in range(cfg.top_k):
            e = int(r.idx[t, k])
            if e != hot:
                o[t, k] = oracle_mod.expert_swiglu(x[t:t + 1], *W[e])[0]
    np.testing.assert_allclose(y0, oracle_mod.combine(r.w, o), rtol=1e-12, atol=1e-15)
    # all-zero W_down everywhere gives an exactly zero output
    Wz = [(a, u, np.zeros_like(d)) for a, u, d in W]
    yz, _ = oracle_mod.moe_forward(x, wr, b, lambda e: Wz[e], cfg.n_group, cfg.topk_group,
                                   cfg.top_k, cfg.routed_scale)
    assert np.all(yz == 0.0)


def test_linear_in_down_weights_and_token_equivariant(oracle_mod):
    cfg, x, wr, b, W = _tiny_block(3)
    args = (cfg.n_group, cfg.topk_group, cfg.top_k, cfg.routed_scale)
    y, r = oracle_mod.moe_forward(x, wr, b, lambda e: W[e], *args)
    # doubling bf16 W_down is exact, so y doubles exactly
    W2 = [(a, u, bits(2 * (d.astype(np.uint32) << 16).view(np.float32))) for a, u, d in W]
    y2, _ = oracle_mod.moe_forward(x, wr, b, lambda e: W2[e], *args)
    np.testing.assert_array_equal(y2, 2 * y)
    perm = np.random.default_rng(0).permutation(cfg.T)
    yp, _ = oracle_mod.moe_forward(np.ascontiguousarray(x[perm]), wr, b, lambda e: W[e], *args)
    np.testing.assert_array_equal(yp, y[perm])
    # a token subset gives the same rows
    ys = oracle_mod.experts_forward(x, r.idx, r.w, lambda e: W[e], tokens=[5, 1, 40])
    np.testing.assert_array_equal(ys, y[[5, 1, 40]])


# ------------------------------------------------------------------ NVFP4 decoding


def test_e2m1_and_e4m3_tables(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_formats.json")))
    for code, v in g["e2m1"].items():
        assert oracle_mod.e2m1_value(int(code)) == v
    for code, v in g["e4m3"].items():
        assert oracle_mod.e4m3_value(int(code)) == v
    for code in g["e4m3_nan_codes"]:
        assert np.isnan(oracle_mod.e4m3_value(code))


def test_e4m3_matches_torch_for_all_codes(oracle_mod):
    """Every E4M3 code against torch's float8_e4m3fn conversion (a library routine)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(got[m], ref[m])


def test_nvfp4_matrix_decoding(oracle_mod):
    """Hand-built 2x32 NVFP4 matrix: value = e2m1(code) * e4m3(block scale) * global,
    low nibble = even column."""
    N, K = 2, 32
    codes = np.array([[(c + r) % 16 for c in range(K)] for r in range(N)], np.uint8)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = np.array([[56, 64], [57, 1]], np.uint8)       # 1.0, 2.0 | 1.125, 2^-9
    glob = 0.75
    dec = oracle_mod.decode_matrix(oracle_mod.Nvfp4Matrix(q, s, glob))
    e2m1 = [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]
    scale = {56: 1.0, 64: 2.0, 57: 1.125, 1: 2.0 ** -9}
    for r in range(N):
        for c in range(K):
            assert dec[r, c] == e2m1[codes[r, c]] * scale[int(s[r, c // 16])] * glob


def test_nvfp4_expert_equals_bf16_path_on_decoded_weights(oracle_mod):
    """An NVFP4 expert gives the same result as the fp64 library matmul on its
    decoded weights."""
    cfg = mi.CONFIGS["tiny"]
    wg, wu, wd = mi.make_expert_weights(cfg, seed=4)
    packed = [mi.quantize_nvfp4(w[2]) for w in (wg, wu, wd)]
    mats = [oracle_mod.Nvfp4Matrix(q.numpy(), s.numpy(), float(g)) for q, s, g in packed]
    x, _, _ = mi.make_router_inputs(cfg, seed=4, T=6)
    o = oracle_mod.expert_swiglu(mi.bf16_bits(x), *mats)
    dg, du, dd = [oracle_mod.decode_matrix(m) for m in mats]
    xd = x.double().numpy()
    ref = (silu(xd @ dg.T) * (xd @ du.T)) @ dd.T
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    # quantisation error of the packed weights is a few percent of their size
    rel = np.linalg.norm(dg - wg[2].double().numpy()) / np.linalg.norm(wg[2].double().numpy())
    assert rel < 0.12


# ------------------------------------------------------------------ FP8 (one scale per row)


def test_fp8_matrix_decoding(oracle_mod):
    """Hand-built FP8 matrix: value = e4m3(code) * row scale."""
    q = np.array([[56, 64, 1, 184], [126, 0, 57, 63]], np.uint8)  # 1, 2, 2^-9, -1 | 448, 0, 1.125, 1.875
    rs = np.array([0.5, 3.0], np.float32)
    dec = oracle_mod.decode_matrix(oracle_mod.Fp8Matrix(q, rs))
    np.testing.assert_array_equal(dec, [[0.5, 1.0, 2.0 ** -10, -0.5], [1344.0, 0.0, 3.375, 5.625]])


def test_fp8_expert_equals_library_matmul_on_decoded_weights(oracle_mod):
    cfg = mi.CONFIGS["tiny"]
    wg, wu, wd = mi.make_expert_weights(cfg, seed=6)
    mats = [oracle_mod.Fp8Matrix(*[t.numpy() for t in mi.quantize_fp8_rows(w[1])])
            for w in (wg, wu, wd)]
    x, _, _ = mi.make_router_inputs(cfg, seed=6, T=5)
    o = oracle_mod.expert_swiglu(mi.bf16_bits(x), *mats)
    dg, du, dd = [oracle_mod.decode_matrix(m) for m in mats]
    xd = x.double().numpy()
    ref = (silu(xd @ dg.T) * (xd @ du.T)) @ dd.T
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    # e4m3 with a per-row scale keeps about 2^-4 relative error per weight
    rel = np.linalg.norm(dg - wg[1].double().numpy()) / np.linalg.norm(wg[1].double().numpy())
    assert rel < 0.05
