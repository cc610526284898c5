"""Pins for the oracle's NVFP4 activation quantiser and its W4A4 expert (CPU only).

The pages name NVFP4 as Beam's Blackwell checkpoint format ("Reflection
Releases Beam ...", section "Where Beam Saves and Where the Memory Bill Comes
In"; "Hugging Face releases Beam ...", hardware paragraph) and nothing more.
The W4A4 mode reads it as the same two-level format applied to activations:
one E4M3 scale per 16 consecutive values of a row and a static fp32 global
scale per tensor, codes rounded to nearest-even with saturation.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi

E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_val(code):
    v = E2M1_MAG[code & 7]
    return -v if code & 8 else v


def e4m3_val(code):
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).double())


# ------------------------------------------------------------------ scalar rounding


@pytest.mark.parametrize("v,code", [
    # exact values
    (0.0, 0), (0.5, 1), (1.0, 2), (1.5, 3), (2.0, 4), (3.0, 5), (4.0, 6), (6.0, 7),
    # midpoints go to the neighbour with mantissa bit 0 (the even code)
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    # just off the midpoints
    (0.2500001, 1), (0.7499999, 1), (1.2500001, 3), (4.9999995, 7 - 1), (5.0000005, 7),
    # saturation, sign, signed zero
    (6.5, 7), (1e30, 7), (-1e30, 15), (-1.0, 10), (-5.0, 14), (-0.0, 8), (-0.1, 8), (0.1, 0),
])
def test_e2m1_rounding_cases(oracle_mod, v, code):
    """Cases fixed by the E2M1 definition (1 sign, 2 exponent bits with bias 1,
    1 mantissa bit: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6) and round-to-nearest-even."""
    assert oracle_mod.e2m1_rne(np.float32(v)) == code


def test_e2m1_is_nearest_with_even_ties(oracle_mod):
    """Over a dense grid: the chosen magnitude is a nearest one, and among two
    equally near the one with an even code."""
    grid = np.concatenate([np.linspace(-7, 7, 5601, dtype=np.float32),
                           np.float32(np.arange(-14, 15)) / np.float32(4)])
    for v in grid:
        c = oracle_mod.e2m1_rne(float(v))
        a = min(abs(float(v)), 6.0)
        d = [abs(a - m) for m in E2M1_MAG]
        best = min(d)
        assert d[c & 7] == best
        near = [i for i in range(8) if d[i] == best]
        if len(near) == 2:
            assert (c & 7) % 2 == 0
        assert (c >> 3) == (1 if np.signbit(v) else 0)


def test_e4m3_rounding_matches_torch(oracle_mod):
    """Against torch's float8_e4m3fn conversion (a library round-to-nearest-even)
    on every midpoint between codes, its neighbours, and random values below
    the saturation point."""
    vals = [e4m3_val(c) for c in range(127)]
    pts = []
    for c in range(126):
        m = np.float32((vals[c] + vals[c + 1]) / 2)
        pts += [m, np.nextafter(m, np.float32(1e9)), np.nextafter(m, np.float32(-1e9)),
                np.float32(vals[c])]
    rng = np.random.default_rng(3)
    pts += list((rng.random(3000) * 440).astype(np.float32))
    pts += list((2.0 ** rng.uniform(-12, 8, 3000)).astype(np.float32))
    pts = np.array(pts, np.float32)
    pts = pts[pts < 448]
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_rne(float(v)) for v in pts], np.uint8)
    np.testing.assert_array_equal(got, ref)
    neg = np.array([oracle_mod.e4m3_rne(float(-v)) for v in pts[:200]], np.uint8)
    np.testing.assert_array_equal(neg, ref[:200] | 0x80)


def test_e4m3_saturates(oracle_mod):
    for v in (448.0, 460.0, 464.0, 1000.0, 3e38):
        assert oracle_mod.e4m3_rne(v) == 0x7E
    assert oracle_mod.e4m3_rne(-500.0) == 0xFE
    assert oracle_mod.e4m3_rne(2.0 ** -10) == 0      # half the smallest subnormal: tie to 0
    assert oracle_mod.e4m3_rne(3 * 2.0 ** -10) == 2  # 1.5 subnormal steps: tie to the even code


# ------------------------------------------------------------------ block quantiser


def unpack(q):
    lo, hi = q & 15, q >> 4
    out = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    out[:, 0::2], out[:, 1::2] = lo, hi
    return out


def dequant(q, s, g):
    codes = unpack(q)
    val = np.vectorize(e2m1_val)(codes).astype(np.float64)
    sc = np.vectorize(e4m3_val)(s).astype(np.float64)
    return val * np.repeat(sc, 16, axis=1) * g


def test_representable_rows_round_trip(oracle_mod):
    """Blocks built from codes and a scale, with one element at +-6 * scale,
    come back with the same codes and scale: pins amax/6, the division by
    scale * g, nibble order and the scale layout."""
    rng = np.random.default_rng(0)
    rows, cols, g = 5, 64, np.float32(0.0371)
    scodes = rng.choice(np.arange(0x20, 0x60), size=(rows, cols // 16)).astype(np.uint8)
    codes = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    codes[codes == 8] = 0  # -0 reads back as +0 only when the value is exactly zero
    for r in range(rows):
        for b in range(cols // 16):
            codes[r, 16 * b + (r + b) % 16] = 7 if (r + b) % 2 else 15
    v = np.vectorize(e2m1_val)(codes) * np.repeat(np.vectorize(e4m3_val)(scodes), 16, axis=1)
    v = (v * np.float64(g)).astype(np.float32)
    q, s = oracle_mod.quantize_nvfp4(v, float(g))
    np.testing.assert_array_equal(s, scodes)
    np.testing.assert_array_equal(unpack(q), codes)
    # v itself is the fp32 rounding of code * scale * g
    np.testing.assert_allclose(dequant(q, s, np.float64(g)), v.astype(np.float64), rtol=2.0 ** -24)


def test_zero_block_and_bound(oracle_mod):
    """An all-zero block gets scale code 0 and zero codes; every other value is
    within one scale step (half the widest E2M1 gap) of its dequantised value,
    plus whatever saturation clips."""
    rng = np.random.default_rng(1)
    v = rng.standard_normal((7, 96)).astype(np.float32) * np.float32(3)
    v[2, 16:32] = 0.0
    v[4, :16] *= np.float32(1e-3)
    g = 0.01
    q, s = oracle_mod.quantize_nvfp4(v, g)
    assert s[2, 1] == 0 and np.all(q[2, 8:16] == 0)
    vh = dequant(q, s, g)
    scale = np.repeat(np.vectorize(e4m3_val)(s), 16, axis=1) * g
    clip = np.maximum(0.0, np.abs(v) - 6 * scale)
    assert np.all(np.abs(v - vh) <= scale * 1.0 + clip + 1e-12)
    # relative error of the whole matrix: NVFP4 keeps roughly 10-15%
    assert np.linalg.norm(v - vh) / np.linalg.norm(v) < 0.15


def test_quantiser_matches_brute_force(oracle_mod):
    """Tiny rows against a brute-force restatement: torch's E4M3 rounding for the
    block scale, exhaustive nearest-value search for the codes."""
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((3, 48)) * 2).astype(np.float32)
    g = np.float32(0.02)
    q, s = oracle_mod.quantize_nvfp4(v, float(g))
    codes = unpack(q)
    for r in range(3):
        for b in range(3):
            blk = v[r, 16 * b:16 * b + 16]
            amax = np.float32(np.max(np.abs(blk)))
            u = np.float32(amax / np.float32(np.float32(6) * g))
            sc = int(torch.tensor([u]).to(torch.float8_e4m3fn).view(torch.uint8))
            assert s[r, b] == sc
            scale = np.float32(np.float32(e4m3_val(sc)) * g)
            for i in range(16):
                t = np.float32(blk[i] / scale)
                dist = [abs(abs(float(t)) - m) for m in E2M1_MAG]
                best = min(dist)
                cands = [c for c in range(8) if dist[c] == best]
                c = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
                c = 7 if abs(float(t)) >= 6 else c
                assert codes[r, 16 * b + i] == (c | (8 if t < 0 or np.signbit(t) else 0))


# ------------------------------------------------------------------ W4A4 expert


def _nvfp4_identity(n):
    """NVFP4 identity matrix [n, n]: code 2 (1.0), scale 1.0 (0x38), global 1."""
    codes = np.zeros((n, n), np.uint8)
    np.fill_diagonal(codes, 2)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = np.full((n, n // 16), 0x38, np.uint8)
    return q, s


def test_w4a4_expert_steps_and_order(oracle_mod):
    """With x exactly representable (x_hat = x) and W_down the identity, the
    W4A4 expert returns dequant(quantize(fp32(h), gh)) where h is the W4A16
    expert's output: x is quantised before gate/up, h after SwiGLU, in that order."""
    H = I = 64
    rng = np.random.default_rng(5)
    gx, gh = np.float32(2.0 ** -4), np.float32(0.013)
    # representable activations: codes times power-of-two block scales times gx
    # (exact in bf16), with a +-6 in every block so that amax fixes the scale
    codes = rng.integers(0, 16, size=(3, H)).astype(np.uint8)
    codes[codes == 8] = 0
    for r in range(3):
        for b in range(H // 16):
            codes[r, 16 * b + (3 * r + b) % 16] = 7 if (r + b) % 2 else 15
    sc = rng.choice([0x30, 0x38, 0x40], size=(3, H // 16))
    xv = np.vectorize(e2m1_val)(codes) * np.repeat(np.vectorize(e4m3_val)(sc), 16, axis=1)
    xv = (xv * np.float64(gx)).astype(np.float32)
    xt = torch.from_numpy(xv).to(torch.bfloat16)
    assert np.array_equal(xt.float().numpy(), xv)
    xb = mi.bf16_bits(xt)
    M = oracle_mod.Nvfp4Matrix
    wq = [mi.quantize_nvfp4(torch.randn(I, H, generator=torch.Generator().manual_seed(k)) / 8)
          for k in (1, 2)]
    wg, wu = [M(q.numpy(), s.numpy(), float(g)) for q, s, g in wq]
    iq, isc = _nvfp4_identity(I)
    wd = M(iq, isc, 1.0)
    h16 = oracle_mod.expert_swiglu(xb, wg, wu, wd)          # W4A16: o = h (fp64)
    o4 = oracle_mod.expert_swiglu_w4a4(xb, wg, wu, wd, float(gx), float(gh))
    # x quantisation must be lossless here
    qx, sx = oracle_mod.quantize_nvfp4(xv, float(gx))
    np.testing.assert_array_equal(dequant(qx, sx, np.float64(gx)), xv.astype(np.float64))
    qh, sh = oracle_mod.quantize_nvfp4(h16.astype(np.float32), float(gh))
    np.testing.assert_array_equal(o4, dequant(qh, sh, np.float64(gh)))
    assert np.linalg.norm(o4 - h16) / np.linalg.norm(h16) < 0.15


def test_w4a4_expert_close_to_w4a16(oracle_mod):
    """On the tiny workload W4A4 stays within NVFP4 quantisation noise of W4A16."""
    H, I = 256, 256
    g = torch.Generator().manual_seed(9)
    ws = [torch.randn(I, H, generator=g) / 16, torch.randn(I, H, generator=g) / 16,
          torch.randn(H, I, generator=g) / 16]
    mats = [oracle_mod.Nvfp4Matrix(q.numpy(), s.numpy(), float(gg))
            for q, s, gg in (mi.quantize_nvfp4(w) for w in ws)]
    x = torch.randn(6, H, generator=g).to(torch.bfloat16)
    xb = mi.bf16_bits(x)
    o16 = oracle_mod.expert_swiglu(xb, *mats)
    o4 = oracle_mod.expert_swiglu_w4a4(xb, *mats, 8.0 / 2688, 4.0 / 2688)
    rel = np.linalg.norm(o4 - o16) / np.linalg.norm(o16)
    assert 1e-3 < rel < 0.2
