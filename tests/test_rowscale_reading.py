"""The per-row power-of-two scaling that carries bf16 activations as f16
operands of the packed-weight GEMMs, checked on the CPU against numpy's IEEE
half precision (no GPU): with the factor 2^min(127, 141 - e), e the fp32
exponent field of the row's largest magnitude, the largest magnitude lands in
[2^14, 2^15), every bf16 value of the row that is at least 2^-28 of it is
exact in f16 after scaling, the smaller ones are off by at most 2^-39 of it,
nothing overflows, and multiplying back by the inverse factor is exact."""
import numpy as np
import pytest


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def row_factor_exp(row: np.ndarray) -> int:
    m = np.abs(row).max()
    e32 = int(np.float32(m).view(np.uint32) >> 23) & 0xFF
    return min(127, 141 - e32)


@pytest.mark.parametrize("scale", [1e-30, 1e-6, 1e-3, 1.0, 37.0, 1e5, 3e30])
def test_scaled_rows_are_exact_in_f16(scale):
    rng = np.random.default_rng(7)
    row = bf16_round((rng.standard_normal(5120) * scale).astype(np.float32))
    # a wide spread inside the row: some values 2^-20 .. 2^-40 of the rest
    row[:64] = bf16_round(row[:64] * np.float32(2.0) ** -rng.integers(20, 40, 64).astype(np.float32))
    sx = row_factor_exp(row)
    scaled = row.astype(np.float64) * 2.0 ** sx
    mx = np.abs(scaled).max()
    assert 2.0 ** 14 <= mx < 2.0 ** 15
    h = scaled.astype(np.float16)  # round to nearest even, as cvt.rn.f16x2.f32
    assert np.isfinite(h).all()
    err = np.abs(h.astype(np.float64) - scaled)
    big = np.abs(scaled) >= mx * 2.0 ** -28
    assert (err[big] == 0).all()
    assert (err <= mx * 2.0 ** -39).all()
    # the inverse factor is an fp32 power of two (subnormal at 2^-127): exact
    inv = np.float32(2.0 ** -sx)
    assert float(inv) == 2.0 ** -sx
    back = h[big].astype(np.float64) * float(inv)
    assert (back == row[big].astype(np.float64)).all()


def test_zero_and_tiny_rows_take_the_largest_factor():
    assert row_factor_exp(np.zeros(16, np.float32)) == 127
    tiny = np.full(16, 2.0 ** -120, np.float32)
    assert row_factor_exp(tiny) == 127  # 2^-120 * 2^127 = 2^7: no overflow
    assert float(np.float32(2.0 ** -127)) == 2.0 ** -127


def test_largest_bf16_row_does_not_overflow():
    big = np.float32(3.3895314e38)  # the largest finite bf16
    sx = row_factor_exp(np.array([big], np.float32))
    assert sx == 141 - 254
    assert np.isfinite(np.float16(float(big) * 2.0 ** sx))
