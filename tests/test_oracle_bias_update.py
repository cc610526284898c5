"""Pins for the oracle's auxiliary-loss-free bias update ("Beam 1.0":
DeepSeek-V3's bias updates with a cosine decay; the rule and schedule are
readings, stated in oracle/moe_oracle.c)."""
import math

import numpy as np
import pytest

import oracle


def test_hand_example_signs():
    # loads: e0=2, e1=0, e2=1, e3=1; mean = 4*... T*k/E = 2*2/4 = 1
    idx = np.array([[0, 2], [0, 3]], np.int32)
    b0 = np.array([0.5, -0.25, 0.0, 1.0], np.float32)
    b, g = oracle.bias_update(idx, b0, 4, 0.001, 0, 100)
    assert g == np.float32(0.001)
    np.testing.assert_array_equal(b, b0 + np.float32(0.001) * np.array([-1, 1, 0, 0], np.float32))


@pytest.mark.parametrize("step,total,factor", [(0, 100, 1.0), (50, 100, 0.5), (100, 100, 0.0),
                                               (300, 100, 0.0), (-5, 100, 1.0), (10, 30, 0.75)])
def test_cosine_schedule_closed_forms(step, total, factor):
    """gamma_t = gamma_max (1 + cos(pi t / T)) / 2: cos 0 = 1, cos(pi/2) = 0,
    cos(pi/3) = 1/2, cos(pi) = -1; steps outside [0, T] clamp."""
    idx = np.zeros((1, 1), np.int32)
    _, g = oracle.bias_update(idx, np.zeros(2, np.float32), 2, 0.004, step, total)
    assert g == pytest.approx(0.004 * factor, abs=1e-9)


def test_balanced_load_leaves_bias_unchanged_and_signs_follow_load():
    rng = np.random.default_rng(0)
    E, T, k = 32, 256, 4
    # perfectly balanced: every expert exactly T*k/E = 32 times
    flat = np.repeat(np.arange(E), T * k // E)
    rng.shuffle(flat)
    b0 = rng.standard_normal(E).astype(np.float32)
    b, _ = oracle.bias_update(flat.reshape(T, k).astype(np.int32), b0, E, 0.01, 3, 10)
    np.testing.assert_array_equal(b, b0)
    # skewed: overloaded experts go down, underloaded up, by exactly one step
    idx = rng.choice(E, size=(T, k), p=np.arange(1, E + 1) / np.arange(1, E + 1).sum()).astype(np.int32)
    b, g = oracle.bias_update(idx, b0, E, 0.01, 0, 10)
    load = np.bincount(idx.ravel(), minlength=E)
    step = (b.astype(np.float64) - b0) / g
    mean = T * k / E
    for e in range(E):
        assert round(step[e]) == (1 if load[e] < mean else -1 if load[e] > mean else 0)
