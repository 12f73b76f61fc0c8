"""Pins of the SiLU-times-up oracle (CPU).

``oracle.mlp.silu`` is checked against values fixed by the mathematics rather
than by its own formula: SiLU(0) = 0; SiLU(ln 3) = (3/4) ln 3, because the
logistic function of ln 3 is 1 / (1 + 1/3); the identity
SiLU(z) - SiLU(-z) = z (the logistic function of z and of -z add up to 1);
the limits SiLU(z) -> z and SiLU(-z) -> -z e^-z for large z; and the
independent form z (1 + tanh(z / 2)) / 2 computed with numpy's tanh.  The
tolerance helper is checked to separate a correct fp32 evaluation from
plausible mistakes (the logistic function of -g, the factors swapped)."""
import math

import numpy as np

from oracle import mlp


def test_silu_zero_and_ln3():
    assert mlp.silu(0.0) == 0.0
    assert mlp.silu(-0.0) == 0.0
    z = math.log(3.0)
    assert abs(float(mlp.silu(z)) - 0.75 * z) <= 1e-15 * z
    # h = silu(g) * u by hand: g = ln 3, u = 4 gives 3 ln 3
    assert abs(float(mlp.silu_mul(z, 4.0)) - 3.0 * z) <= 1e-15 * 3.0 * z


def test_silu_odd_part_identity():
    rng = np.random.default_rng(3)
    z = rng.uniform(-30.0, 30.0, 2000)
    lhs = mlp.silu(z) - mlp.silu(-z)
    assert np.all(np.abs(lhs - z) <= 4e-16 * np.abs(z) + 1e-300)


def test_silu_limits():
    assert abs(float(mlp.silu(40.0)) - 40.0) <= 1e-13
    neg = float(mlp.silu(-40.0))
    ref = -40.0 * math.exp(-40.0)
    assert neg < 0 and abs(neg - ref) <= 1e-12 * abs(ref)
    assert float(mlp.silu(-800.0)) == 0.0  # the exponential overflows; the value is -0


def test_silu_matches_tanh_form():
    rng = np.random.default_rng(4)
    z = rng.uniform(-8.0, 8.0, 5000)
    other = z * (1.0 + np.tanh(z / 2.0)) / 2.0
    assert np.allclose(mlp.silu(z), other, rtol=1e-13, atol=1e-15)


def test_bound_accepts_fp32_evaluation_and_rejects_mistakes():
    rng = np.random.default_rng(5)
    g = rng.normal(0.0, 3.0, 20000)
    u = rng.normal(0.0, 3.0, 20000)
    bg = 1e-5 * np.abs(g) + 1e-6
    bu = 1e-5 * np.abs(u) + 1e-6
    # perturb within the bounds, evaluate in fp32 as a kernel would
    g32 = (g + bg * rng.uniform(-1, 1, g.size)).astype(np.float32)
    u32 = (u + bu * rng.uniform(-1, 1, u.size)).astype(np.float32)
    h32 = (g32 / (np.float32(1) + np.exp(-g32))) * u32
    ref = mlp.silu_mul(g, u)
    bound = mlp.silu_mul_bound(g, u, bg, bu)
    assert np.all(np.abs(h32.astype(np.float64) - ref) <= bound)
    # plausible mistakes fail it
    wrong_sign = (g32 / (np.float32(1) + np.exp(g32))) * u32
    swapped = (u32 / (np.float32(1) + np.exp(-u32))) * g32
    for bad in (wrong_sign, swapped):
        assert np.mean(np.abs(bad.astype(np.float64) - ref) > bound) > 0.5
