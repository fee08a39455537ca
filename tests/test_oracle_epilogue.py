"""Pins of the oracle's epilogues (residual add, gate/up SwiGLU) to things
other than their own formulas: scipy's logistic function, exact integer
matmuls, the derivative bound by finite differences, and planted mistakes
(gate and up swapped, the residual dropped) that must be caught."""
import numpy as np
import pytest

import oracle as O

scipy_special = pytest.importorskip("scipy.special")


def test_silu_matches_x_times_scipy_expit():
    x = np.concatenate([np.linspace(-40, 40, 20001), [-700.0, -100.0, 100.0, 700.0, 0.0]])
    ref = x * scipy_special.expit(x)
    got = O.silu(x)
    assert np.all(np.abs(got - ref) <= 1e-15 * np.abs(ref) + 1e-300)


def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    x = np.linspace(-30, 30, 6001)
    # silu(-x) = silu(x) - x (sigmoid(-x) = 1 - sigmoid(x))
    assert np.allclose(O.silu(-x), O.silu(x) - x, rtol=0, atol=1e-12)
    assert O.silu(-1e4) == 0.0 and np.signbit(O.silu(-1e4))   # limit, no NaN
    assert O.silu(60.0) == 60.0


def test_silu_lipschitz_constant():
    x = np.linspace(-20, 20, 400001)
    slope = np.abs(np.diff(O.silu(x)) / np.diff(x))
    assert slope.max() <= O.SILU_LIPSCHITZ
    assert slope.max() >= 1.0995  # the constant is tight


def _integer_case(M=3, I=5, K=7, seed=0):
    rng = np.random.default_rng(seed)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-2, 3, size=(2 * I, K)).astype(np.float32)
    # exact products and sums in Python integers
    y = np.array([[sum(int(A[m, k]) * int(W[n, k]) for k in range(K)) for n in range(2 * I)]
                  for m in range(M)], dtype=np.float64)
    return A, W, y


def test_swiglu_reference_exact_integer_case():
    A, W, y_int = _integer_case()
    I = W.shape[0] // 2
    y, B = O.matmul_ref(A, W)
    assert np.array_equal(y, y_int)
    h, tol = O.swiglu_reference(y, np.zeros_like(y), I)
    g, u = y_int[:, :I], y_int[:, I:]
    assert np.allclose(h, g * scipy_special.expit(g) * u, rtol=1e-15, atol=0)
    assert np.all(tol <= 8 * O.F32_EPS * np.abs(h) + 1e-29)


def test_swiglu_reference_catches_swapped_halves():
    A, W, y = _integer_case(seed=1)
    I = W.shape[0] // 2
    tol = np.full_like(y, 1e-3)
    h, t = O.swiglu_reference(y, tol, I)
    swapped = np.concatenate([y[:, I:], y[:, :I]], axis=1)
    h2, _ = O.swiglu_reference(swapped, tol, I)
    assert np.any(np.abs(h2 - h) > t)


def test_swiglu_tolerance_covers_perturbed_inputs():
    rng = np.random.default_rng(3)
    M, I = 64, 300
    y = rng.standard_normal((M, 2 * I)) * 4
    tol = np.abs(rng.standard_normal((M, 2 * I))) * 1e-3
    h, th = O.swiglu_reference(y, tol, I)
    for _ in range(20):
        yp = y + tol * rng.choice([-1.0, 1.0], size=y.shape)
        hp, _ = O.swiglu_reference(yp, np.zeros_like(yp), I)
        assert np.all(np.abs(hp - h) <= th)


def test_residual_reference():
    A, W, y_int = _integer_case(seed=2)
    R = np.arange(y_int.size, dtype=np.float32).reshape(y_int.shape) - 7
    y, _ = O.matmul_ref(A, W)
    c, t = O.residual_reference(y, np.zeros_like(y), R)
    assert np.array_equal(c, y_int + R)
    assert np.all(t <= O.F32_EPS * np.abs(c) + 1e-300)
    # a dropped residual is outside the tolerance
    assert np.any(np.abs(y - c) > t)
