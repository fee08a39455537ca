"""Pins for the oracle's matmul reference C = A @ dequant(W)^T.

Identity and one-hot weights, constant blocks and brute-force integer cases
give exact answers computed here with Python integers; linearity and row
permutation are invariants; a float64 torch matmul on the dequantised
weights is the library cross-check.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic


def _f16r(v) -> float:
    """Round one float32 value through the oracle's f16 encoding."""
    return float(O.f16_bits_to_f32(O.f32_to_f16_bits(np.array([v], dtype=np.float32)))[0])


def _exact_int_sum(a_row, w_row):
    return sum(int(x) * int(y) for x, y in zip(a_row, w_row))


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_identity_weights(fmt):
    K = 64
    W = np.eye(K, dtype=np.float32)
    A = np.random.default_rng(0).standard_normal((3, K)).astype(np.float32)
    y, _ = O.reference(fmt, A, O.pack(fmt, W), K, K)
    if fmt in ("f16", "q4_0"):
        # f16: 1.0 exact; Q4_0: m = 1, d = -1/8 exact, q_diag = 0 -> w = 1
        assert np.array_equal(y, A.astype(np.float64))
    else:
        # Q8_0: d = 1/127 in f32, stored as f16 -> w_diag = f16(1/127) * 127
        w = _f16r(np.float32(1) / np.float32(127)) * 127
        assert np.array_equal(y, A.astype(np.float64) * w)
        assert w != 1.0


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_one_hot_weights(fmt):
    N, K = 8, 96
    rng = np.random.default_rng(1)
    A = rng.standard_normal((2, K)).astype(np.float32)
    cols = rng.integers(0, K, size=N)
    vals = np.array([0.5, -0.75, 3.0, -2.0, 0.125, 1.5, -0.25, 7.0], dtype=np.float32)
    W = np.zeros((N, K), dtype=np.float32)
    W[np.arange(N), cols] = vals
    y, _ = O.reference(fmt, A, O.pack(fmt, W), N, K)
    if fmt == "q8_0":
        wv = O.f16_bits_to_f32(O.f32_to_f16_bits(np.abs(vals) / np.float32(127))).astype(np.float64) * 127 * np.sign(vals)
    else:  # f16 and Q4_0 reproduce these values exactly (v/8 is f16-exact)
        wv = vals.astype(np.float64)
    want = A.astype(np.float64)[:, cols] * wv[None, :]
    assert np.array_equal(y, want)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_constant_block_equals_scaled_block_sum(fmt):
    K = 128
    c = np.float32(0.3)
    W = np.zeros((1, K), dtype=np.float32)
    W[0, 32:64] = c
    A = np.random.default_rng(2).standard_normal((1, K)).astype(np.float32)
    y, _ = O.reference(fmt, A, O.pack(fmt, W), 1, K)
    if fmt == "q8_0":
        w = _f16r(c / np.float32(127)) * 127
    else:
        w = -8.0 * _f16r(c / np.float32(-8))
    assert y[0, 0] == pytest.approx(w * A[0, 32:64].astype(np.float64).sum(), rel=1e-15, abs=1e-15)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M", [1, 4])
def test_brute_force_4x32_integers(fmt, M):
    """N=4 rows, K=32: weights are integers times 2^-3 chosen so that every
    block quantises exactly (Q8_0: a +-127 in each block, Q4_0: a -8 first),
    activations are integers in [-3, 3]; the answer is an integer sum."""
    rng = np.random.default_rng(100 + M)
    N, K, s = 4, 32, 0.125
    if fmt == "q8_0":
        t = rng.integers(-127, 128, size=(N, K))
        t[:, 5] = 127
        t[2, 5] = -127
    elif fmt == "q4_0":
        t = rng.integers(-7, 8, size=(N, K))
        t[:, 0] = -8
    else:
        t = rng.integers(-2000, 2001, size=(N, K))
    a = rng.integers(-3, 4, size=(M, K))
    W = (t * s).astype(np.float32)
    A = a.astype(np.float32)
    y, _ = O.reference(fmt, A, O.pack(fmt, W), N, K)
    _, B = O.matmul_ref(A, O.dequantize(fmt, O.pack(fmt, W), N, K))
    for m in range(M):
        for n in range(N):
            assert y[m, n] == _exact_int_sum(a[m], t[n]) * s
            assert B[m, n] == sum(abs(int(x) * int(z)) for x, z in zip(a[m], t[n])) * s


def test_linearity_and_row_permutation():
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    A1 = rng.standard_normal((2, 256)).astype(np.float32)
    A2 = rng.standard_normal((2, 256)).astype(np.float32)
    for fmt in ("f16", "q8_0", "q4_0"):
        p = O.pack(fmt, W)
        y1, _ = O.reference(fmt, A1, p, 32, 256)
        y2, _ = O.reference(fmt, A2, p, 32, 256)
        y12, _ = O.reference(fmt, A1 + A2, p, 32, 256)
        # A1 + A2 is rounded to f32, so compare within that rounding
        assert np.allclose(y12, y1 + y2, rtol=0, atol=1e-5)
        perm = rng.permutation(32)
        yp, _ = O.reference(fmt, A1, O.pack(fmt, W[perm]), 32, 256)
        assert np.array_equal(yp, y1[:, perm])


def test_matches_torch_float64_on_dequantised_weights():
    rng = np.random.default_rng(4)
    W = (rng.standard_normal((48, 512)) * 0.02).astype(np.float32)
    A = rng.standard_normal((5, 512)).astype(np.float32)
    for fmt in ("f16", "q8_0", "q4_0"):
        p = O.pack(fmt, W)
        What = O.dequantize(fmt, p, 48, 512)
        y, _ = O.reference(fmt, A, p, 48, 512)
        _, B = O.matmul_ref(A, What)
        t = torch.from_numpy(A).double() @ torch.from_numpy(What).double().T
        assert np.allclose(y, t.numpy(), rtol=1e-13, atol=1e-13)
        assert np.all(B >= np.abs(y) - 1e-12)


def test_tensor_core_reference_rounds_activations_to_bf16():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    A = rng.standard_normal((3, 256)).astype(np.float32)
    p = O.pack("q8_0", W)
    y, tol = O.reference("q8_0", A, p, 16, 256, tensor_core=True)
    Ab = torch.from_numpy(A).to(torch.bfloat16).double()
    t = Ab @ torch.from_numpy(O.dequantize("q8_0", p, 16, 256)).double().T
    assert np.allclose(y, t.numpy(), rtol=1e-13, atol=1e-13)
    _, B = O.matmul_ref(O.f32_to_bf16_rne(A), O.dequantize("q8_0", p, 16, 256))
    assert np.array_equal(tol, O.GEMM_RTOL * B + O.GEMM_ATOL)


def test_argmax_first():
    assert O.argmax_first([1.0, 3.0, 3.0, 2.0]) == 1
    assert O.argmax_first([np.nan, 1.0, np.nan, 1.0]) == 1
    assert O.argmax_first([-np.inf, -5.0]) == 1
    assert O.argmax_first([np.nan, np.nan]) == -1


def test_planted_transposed_weights_are_caught():
    """Feeding W instead of W^T orientation (a transposed operand) breaks the
    brute-force integer check."""
    rng = np.random.default_rng(6)
    t = rng.integers(-3, 4, size=(32, 32))
    a = rng.integers(-3, 4, size=(1, 32))
    W = t.astype(np.float32)
    y, _ = O.matmul_ref(a.astype(np.float32), W)
    yT, _ = O.matmul_ref(a.astype(np.float32), W.T.copy())
    want = [_exact_int_sum(a[0], t[n]) for n in range(32)]
    assert list(y[0]) == want
    assert list(yT[0]) != want


def test_synthetic_recipe():
    w = synthetic.WORKLOADS["gemv_q4_0_11008x4096_outliers"]
    assert synthetic.n_outlier_blocks(w.N, w.K, w.outlier_frac) == 70451
    W1, A1 = synthetic.draw(1, 64, 128, seed=3, outlier_frac=0.05)
    W2, A2 = synthetic.draw(1, 64, 128, seed=3, outlier_frac=0.05)
    assert torch.equal(W1, W2) and torch.equal(A1, A2)
    W0, _ = synthetic.draw(1, 64, 128, seed=3)
    ratio = (W1 / W0).view(-1, 32)[:, 0]
    big = torch.isclose(ratio, torch.tensor(20.0))
    assert int(big.sum()) == synthetic.n_outlier_blocks(64, 128, 0.05)
    assert abs(float(W0.std()) - 0.02) < 0.002


def test_topk_first_against_lexsort_and_brute_force():
    """topk_first against numpy's lexsort (an independent ordering routine)
    on random data with planted ties and NaN, and against argmax_first."""
    rng = np.random.default_rng(3)
    for n, k in [(1, 1), (7, 3), (100, 64), (1000, 50), (5, 9)]:
        y = rng.standard_normal(n)
        if n > 10:
            y[rng.choice(n, n // 10, replace=False)] = np.nan
            y[rng.choice(n, 5, replace=False)] = np.nanmax(y)     # a tie at the top
            y[rng.choice(n, 3, replace=False)] = -np.inf
        v, i = O.topk_first(y, k)
        ok = np.nonzero(~np.isnan(y))[0]
        order = ok[np.lexsort((ok, -y[ok]))][:k]
        assert list(i[:len(order)]) == list(order)
        assert np.all(i[len(order):] == -1) and np.all(np.isneginf(v[len(order):]))
        assert np.array_equal(v[:len(order)], y[order])
        assert i[0] == O.argmax_first(y)


def test_topk_first_special_values():
    v, i = O.topk_first([0.0, -0.0, 1.0, np.nan, -0.0], 4)
    assert list(i) == [2, 0, 1, 4]          # -0 and +0 tie: by index
    v, i = O.topk_first([np.nan, np.nan], 2)
    assert list(i) == [-1, -1] and np.all(np.isneginf(v))
    v, i = O.topk_first([-np.inf, 3.0, -np.inf], 3)
    assert list(i) == [1, 0, 2]             # real -inf entries come before the sentinel
