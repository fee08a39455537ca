"""lq_gemv_argmax (the GEMV fused with the argmax of its outputs) and
lq_argmax_f32, against the oracle.

The argmax is an integer decided by floating point, so both sides decide it
in the kernel's precision: the chosen index must equal the oracle's
argmax_first over the GPU's own f32 logits (and the value must be that logit,
bit for bit). Against the exact f64 reference the index must be the
reference's, or a near-tie within the two rows' GEMV tolerances. Ties are
planted with identical weight rows (their outputs are bit-identical), NaN
with NaN weights in the packed bytes.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, reference_rows, to_dev

pytestmark = pytest.mark.gpu

F16_NAN = 0x7E00


def _dev_weights(lq, fmt, Wn, dev):
    return to_dev(lq.pack(fmt, Wn).reshape(-1).view(np.uint8), dev)


def _fused(lq, fmt, A, Wd, N, K, dev, with_c=True):
    C = nan_filled(1, N, dev)[0] if with_c else None
    res = lq.argmax_result(dev)
    lq.lq_gemv_argmax(fmt, A, Wd, C, N, K, res)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    v, i = lq.read_argmax(res)
    return v, i, (C.cpu().numpy() if with_c else None)


def _assert_self_consistent(v, i, c):
    """The index is argmax_first of the kernel's own logits, value = c[i]."""
    assert i == O.argmax_first(c), (i, O.argmax_first(c))
    assert np.float32(v).tobytes() == np.float32(c[i]).tobytes()


def test_lmhead_config_fused_argmax(lq, cuda_dev):
    """The LM-head shape (f16, 151936 x 2048): index and value from the fused
    kernel, with and without storing the logits; the logits match the
    oracle."""
    w = synthetic.WORKLOADS["gemv_f16_lmhead_151936x2048"]
    W, A = synthetic.draw_workload(w)
    Wn = W.numpy()
    del W
    Wd = _dev_weights(lq, "f16", Wn, cuda_dev)
    Ad = A.to(cuda_dev)[0]
    lq.reset_counts()
    v, i, c = _fused(lq, "f16", Ad, Wd, w.N, w.K, cuda_dev)
    assert lq.route_count(0) == 1
    _assert_self_consistent(v, i, c)
    v2, i2, _ = _fused(lq, "f16", Ad, Wd, w.N, w.K, cuda_dev, with_c=False)
    assert (v2, i2) == (v, i)
    y, tol = reference_rows("f16", A.numpy(), Wn, np.arange(w.N))
    check(c[None, :], y, tol, "lm head logits")
    i_ref = O.argmax_first(y[0])
    assert i == i_ref or y[0, i_ref] - y[0, i] <= tol[0, i_ref] + tol[0, i], (i, i_ref)


@pytest.mark.parametrize("fmt,N,K", [("q8_0", 4096, 4096), ("q4_0", 11008, 4096), ("f16", 1000, 512),
                                     ("q8_0", 100, 2048), ("f16", 7, 2048), ("q4_0", 152 * 16 + 3, 8192)])
def test_fused_argmax_formats(lq, cuda_dev, fmt, N, K):
    W, A = synthetic.draw(1, N, K, seed=N + K, outlier_frac=0.05)
    Wn = W.numpy()
    v, i, c = _fused(lq, fmt, A.to(cuda_dev)[0], _dev_weights(lq, fmt, Wn, cuda_dev), N, K, cuda_dev)
    _assert_self_consistent(v, i, c)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, Wn), N, K)
    check(c[None, :], y, tol, f"{fmt} {N}x{K} logits")
    i_ref = O.argmax_first(y[0])
    assert i == i_ref or y[0, i_ref] - y[0, i] <= tol[0, i_ref] + tol[0, i]


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_ties_go_to_the_lowest_row(lq, cuda_dev, fmt):
    """A dominant row copied to several places (bit-identical outputs): the
    lowest copy wins, in whichever CTA and stage it lands."""
    N, K = 5000, 1024
    W, A = synthetic.draw(1, N, K, seed=21)
    Wn = W.numpy().copy()
    top = (np.sign(A.numpy()[0]) * 0.05).astype(np.float32)
    for r in (4999, 1234, 37, 2500):
        Wn[r] = top
    v, i, c = _fused(lq, fmt, A.to(cuda_dev)[0], _dev_weights(lq, fmt, Wn, cuda_dev), N, K, cuda_dev)
    assert i == 37
    assert c[37] == c[1234] == c[2500] == c[4999]
    _assert_self_consistent(v, i, c)


@pytest.mark.parametrize("fmt", ["f16", "q8_0"])
def test_nan_never_wins(lq, cuda_dev, fmt):
    N, K = 3000, 512
    W, A = synthetic.draw(1, N, K, seed=22)
    Wn = W.numpy().copy()
    top = (np.sign(A.numpy()[0]) * 0.05).astype(np.float32)
    Wn[10] = top
    Wn[2000] = top
    packed = lq.pack(fmt, Wn)
    # row 10 gets a NaN (an element for f16, a block scale for Q8_0): its
    # output is NaN and the copy at 2000 must win
    if fmt == "f16":
        packed[10, 5] = F16_NAN
    else:
        packed[10, 34 * 3:34 * 3 + 2] = np.frombuffer(np.uint16(F16_NAN).tobytes(), np.uint8)
    Wd = to_dev(packed.reshape(-1).view(np.uint8), cuda_dev)
    v, i, c = _fused(lq, fmt, A.to(cuda_dev)[0], Wd, N, K, cuda_dev)
    assert np.isnan(c[10])
    assert i == 2000
    _assert_self_consistent(v, i, c)


def test_all_nan_gives_the_sentinel(lq, cuda_dev):
    N, K = 400, 256
    W, A = synthetic.draw(1, N, K, seed=23)
    packed = lq.pack("f16", W.numpy())
    packed[:, 17] = F16_NAN
    Wd = to_dev(packed.reshape(-1).view(np.uint8), cuda_dev)
    v, i, c = _fused(lq, "f16", A.to(cuda_dev)[0], Wd, N, K, cuda_dev)
    assert np.isnan(c).all()
    assert i == -1 and v == -np.inf


@pytest.mark.parametrize("fmt,K", [("q8_0", 96), ("f16", 20000), ("q4_0", 320)])
def test_unfused_fallback_outside_the_fast_path(lq, cuda_dev, fmt, K):
    """Shapes the streaming kernel does not take: GEMV into C, then the
    argmax of C; without C the call refuses."""
    N = 777
    W, A = synthetic.draw(1, N, K, seed=K)
    Wd = _dev_weights(lq, fmt, W.numpy(), cuda_dev)
    Ad = A.to(cuda_dev)[0]
    v, i, c = _fused(lq, fmt, Ad, Wd, N, K, cuda_dev)
    _assert_self_consistent(v, i, c)
    res = lq.argmax_result(cuda_dev)
    with pytest.raises(lq.LQError):
        lq.lq_gemv_argmax(fmt, Ad, Wd, None, N, K, res)


def test_forced_generic_route_agrees(lq, cuda_dev):
    fmt, N, K = "q8_0", 4096, 2048
    W, A = synthetic.draw(1, N, K, seed=24)
    Wd = _dev_weights(lq, fmt, W.numpy(), cuda_dev)
    Ad = A.to(cuda_dev)[0]
    _, i_fast, c_fast = _fused(lq, fmt, Ad, Wd, N, K, cuda_dev)
    try:
        lq.force_route(lq.ROUTE_GENERIC)
        v, i, c = _fused(lq, fmt, Ad, Wd, N, K, cuda_dev)
    finally:
        lq.force_route(0)
    _assert_self_consistent(v, i, c)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    for j in (i, i_fast):
        i_ref = O.argmax_first(y[0])
        assert j == i_ref or y[0, i_ref] - y[0, j] <= tol[0, i_ref] + tol[0, j]


def _argmax_vec(lq, x, dev):
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)
    res = lq.argmax_result(dev)
    lq.lq_argmax_f32(xd, len(x), res)
    torch.cuda.synchronize()
    return lq.read_argmax(res)


@pytest.mark.parametrize("n", [1, 31, 1000, 1 << 20, 3_000_001])
def test_argmax_f32_random_with_ties_and_nan(lq, cuda_dev, n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n).astype(np.float32)
    if n > 10:
        m = np.float32(x.max() + 1)
        pos = np.sort(rng.choice(n, size=3, replace=False))
        x[pos] = m                                # tie: lowest of the three
        x[rng.choice(n, size=n // 10, replace=False)] = np.nan
        x[pos[0]] = m                             # keep the lowest one finite
    v, i = _argmax_vec(lq, x, cuda_dev)
    assert i == O.argmax_first(x)
    assert np.float32(v).tobytes() == x[i].tobytes()


def test_argmax_f32_special_values(lq, cuda_dev):
    nan, inf = np.nan, np.inf
    cases = [
        [-0.0, 0.0, -0.0],              # -0 and +0 are equal: the first
        [0.0, -0.0],
        [-inf, -inf, -inf],             # a real -inf beats "nothing"
        [nan, -inf, nan],
        [nan, nan, nan],                # nothing: the sentinel
        [1.0, inf, 2.0, inf],
        [-3.0, -1e-38, -1e-45, -2.0],   # subnormals
        [float(np.finfo(np.float32).max), inf, nan],
    ]
    for x in cases:
        x = np.array(x, dtype=np.float32)
        v, i = _argmax_vec(lq, x, cuda_dev)
        assert i == O.argmax_first(x), (x, i)
        if i < 0:
            assert v == -np.inf
        else:
            assert v == x[i] or (np.isnan(v) and np.isnan(x[i]))
