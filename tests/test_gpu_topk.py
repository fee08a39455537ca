"""lq_topk_f32 and lq_gemv_topk against the oracle's topk_first (inputs up to
4 Mi entries take the radix selection, larger ones the sorting passes).

The order is decided in f32 on both sides: the oracle ranks the GPU's own
float32 inputs (or logits), so indices must agree exactly and values bit for
bit. Ties are planted, NaN inserted, and k runs from 1 to the limit 64,
including more than the non-NaN entries (sentinels)."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _topk(lq, x, k, dev):
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)
    v, i, w = lq.topk_buffers(len(x), k, dev)
    lq.lq_topk_f32(xd, len(x), k, v, i, w)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return v.cpu().numpy(), i.cpu().numpy()


def _expect(x, k):
    v, i = O.topk_first(np.asarray(x, dtype=np.float32), k)
    return v.astype(np.float32), i


@pytest.mark.parametrize("n,k", [(1, 1), (5, 9), (1000, 1), (1000, 64), (151936, 50), (1 << 20, 40),
                                 (3_000_001, 64), (1985, 17), (3968, 64), (4096, 64), (4097, 33),
                                 ((1 << 22) + 1, 50)])  # past 4 Mi entries: the sorting passes
def test_topk_random_with_ties_and_nan(lq, cuda_dev, n, k):
    rng = np.random.default_rng(n + k)
    x = rng.standard_normal(n).astype(np.float32)
    if n > 20:
        x[rng.choice(n, n // 20, replace=False)] = np.nan
        top = np.float32(np.nanmax(x) + 1)
        x[rng.choice(n, min(n // 4, 2 * k), replace=False)] = top  # ties across tiles and CTAs
        x[rng.choice(n, 3, replace=False)] = -np.inf
    v, i = _topk(lq, x, k, cuda_dev)
    ev, ei = _expect(x, k)
    assert list(i) == list(ei)
    assert np.array_equal(v.view(np.uint32), ev.view(np.uint32)) or np.array_equal(v, ev)


def test_topk_all_nan_and_special_values(lq, cuda_dev):
    v, i = _topk(lq, np.full(300, np.nan, np.float32), 4, cuda_dev)
    assert list(i) == [-1] * 4 and np.all(np.isneginf(v))
    x = np.array([0.0, -0.0, 1.0, np.nan, -0.0, np.inf, -np.inf], np.float32)
    v, i = _topk(lq, x, 7, cuda_dev)
    assert list(i) == list(_expect(x, 7)[1])


def test_topk_k1_equals_argmax(lq, cuda_dev):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32)
    x[rng.choice(200000, 7, replace=False)] = np.float32(10.0)
    v, i = _topk(lq, x, 1, cuda_dev)
    assert i[0] == O.argmax_first(x) and v[0] == 10.0


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_gemv_topk_lm_head_shape(lq, cuda_dev, fmt):
    N, K, k = 151936 if fmt == "f16" else 32000, 2048, 50
    W, A = synthetic.draw(1, N, K, seed=3)
    Wd = to_dev(lq.pack(fmt, W.numpy()).reshape(-1).view(np.uint8), cuda_dev)
    C = nan_filled(1, N, cuda_dev)[0]
    v, i, w = lq.topk_buffers(N, k, cuda_dev)
    lq.lq_gemv_topk(fmt, A.to(cuda_dev)[0], Wd, C, N, K, k, v, i, w)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    c = C.cpu().numpy()
    ev, ei = _expect(c, k)
    assert list(i.cpu().numpy()) == list(ei)
    assert np.array_equal(v.cpu().numpy(), ev)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    check(c[None, :], y, tol, f"{fmt} logits")
