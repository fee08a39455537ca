"""A CPU model of the 64-bit candidate keys of the argmax and top-k kernels
(lq_argmax.cuh: make_key, decode), checked against the oracle's order.

The key of (v, i): high word the f32 bits of v + 0 (so -0 becomes +0) mapped
to an unsigned order (negative values bit-flipped, others with the sign bit
set), low word 0xFFFFFFFF - i; NaN has key 0. The largest key must be the
oracle's best candidate (larger value first, equal values by the lower index,
NaN never), and the top keys in order its top-k.
"""
import numpy as np
import pytest

import oracle as O


def make_key(v, idx):
    v = np.asarray(v, dtype=np.float32)
    idx = np.asarray(idx, dtype=np.uint64)
    u = (v + np.float32(0.0)).view(np.uint32).astype(np.uint64)
    hi = np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000)
    key = (hi << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - idx)
    return np.where(np.isnan(v), np.uint64(0), key).astype(np.uint64)


def decode(key):
    key = int(key)
    if key == 0:
        return -np.inf, -1
    hi, lo = key >> 32, key & 0xFFFFFFFF
    u = (hi & 0x7FFFFFFF) if (hi & 0x80000000) else (~hi & 0xFFFFFFFF)
    return float(np.uint32(u).view(np.float32)), 0xFFFFFFFF - lo


def _values(rng, n, kind):
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "ties":
        return rng.integers(-3, 3, size=n).astype(np.float32)
    if kind == "specials":
        pool = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 3.4e38, -3.4e38, 1.0, -1.0],
                        dtype=np.float32)
        return pool[rng.integers(0, len(pool), size=n)]
    if kind == "all nan":
        return np.full(n, np.nan, dtype=np.float32)
    return np.full(n, -np.inf, dtype=np.float32)


@pytest.mark.parametrize("kind", ["normal", "ties", "specials", "all nan", "all -inf"])
def test_largest_key_is_the_oracle_argmax(kind):
    rng = np.random.default_rng(4)
    for n in (1, 2, 37, 1000):
        x = _values(rng, n, kind)
        keys = make_key(x, np.arange(n))
        best = keys.max()
        v, i = decode(best)
        assert i == O.argmax_first(x)
        if i >= 0:
            assert v == x[i] or (v == 0.0 and x[i] == 0.0)  # -0 comes back as +0


@pytest.mark.parametrize("kind", ["normal", "ties", "specials"])
def test_key_order_is_the_oracle_top_k(kind):
    rng = np.random.default_rng(5)
    x = _values(rng, 500, kind)
    keys = make_key(x, np.arange(500))
    order = np.argsort(keys, kind="stable")[::-1]
    k = 40
    vals, idx = O.topk_first(x, k)
    real = keys[order[:k]] != 0
    assert np.array_equal(order[:k][real], idx[idx >= 0])


def test_every_real_candidate_beats_nan_and_nothing():
    x = np.array([-np.inf, np.nan, -np.inf], dtype=np.float32)
    keys = make_key(x, np.array([0, 1, 0xFFFFFFFE]))
    assert keys[1] == 0 and keys[0] > 0 and keys[2] > 0
    assert decode(0) == (-np.inf, -1)
