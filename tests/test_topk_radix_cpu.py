"""A CPU model of the radix selection of the top-k kernels (lq_topk.cu:
radix_topk_block), checked against a plain sort of the same keys and against
the oracle's top-k.

Each CTA holds keys of 64 bits (lq_argmax.cuh: make_key; 0 = NaN or no
entry). With more than 128 valid keys it looks for the k-th largest a byte at
a time from the top: a histogram of byte d among the keys whose higher bytes
equal the bytes found so far, then, counting bins from 255 down, the first
bin where the count reaches the number of keys still wanted; that byte is
appended and the count above it subtracted. It stops as soon as the keys at
or above the prefix (lower bytes zero), i.e. those taken so far plus the
bin, number at most 128 (at the last byte the bin is one key: keys are
unique). Those keys are gathered and each goes to the place given by its
rank among them (the number of gathered keys above it); places past k are
dropped, places past the gathered keys stay empty. A second round runs the
same selection over the first round's candidates.
"""
import numpy as np
import pytest

import oracle as O
from test_argmax_key_cpu import decode, make_key


def radix_select(keys, k, first_crossing=True, gather=128, strict_rank=True):
    """The model. Planted mistakes: first_crossing=False takes the nearest
    non-empty bin above the crossing (too high a prefix drops keys; a bin
    below would only gather more, which the ranking absorbs); strict_rank=False
    counts a key among those at or above itself."""
    valid = [int(x) for x in keys if int(x) != 0]
    threshold = 1
    if len(valid) > gather:
        prefix, remaining = 0, k
        for d in range(7, -1, -1):
            sh = 8 * d
            hist = [0] * 256
            for x in valid:
                if d == 7 or (x >> (sh + 8)) == (prefix >> (sh + 8)):
                    hist[(x >> sh) & 255] += 1
            above, done = 0, False
            for dig in range(255, -1, -1):
                if above + hist[dig] >= remaining:
                    if not first_crossing:
                        up = next((u for u in range(dig + 1, 256) if hist[u]), None)
                        if up is not None:
                            above -= sum(hist[dig + 1:up + 1])
                            dig = up
                    prefix |= dig << sh
                    remaining -= above
                    done = k - remaining + hist[dig] <= gather
                    break
                above += hist[dig]
            if done:
                break
        threshold = prefix
    gathered = [x for x in valid if x >= threshold]
    assert len(gathered) <= gather
    places = [0] * k
    for x in gathered:
        rank = sum(1 for y in gathered if (y > x if strict_rank else y >= x))
        if rank < k:
            places[rank] = x
    return [x for x in places if x]


def two_rounds(values, k, tile=4096):
    keys = make_key(values, np.arange(len(values)))
    cands = []
    for b in range(0, len(keys), tile):
        sel = radix_select(keys[b:b + tile], k)
        assert len(sel) == min(k, int(np.count_nonzero(keys[b:b + tile])))
        cands += sel + [0] * (k - len(sel))
    return radix_select(np.array(cands, dtype=np.uint64), k) if len(keys) > tile else radix_select(keys, k)


@pytest.mark.parametrize("n,k,kind", [(1000, 50, "normal"), (40000, 64, "normal"), (40000, 1, "ties"),
                                      (5000, 64, "ties"), (300, 64, "nan"), (20, 50, "normal"),
                                      (33000, 17, "big_ties"), (9000, 64, "normal"), (70000, 50, "normal")])
def test_radix_selection_equals_sort_and_oracle(n, k, kind):
    rng = np.random.default_rng(n + k)
    if kind == "normal":
        v = rng.standard_normal(n).astype(np.float32)
    elif kind == "ties":
        v = rng.integers(-2, 3, size=n).astype(np.float32)   # a few values, many equal keys' high words
    elif kind == "big_ties":
        v = rng.standard_normal(n).astype(np.float32)
        v[rng.choice(n, 3 * k, replace=False)] = np.float32(9.0)  # the top spread over both tiles
    else:
        v = rng.standard_normal(n).astype(np.float32)
        v[rng.choice(n, n - 30, replace=False)] = np.nan      # fewer valid keys than k
    got = two_rounds(v, k)
    keys = sorted((int(x) for x in make_key(v, np.arange(n)) if int(x) != 0), reverse=True)[:k]
    assert got == keys
    ov, oi = O.topk_first(v, k)
    dec = [decode(x) for x in got] + [(-np.inf, -1)] * (k - len(got))
    assert [i for _, i in dec] == list(oi)
    assert np.array_equal(np.array([x for x, _ in dec], dtype=np.float32), ov.astype(np.float32))


def test_radix_model_catches_planted_mistakes():
    # 40000 normal values: the top byte's bin holds ~900 keys, so the second
    # byte decides (the mistakes act there)
    rng = np.random.default_rng(5)
    v = rng.standard_normal(40000).astype(np.float32)
    keys = make_key(v, np.arange(len(v)))
    want = sorted((int(x) for x in keys), reverse=True)[:40]
    assert radix_select(keys, 40) == want
    assert radix_select(keys, 40, first_crossing=False) != want
    assert radix_select(keys, 40, strict_rank=False) != want
