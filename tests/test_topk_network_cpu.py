"""A CPU model of the top-k kernel's selection network (lq_topk.cu: cx_step,
top64_desc, running_topk), step for step over its 1024 threads, checked
against a plain sort.

Thread t holds positions 2t and 2t + 1 of the 2048 keys (warp w = t / 32 holds
the run 64w .. 64w + 63). A shuffle with lane mask m reaches thread t ^ m. The
network first sorts every run of 64 (even runs descending, odd ascending),
then five rounds each take, in warp w a multiple of 2^(r+1), the elementwise
maximum of its run and the run of warp w + 2^r (read through shared memory)
and sort that bitonic run in the direction the next round needs. The best 64
keys end in positions 0 .. 63, descending.
"""
import numpy as np
import pytest

THREADS = 1024
T = np.arange(THREADS)
P0 = 2 * T                 # each thread's even position
WARP = T >> 5


def cx_step(e, p, stride, desc, active):
    """One compare-exchange step on the threads in `active`."""
    e = e.copy()
    if stride == 1:
        swap = active & np.where(desc, e[:, 0] < e[:, 1], e[:, 0] > e[:, 1])
        e[swap] = e[swap][:, ::-1]
        return e
    q = e[T ^ (stride >> 1)]
    keep_max = ((p & stride) == 0) == desc
    new = np.where(keep_max[:, None], np.maximum(e, q), np.minimum(e, q))
    return np.where(active[:, None], new, e)


def top64_desc(s, round_dir=None):
    """s: 2048 uint64 keys; returns s with its best 64 keys first, descending.
    round_dir plants a different direction rule for the rounds (tests only)."""
    s = s.copy()
    e = np.stack([s[P0], s[P0 + 1]], axis=1)
    every = np.ones(THREADS, dtype=bool)
    for ls in range(1, 7):
        for lst in range(ls - 1, -1, -1):
            stride = 1 << lst
            desc = ((P0 & ~stride) & (1 << ls)) == 0
            e = cx_step(e, P0, stride, desc, every)
    for r in range(5):
        s[P0], s[P0 + 1] = e[:, 0], e[:, 1]
        active = (WARP & ((2 << r) - 1)) == 0
        q = P0 + (64 << r)
        q = np.where(active, q, 0)           # inactive threads read nothing
        b = np.stack([s[q], s[q + 1]], axis=1)
        e = np.where(active[:, None], np.maximum(e, b), e)
        desc = ((WARP >> (r + 1)) & 1) == 0 if round_dir is None else round_dir(WARP, r)
        for lst in range(5, -1, -1):
            e = cx_step(e, P0 & 63, 1 << lst, desc, active)
    first = WARP == 0
    s[P0[first]], s[P0[first] + 1] = e[first, 0], e[first, 1]
    return s


def running_topk(keys, k=64):
    """The kernel's running top-64 over tiles of 1984 new keys."""
    s = np.zeros(2048, dtype=np.uint64)
    for base in range(0, len(keys), 1984):
        tile = keys[base:base + 1984]
        s[64:] = 0
        s[64:64 + len(tile)] = tile
        s = top64_desc(s)
    return s[:k]


def _keys(rng, n, kind):
    if kind == "random":
        return rng.integers(0, 2**63, size=n, dtype=np.uint64) * np.uint64(2) + rng.integers(0, 2, size=n, dtype=np.uint64)
    if kind == "few values":
        return rng.integers(0, 8, size=n).astype(np.uint64)
    if kind == "zeros":
        return np.zeros(n, dtype=np.uint64)
    if kind == "ascending":
        return np.arange(n, dtype=np.uint64)
    return np.arange(n, dtype=np.uint64)[::-1].copy()


@pytest.mark.parametrize("kind", ["random", "few values", "zeros", "ascending", "descending"])
def test_top64_of_one_tile_matches_a_sort(kind):
    rng = np.random.default_rng(1)
    for _ in range(3):
        s = _keys(rng, 2048, kind)
        got = top64_desc(s)[:64]
        assert np.array_equal(got, np.sort(s)[::-1][:64])


@pytest.mark.parametrize("n", [1, 63, 64, 1984, 1985, 5000, 9921])
def test_running_top64_over_tiles_matches_a_sort(n):
    rng = np.random.default_rng(n)
    keys = _keys(rng, n, "random")
    want = np.zeros(64, dtype=np.uint64)
    top = np.sort(keys)[::-1][:64]
    want[:len(top)] = top                    # fewer than 64 keys: the rest stay 0 (no candidate)
    assert np.array_equal(running_topk(keys), want)


def test_planted_round_direction_is_caught():
    """Sorting every round's run descending (ignoring the direction the next
    round needs) breaks the half-cleaner's bitonic input."""
    rng = np.random.default_rng(3)
    wrong = 0
    for _ in range(5):
        s = _keys(rng, 2048, "random")
        got = top64_desc(s, round_dir=lambda w, r: np.ones_like(w, dtype=bool))[:64]
        wrong += not np.array_equal(got, np.sort(s)[::-1][:64])
    assert wrong > 0
