"""A CPU model of how the small-M tensor-core GEMM (lq_gemm_small.cu:
gemm_small_kernel) splits a CTA's work over its 16 warps and adds the warps'
partial tiles, for both stage shapes.

A stage holds PPS pieces of 256 K (PPS = 2 up to 32 rows of A, 1 beyond);
a piece is 8 blocks of 32 K; the CTA's W rows form T tiles of 8 rows, taken
in pairs (NP pairs, the last one repeating its first tile when T is odd).
With PPS = 2 warp w takes block w % 8 of piece w / 8 of every stage for all
pairs and writes its partial tiles at position w (16 positions); with PPS = 1
warp w takes block w % 8 of the stage's piece for pairs w / 8, w / 8 + 2, ...
and writes at position w % 8 (8 positions). The final sum adds a tile's
positions in order.

The model checks, for every tile of the CTA, that each (piece, block) of K
reaches the sum exactly once, that no two warps write the same position of a
tile, that every stage's pieces land in distinct regions of the slot (A of
piece 0, A of piece 1, then W of piece 0, W of piece 1), and that planted
mistakes in the split are caught.
"""
import itertools

import pytest

WARPS, BLOCKS = 16, 8


def split(pps, NP, T, npieces, pair_stride=2, pos_mode="kernel"):
    """{(tile, position): [(piece, block), ...]} as the kernel stores them."""
    npa = NP if pps == 2 else (NP + 1) // 2
    nstages = (npieces + pps - 1) // pps
    red = {}
    for w in range(WARPS):
        bp, sp, half = w & 7, (w >> 3 if pps == 2 else 0), w >> 3
        acc = {}
        for st in range(nstages):
            if pps * st + sp >= npieces:
                continue
            piece = pps * st + sp
            for m in range(npa):
                pr = m if pps == 2 else half + pair_stride * m
                if pps == 1 and pr >= NP:
                    break
                t0, t1 = 2 * pr, min(2 * pr + 1, T - 1)
                acc.setdefault(2 * m, []).append((t0, piece, bp))
                acc.setdefault(2 * m + 1, []).append((t1, piece, bp))
        pos = w if pps == 2 else (bp if pos_mode == "kernel" else w)
        for m in range(npa):
            pr = m if pps == 2 else half + pair_stride * m
            if pps == 1 and pr >= NP:
                break
            for h2 in range(2):
                t = 2 * pr + h2
                if t < T:
                    key = (t, pos)
                    assert all(tt == t for tt, _, _ in acc.get(2 * m + h2, [])), "accumulator mixes tiles"
                    red.setdefault(key, []).append([(pc, b) for _, pc, b in acc.get(2 * m + h2, [])])
    return red


def covered(red, T, npieces, npos):
    """Every tile's sum over positions 0 .. npos-1 holds each (piece, block) once,
    and no position was written twice."""
    for (t, pos), writes in red.items():
        if len(writes) != 1 or pos >= npos:
            return False
    for t in range(T):
        got = []
        for pos in range(npos):
            got += red.get((t, pos), [[]])[0]
        if sorted(got) != [(pc, b) for pc in range(npieces) for b in range(BLOCKS)]:
            return False
    return True


@pytest.mark.parametrize("pps", [1, 2])
@pytest.mark.parametrize("NP", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("odd", [False, True])
@pytest.mark.parametrize("npieces", [1, 2, 3, 8, 17])
def test_every_piece_and_block_reaches_each_tile_once(pps, NP, odd, npieces):
    if pps == 1 and NP > 4:
        pytest.skip("single-piece stages take at most 4 pairs (48 W rows, three token groups)")
    T = 2 * NP - (1 if odd else 0)
    red = split(pps, NP, T, npieces)
    assert covered(red, T, npieces, 8 * pps)


def test_slot_regions_are_disjoint():
    """Stage slot layout: A of each piece (M rows of 1 KB), then W of each
    piece (w_pitch apart, w_pitch at least the piece's W bytes)."""
    kA = 1024
    for pps, M, w_bytes in itertools.product([1, 2], [2, 17, 33, 48], [41 * 272, 64 * 512, 48 * 144]):
        w_pitch = (w_bytes + 127) // 128 * 128
        regions = []
        for sp in range(pps):
            regions.append((sp * M * kA, (sp + 1) * M * kA))                     # A of piece sp
            w0 = pps * M * kA + sp * w_pitch
            regions.append((w0, w0 + w_bytes))                                   # W of piece sp
        regions.sort()
        assert all(a1 <= b0 for (_, a1), (b0, _) in zip(regions, regions[1:])), (pps, M, w_bytes)


def test_split_model_catches_planted_mistakes():
    # pairs w / 8, w / 8 + 1, ... with single-piece stages: two warps share pairs
    assert not covered(split(1, 4, 8, 8, pair_stride=1), 8, 8, 8)
    # positions by warp instead of block with single-piece stages: 16 positions,
    # of which the sum reads only 8
    assert not covered(split(1, 3, 6, 8, pos_mode="warp"), 6, 8, 8)
    # the sum over 8 positions with two-piece stages misses the odd pieces
    assert not covered(split(2, 2, 4, 8), 4, 8, 8)
