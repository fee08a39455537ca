"""A CPU model of the small-M tensor-core GEMM's operand loads
(lq_gemm_small.cu: load_weights, load_a), run on rows packed by the oracle.

A stage piece holds, for the CTA's W rows, 256 K of each row: Q8_0 272 bytes
(8 blocks of 34), Q4_0 144 (8 of 18), f16 512 bytes as four 128-byte-swizzled
boxes (16-byte chunk c of row r stored at chunk c ^ (r % 8)); and the M rows
of A, 1 KB (256 f32) each. Lane (g, q) of a warp builds, for block bp, its
eight weights of W row g / 2 + 4 (g % 2) of the tile for f16, row g for the
block formats (MMA column g), and the eight A values of token g (and g + 8) that
go into two mma.m16n8k16: values 0..3 in the first (K slots 2q, 2q+1, 2q+8,
2q+9), values 4..7 in the second. The model decodes those words as the
kernel addresses them (little-endian 32-bit words, funnel shifts for the
blocks that start 2 bytes into a word) and checks:

* the weight and the activation a lane pairs in each K slot are the same
  element of the block, and every element of the block meets the MMA once;
* the decoded weights equal the oracle's dequantisation of that element;
* the loads the kernel documents as conflict-free are: every 32-bit load of
  a warp hits 32 different banks (or one word), and every 16-byte load's
  quarter-warps cover the 32 banks once.
"""
import numpy as np
import pytest

import oracle as O
import synthetic

ROWS = 8          # W rows of the model stage (one tile: lanes g = 0..7)


def _word(buf, addr):
    return int.from_bytes(bytes(buf[addr:addr + 4]), "little")


def _funnel(lo, hi, sh):
    return ((hi << 32 | lo) >> sh) & 0xFFFFFFFF


def _f16(bits):
    return float(O.f16_bits_to_f32(np.array([bits & 0xFFFF], dtype=np.uint16))[0])


class Loads:
    """Records the byte address of each of one lane's loads, by load instruction."""

    def __init__(self):
        self.ops = {}

    def add(self, key, addr, size):
        self.ops[key] = (addr, size)


def stage_bytes(fmt, wq, piece):
    """The piece's W rows as the kernel's tensor-map boxes lay them out."""
    if fmt == "f16":
        w16 = wq.view(np.uint16).reshape(ROWS, -1)[:, 256 * piece:256 * (piece + 1)]
        buf = np.zeros(4 * ROWS * 128, np.uint8)
        for box in range(4):
            for r in range(ROWS):
                row = w16[r, 64 * box:64 * (box + 1)].view(np.uint8)
                for c in range(8):
                    dst = box * ROWS * 128 + r * 128 + ((c ^ (r % 8)) << 4)
                    buf[dst:dst + 16] = row[16 * c:16 * c + 16]
        return buf
    per = 272 if fmt == "q8_0" else 144
    rows = wq.reshape(ROWS, -1)
    return np.concatenate([rows[r, per * piece:per * (piece + 1)] for r in range(ROWS)] +
                          [np.zeros(8, np.uint8)])  # the ring's tail behind the last row


def load_weights(fmt, big, buf, row, bp, q, rec):
    """The lane's 8 weights as (value, element of the block) pairs, in order."""
    out = []
    if fmt == "f16":
        c = ((bp & 1) * 4 + q) ^ (row & 7)
        addr = (bp >> 1) * ROWS * 128 + row * 128 + (c << 4)
        rec.add("w128", addr, 16)
        h = buf[addr:addr + 16].view(np.uint16)
        for j in range(8):
            out.append((_f16(int(h[j])), 8 * q + j))
        return out
    if fmt == "q8_0":
        rowa = row * 272
        mis = bp % 2 == 0
        sh = 16 if mis else 0
        d = _word(buf, rowa + ((34 * bp) & ~3))
        d = _f16(d if mis else d >> 16)
        if big:
            o = 34 * bp + 2 + 4 * q
            wa = rowa + (o & ~3)
            groups = [(wa, wa + 4, 4 * q), (wa + 16, wa + 20, 16 + 4 * q)]
            for k, (a0, a1, e0) in enumerate(groups):
                rec.add(f"w{k}a", a0, 4)
                if mis:
                    rec.add(f"w{k}b", a1, 4)
            xs = [(_funnel(_word(buf, a0), _word(buf, a1) if mis else 0, sh), e0) for a0, a1, e0 in groups]
        else:
            o = 34 * bp + 2 + 8 * q
            wa = rowa + (o & ~3)
            w = [_word(buf, wa), _word(buf, wa + 4), _word(buf, wa + 8) if mis else 0]
            xs = [(_funnel(w[0], w[1], sh), 8 * q), (_funnel(w[1], w[2], sh), 8 * q + 4)]
        for x, e0 in xs:
            x ^= 0x80808080
            for i in range(4):
                code = ((x >> (8 * i)) & 0xFF) - 128
                out.append((float(np.float32(code) * np.float32(d)), e0 + i))
        return out
    rowa = row * 144
    mis = bp % 2 == 0
    o = 18 * bp + 2 + 4 * q
    wa = rowa + (o & ~3)
    rec.add("w0", wa, 4)
    if mis:
        rec.add("w1", wa + 4, 4)
    x = _funnel(_word(buf, wa), _word(buf, wa + 4) if mis else 0, 16 if mis else 0)
    d = _word(buf, rowa + ((18 * bp) & ~3))
    d = _f16(d if mis else d >> 16)
    for half, e0 in ((x & 0x0F0F0F0F, 4 * q), ((x >> 4) & 0x0F0F0F0F, 16 + 4 * q)):
        for i in range(4):
            code = ((half >> (8 * i)) & 0xFF) - 8
            out.append((float(np.float32(code) * np.float32(d)), e0 + i))
    return out


def load_a(fmt, big, arow_elems, row, bp, q, rec):
    """The lane's 8 A values of token `row` as elements of block bp, in order."""
    quarters = fmt == "q4_0" or (fmt == "q8_0" and big)
    c0, c1 = (q, 4 + q) if quarters else (2 * q, 2 * q + 1)
    odd = big and row % 2 == 1
    first, second = (c1, c0) if odd else (c0, c1)
    base = row * 1024 + bp * 128
    rec.add("a0", base + (first << 4), 16)
    rec.add("a1", base + (second << 4), 16)
    x = [32 * bp + 4 * first + i for i in range(4)]
    y = [32 * bp + 4 * second + i for i in range(4)]
    p = [x[0:2], x[2:4], y[0:2], y[2:4]]
    a = [p[2], p[3], p[0], p[1]] if odd else p
    return [arow_elems[e] for pair in a for e in pair]


def banks_ok(op, size):
    """Conflict-free: 32-bit loads hit 32 different banks (or share words);
    16-byte loads cover each bank once per quarter-warp."""
    lanes = sorted(op)
    if size == 4:
        words = {}
        for ln in lanes:
            a, _ = op[ln]
            words.setdefault((a // 4) % 32, set()).add(a // 4)
        return all(len(w) == 1 for w in words.values())
    for qw in range(4):
        banks = []
        for ln in lanes[8 * qw:8 * qw + 8]:
            a, _ = op[ln]
            banks += [(a // 4 + i) % 32 for i in range(4)]
        if len(set(banks)) != len(banks):
            return False
    return True


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("big", [False, True])
def test_small_kernel_lanes_pair_the_same_elements(fmt, big):
    K = 512
    W, _ = synthetic.draw(1, ROWS, K, seed=11, outlier_frac=0.05)
    W = W.numpy()
    wq = O.pack(fmt, W)
    deq = O.dequantize(fmt, wq, ROWS, K)
    for piece in range(K // 256):
        buf = stage_bytes(fmt, wq, piece)
        for bp in range(8):
            recs = {}
            seen = {g: [] for g in range(ROWS)}
            for lane in range(32):
                g, q = lane // 4, lane % 4
                wr = g // 2 + 4 * (g % 2) if fmt == "f16" else g
                rec = Loads()
                ws = load_weights(fmt, big, buf, wr, bp, q, rec)
                elems = list(range(256))
                tok = load_a(fmt, big, elems, g, bp, q, rec)
                # same element of the block in every K slot
                assert [e for _, e in ws] == [e - 32 * bp for e in tok], (fmt, big, bp, lane)
                for v, e in ws:
                    assert v == float(deq[wr, 256 * piece + 32 * bp + e]), (fmt, big, bp, lane, e)
                seen[wr] += [e for _, e in ws]
                for key, (a, sz) in rec.ops.items():
                    recs.setdefault(key, {})[lane] = (a, sz)
            for g in range(ROWS):
                assert sorted(seen[g]) == list(range(32)), (fmt, big, bp, g)
            # conflict-free where the kernel claims it
            for key, op in recs.items():
                size = next(iter(op.values()))[1]
                if key.startswith("a"):
                    assert banks_ok(op, size) == big, (fmt, big, key)
                elif fmt == "q8_0" and not big:
                    continue  # two lanes a bank, as documented
                else:
                    assert banks_ok(op, size), (fmt, big, bp, key)


def test_small_kernel_model_catches_a_wrong_pairing():
    """A planted mistake: Q8_0 with BIG codes but the A chunks of the 8q
    layout pairs different elements."""
    K = 256
    W, _ = synthetic.draw(1, ROWS, K, seed=3)
    wq = O.pack("q8_0", W.numpy())
    buf = stage_bytes("q8_0", wq, 0)
    rec = Loads()
    ws = load_weights("q8_0", True, buf, 1, 2, 1, rec)
    tok = load_a("q8_0", False, list(range(256)), 1, 2, 1, rec)
    assert [e for _, e in ws] != [e - 64 for e in tok]


def test_small_kernel_model_catches_conflicting_rows():
    """A planted mistake: MMA column g on W row g puts a quarter-warp's two
    f16 rows in the same half of the swizzle (two lanes a bank)."""
    K = 256
    W, _ = synthetic.draw(1, ROWS, K, seed=5)
    wq = O.pack("f16", W.numpy())
    buf = stage_bytes("f16", wq, 0)
    op = {}
    for lane in range(32):
        rec = Loads()
        load_weights("f16", True, buf, lane // 4, 0, lane % 4, rec)
        op[lane] = rec.ops["w128"]
    assert not banks_ok(op, 16)
