"""A CPU model of the M = 1 GEMV slices' block dots (lq_gemv_slices.cuh:
Q8Slice::dot, Q4Slice::dot), run on rows packed by the oracle and checked
against the oracle's dequantised blocks.

Lane l of K-group kg (nk K-groups, two per 64-block segment) takes block
b = 64*seg + 2l + parity with seg = kg/2 (+ nk/2 per further chunk) and
parity = kg % 2. Its bytes start at byte woff of the row: Q8_0 2176*seg +
68l (+32 for odd blocks), Q4_0 1152*seg + 36l (+16), read as little-endian
32-bit words. The scale is the low half of word 0 (even blocks) or the high
half (odd); each word of codes is the funnel shift of words i, i+1 by 16 bits
(even) or 32 (odd: word i+1 as is). Q8_0 codes are bytes with their sign bit
flipped, Q4_0 codes the bytes of (x & 0x0F0F0F0F) and ((x >> 4) & 0x0F0F0F0F);
each goes into the low mantissa byte of 2^23 and the bias comes off with one
exact subtraction. The products here are summed in float64: the model checks
which codes and activations meet, not the order of the f32 sums. For Q4_0 with
interleaved nibbles the same dot runs on A reordered per block as the
kernels spread it (lq_q4i.cuh).
"""
import numpy as np
import pytest

import oracle as O
import synthetic


def _words(row, off, n):
    return [int.from_bytes(bytes(row[off + 4 * i: off + 4 * i + 4]), "little") for i in range(n)]


def _funnel(lo, hi, sh):
    return ((hi << 32 | lo) >> sh) & 0xFFFFFFFF if sh < 32 else hi


def _magic(byte_value, bias):
    # the float 2^23 + byte, minus the bias, in float32 as the kernels do
    return float(np.float32(np.float32(8388608.0 + byte_value) - np.float32(bias)))


def _f16(bits):
    return float(O.f16_bits_to_f32(np.array([bits & 0xFFFF], dtype=np.uint16))[0])


def q8_block_dot(row, a, kg, lane, shift_even=16):
    seg, par = kg >> 1, kg & 1
    b = 64 * seg + 2 * lane + par
    w = _words(row, 2176 * seg + 68 * lane + (32 if par else 0), 9)
    d = _f16(w[0] >> 16 if par else w[0])
    sh = 32 if par else shift_even
    total = 0.0
    for i in range(8):
        x = _funnel(w[i], w[i + 1], sh) ^ 0x80808080
        for j in range(4):
            q = _magic((x >> (8 * j)) & 0xFF, 8388608.0 + 128.0)
            total += q * float(a[32 * b + 4 * i + j])
    return b, d * total


def q4_block_dot(row, a, kg, lane, woff_step=36):
    seg, par = kg >> 1, kg & 1
    b = 64 * seg + 2 * lane + par
    w = _words(row, 1152 * seg + woff_step * lane + (16 if par else 0), 5)
    d = _f16(w[0] >> 16 if par else w[0])
    sh = 32 if par else 16
    total = 0.0
    for i in range(4):
        x = _funnel(w[i], w[i + 1], sh)
        lo, hi = x & 0x0F0F0F0F, (x >> 4) & 0x0F0F0F0F
        for j in range(4):
            total += _magic((lo >> (8 * j)) & 0xFF, 8388608.0 + 8.0) * float(a[32 * b + 4 * i + j])
            total += _magic((hi >> (8 * j)) & 0xFF, 8388608.0 + 8.0) * float(a[32 * b + 16 + 4 * i + j])
    return b, d * total


def _oracle_block_dots(fmt, row_packed, a, K):
    w = O.dequantize(fmt, row_packed[None, :], 1, K)[0].astype(np.float64)
    return (w.reshape(-1, 32) * a.reshape(-1, 32).astype(np.float64)).sum(axis=1)


@pytest.mark.parametrize("fmt,dot", [("q8_0", q8_block_dot), ("q4_0", q4_block_dot)])
@pytest.mark.parametrize("K", [2048, 4096])
def test_every_lane_reads_its_own_block(fmt, dot, K):
    W, A = synthetic.draw(1, 3, K, seed=K, outlier_frac=0.1)
    packed = O.pack(fmt, W.numpy())
    a = A.numpy()[0]
    nk = 2 * ((K // 32 + 63) // 64)
    for r in range(3):
        row = packed[r]
        want = _oracle_block_dots(fmt, row, a, K)
        seen = set()
        for kg in range(nk):
            for lane in range(32):
                b, got = dot(row, a, kg, lane)
                seen.add(b)
                assert abs(got - want[b]) <= 1e-9 * (1 + abs(want[b])), (fmt, K, r, kg, lane, b)
        assert seen == set(range(K // 32))  # every block exactly once over the warps


def test_planted_even_shift_is_caught():
    """Aligning even blocks by 8 bits instead of 16 reads the scale's high
    byte as a code: the model must disagree with the oracle."""
    K = 2048
    W, A = synthetic.draw(1, 1, K, seed=5)
    row = O.pack("q8_0", W.numpy())[0]
    a = A.numpy()[0]
    want = _oracle_block_dots("q8_0", row, a, K)
    bad = [abs(q8_block_dot(row, a, 0, lane, shift_even=8)[1] - want[2 * lane]) > 1e-6 for lane in range(32)]
    assert any(bad)


def test_planted_q4_lane_stride_is_caught():
    """A Q4_0 lane stride of 34 bytes (the Q8_0 habit of 2 x 17) instead of
    36 misplaces every lane after the first."""
    K = 2048
    W, A = synthetic.draw(1, 1, K, seed=6)
    row = O.pack("q4_0", W.numpy())[0]
    a = A.numpy()[0]
    want = _oracle_block_dots("q4_0", row, a, K)
    bad = [abs(q4_block_dot(row, a, 0, lane, woff_step=34)[1] - want[2 * lane]) > 1e-6 for lane in range(1, 32)]
    assert any(bad)


def _q4i_store_chunks(a_block):
    """The kernels' spread of one block's 32 activations for interleaved
    Q4_0 (lq_q4i.cuh, store_chunk): 16-byte chunk i (elements 4i .. 4i+3)
    puts elements 4i, 4i+2 at slots 2i, 2i+1 and 4i+1, 4i+3 at slots
    16+2i, 17+2i."""
    out = np.empty(32, dtype=a_block.dtype)
    for i in range(8):
        x, y, z, w = a_block[4 * i: 4 * i + 4]
        out[2 * i], out[2 * i + 1] = x, z
        out[16 + 2 * i], out[17 + 2 * i] = y, w
    return out


def test_q4_0i_reordered_activations_give_the_interleaved_product():
    """Slot j of a block = element 2j, slot 16+j = element 2j+1 (slot_of);
    the standard-order Q4_0 dot on interleaved bytes and reordered A must
    equal the oracle's interleaved dequantisation times the original A."""
    for e in range(32):
        slot = (16 + (e >> 1)) if (e & 1) else (e >> 1)
        assert _q4i_store_chunks(np.arange(32))[slot] == e
    K = 2048
    W, A = synthetic.draw(1, 2, K, seed=8, outlier_frac=0.1)
    packed = O.pack("q4_0i", W.numpy())
    a = A.numpy()[0]
    a_perm = np.concatenate([_q4i_store_chunks(blk) for blk in a.reshape(-1, 32)])
    for r in range(2):
        row = packed[r]
        want = _oracle_block_dots("q4_0i", row, a, K)
        for kg in range(2 * ((K // 32 + 63) // 64)):
            for lane in range(32):
                b, got = q4_block_dot(row, a_perm, kg, lane)
                assert abs(got - want[b]) <= 1e-9 * (1 + abs(want[b])), (r, kg, lane, b)
        # and without the reorder the standard dot does not give it
        b, plain = q4_block_dot(row, a, 0, 0)
        assert abs(plain - want[b]) > 1e-6
