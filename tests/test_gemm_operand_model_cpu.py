"""A CPU model of the tensor-core GEMM's bf16 operands (lq_gemm_tma.cu: the
a_to_bf16_kernel pre-pass and the converters), pinning the numerical facts
the kernels rely on.

A: every value is rounded to bf16 to nearest even, the same rounding the
tolerance of the tensor-core path is defined on. bf16 keeps f32's exponent
range, so the operand is within 2^-8 |a| of a (the unit roundoff of an 8-bit
significand) for every f32-normal a, with no absolute term (no range of
values loses relative precision), and equals the oracle's rounding bit for
bit.

W: a code byte goes into the low mantissa byte of 2^23 (a float equal to
2^23 + byte), one f32 add takes the bias 2^23 + 128 (Q8_0, whose code has
its sign bit flipped) or 2^23 + 8 (Q4_0) off exactly, and one f32 multiply
by the widened f16 scale is exact (an 11-bit significand times a code of at
most 8 bits). f16 weights widen exactly. Rounding that exact f32 value to
bf16 once gives the weight within 2^-8 of its value, for every block scale
f16 can hold: there is no range limit on this route. The products' error is
then at most 2^-8 sum|a w| (3.9e-3) plus the f32 summation, inside the
tolerance of 5e-3 sum|a w| + 1e-5.
"""
import numpy as np

import oracle as O

MAGIC = np.float32(2.0 ** 23)


def bf16_rne_bits(x):
    """Round f32 values to bf16 (nearest, ties to even) on their bit patterns,
    as cvt.rn.bf16x2.f32 does for finite inputs: the kernel model."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def magic_float(byte):
    """The float whose bits are 0x4B0000 | byte: 2^23 + byte exactly."""
    return (np.uint32(0x4B000000) | np.uint32(byte)).view(np.float32)


def q8_weight(code, d_bits):
    """Converter for one Q8_0 code (int8) with block scale bits d_bits."""
    d = np.float32(np.uint16(d_bits).view(np.float16))
    byte = (int(code) & 0xFF) ^ 0x80                       # sign bit flipped: q + 128
    q = np.float32(magic_float(byte) - np.float32(MAGIC + np.float32(128.0)))  # exact
    w = np.float32(q * d)                                  # exact: 11 x 8 bits
    return w, bf16_rne_bits(w)


def q4_weight(nibble, d_bits):
    d = np.float32(np.uint16(d_bits).view(np.float16))
    q = np.float32(magic_float(int(nibble)) - np.float32(MAGIC + np.float32(8.0)))  # q - 8, exact
    w = np.float32(q * d)
    return w, bf16_rne_bits(w)


def _all_finite_f16_scales():
    b = np.arange(0, 0x7C00, dtype=np.uint32)        # +0 .. largest finite, subnormals included
    return np.concatenate([b, b | 0x8000]).astype(np.uint16)


def test_a_operand_relative_bound_without_absolute_term():
    rng = np.random.default_rng(0)
    # every f32 exponent of the normal range, random significands and signs
    e = rng.integers(-126, 128, 400000)
    a = (rng.uniform(1.0, 2.0, e.size) * np.exp2(e.astype(np.float64))).astype(np.float32)
    a *= np.where(rng.random(e.size) < 0.5, -1, 1).astype(np.float32)
    a = a[np.isfinite(a) & (np.abs(a) < np.float32(3.38e38))]   # rounding up past the largest bf16 -> inf
    h = bf16_value(bf16_rne_bits(a)).astype(np.float64)
    err = np.abs(h - a.astype(np.float64))
    assert np.all(err <= 2.0 ** -8 * np.abs(a.astype(np.float64)))
    # the row of the wide-range example: [1e6, 1e-4, ...] keeps every small term
    row = np.array([1e6] + [1e-4] * 2047, dtype=np.float32)
    hr = bf16_value(bf16_rne_bits(row)).astype(np.float64)
    assert np.all(np.abs(hr - row) <= 2.0 ** -8 * np.abs(row.astype(np.float64)))


def test_a_operand_equals_the_rounding_the_tolerance_is_defined_on():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 2000000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < np.float32(3.38e38))]
    model = bf16_value(bf16_rne_bits(x))
    oracle = O.f32_to_bf16_rne(x)
    assert np.array_equal(model.view(np.uint32), np.asarray(oracle, dtype=np.float32).view(np.uint32))


def test_q8_0_weights_formed_exactly_and_rounded_once_for_every_scale():
    scales = _all_finite_f16_scales()[::7]
    codes = np.arange(-127, 128)
    for d_bits in scales:
        d = float(np.uint16(d_bits).view(np.float16))
        for code in codes:
            w, hb = q8_weight(code, d_bits)
            exact = float(code) * d
            assert float(w) == exact                               # exact in f32
            assert hb == bf16_rne_bits(np.float32(exact))          # one rounding
            assert abs(float(bf16_value(hb)) - exact) <= 2.0 ** -8 * abs(exact)


def test_q4_0_weights_formed_exactly_and_rounded_once_for_every_scale():
    scales = _all_finite_f16_scales()[::5]
    for d_bits in scales:
        d = float(np.uint16(d_bits).view(np.float16))
        for nib in range(16):
            w, hb = q4_weight(nib, d_bits)
            exact = float(nib - 8) * d
            assert float(w) == exact
            assert abs(float(bf16_value(hb)) - exact) <= 2.0 ** -8 * abs(exact)


def test_f16_weights_widen_exactly_and_round_once():
    h = _all_finite_f16_scales()
    f = h.view(np.float16).astype(np.float32)           # exact widening
    got = bf16_value(bf16_rne_bits(f)).astype(np.float64)
    assert np.all(np.abs(got - f.astype(np.float64)) <= 2.0 ** -8 * np.abs(f.astype(np.float64)))


def test_largest_block_scales_stay_finite():
    """The weights of f16's largest scale: Q8_0 127 * 65504, Q4_0 -8 * 65504."""
    top = np.uint16(0x7BFF)                               # 65504
    for code in (-127, 127):
        w, hb = q8_weight(code, top)
        assert np.isfinite(bf16_value(hb)) and abs(float(w)) == 127 * 65504.0
    w, hb = q4_weight(0, top)
    assert np.isfinite(bf16_value(hb)) and float(w) == -8 * 65504.0


def test_error_budget_of_the_products_is_inside_the_tolerance():
    """With A equal to the oracle's bf16 rounding and each weight within
    2^-8 of its value, |C - y_ref| <= 2^-8 sum|a w| plus the f32 summation,
    inside 5e-3 sum|a w| + 1e-5; checked on a random problem in float64 with
    the products summed in f32 in an arbitrary order."""
    rng = np.random.default_rng(3)
    M, N, K = 8, 64, 2048
    A = rng.standard_normal((M, K)).astype(np.float32)
    Wf = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    packed = O.pack("q8_0", Wf)
    Wd = O.dequantize("q8_0", packed, N, K).astype(np.float32)
    y, tol = O.reference("q8_0", A, packed, N, K, tensor_core=True)
    Ab = bf16_value(bf16_rne_bits(A))
    Wb = bf16_value(bf16_rne_bits(Wd))
    perm = rng.permutation(K)
    C = np.zeros((M, N), np.float32)
    for k in perm:
        C += np.float32(Ab[:, k:k + 1]) * Wb[None, :, k]
    err = np.abs(C.astype(np.float64) - y)
    assert np.all(err <= tol)
    B = np.abs(Ab.astype(np.float64)) @ np.abs(Wd.astype(np.float64)).T
    assert np.all(err <= 2.0 ** -8 * B + K * 2.0 ** -24 * B)
