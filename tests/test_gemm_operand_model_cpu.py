"""A CPU model of the tensor-core GEMM's f16 operands (lq_gemm_tma.cu: the
a_to_f16_kernel pre-pass and the Q8_0 / Q4_0 converters), pinning the two
numerical facts the kernels rely on.

A: each token row is divided by s = 2^(e - 15), where amax = m * 2^e with
m in [1/2, 1) (frexp) and e at least -111 (below that, 2^(15 - e) would
overflow f32: the model caught such rows turning into infinities), so every
|a / s| < 2^15 fits f16 without overflow;
rounding to f16 then keeps 11 significant bits, at least bf16's 8, and s is
undone exactly in the epilogue.

W (Q formats): a code byte goes into an f16 of exponent 0x64 (1024 + byte),
the bias 1152 (Q8_0: 1024 + 128) or 1032 (Q4_0: 1024 + 8) comes off exactly,
and one half-precision multiply by f16(256 d) gives 256 w rounded once. The
range is the limit: 256 |w| must stay below f16's largest value, so weights
of magnitude 256 and more overflow on this route.
"""
import numpy as np

import oracle as O

F16_MAX = 65504.0


def prepass(a):
    """One token row -> (f16 values, scale s)."""
    a = np.asarray(a, dtype=np.float32)
    amax = float(np.max(np.abs(a)))
    if amax == 0.0:
        return a.astype(np.float16), 1.0
    _, e = np.frexp(amax)
    e = max(int(e), -111)  # below 2^-112 the row is scaled by 2^126 (2^(15 - e) would overflow f32)
    s, inv = 2.0 ** (e - 15), 2.0 ** (15 - e)
    with np.errstate(over="ignore"):
        return (a * np.float32(inv)).astype(np.float16), s


def q8_weight_times_256(code, d_bits):
    """code: int8 q; d_bits: the block's f16 scale bits."""
    d = np.uint16(d_bits).view(np.float16)
    d256 = np.float16(np.float32(d) * np.float32(256.0))          # __hmul2(d, 256), one rounding
    byte = (int(code) & 0xFF) ^ 0x80                               # sign bit flipped
    magic = np.uint16(0x6400 | byte).view(np.float16)              # 1024 + byte, exact
    q = np.float16(np.float32(magic) - np.float32(1152.0))         # exact: q
    with np.errstate(over="ignore"):                               # q * d256 is exact in f32
        return np.float16(np.float32(q) * np.float32(d256))        # one rounding to f16


def q4_weight_times_256(nibble, d_bits):
    d = np.uint16(d_bits).view(np.float16)
    d256 = np.float16(np.float32(d) * np.float32(256.0))
    magic = np.uint16(0x6400 | int(nibble)).view(np.float16)
    q = np.float16(np.float32(magic) - np.float32(1032.0))
    with np.errstate(over="ignore"):
        return np.float16(np.float32(q) * np.float32(d256))


def test_prepass_never_overflows_and_keeps_eleven_bits():
    rng = np.random.default_rng(0)
    rows = [rng.standard_normal(2048) * 10.0 ** rng.integers(-30, 30) for _ in range(200)]
    rows += [np.array([3.4e38, -1.0, 1e-30]), np.array([1e-38, -2e-38]), np.array([65504.0, 65520.0, 1e9]),
             np.array([1e-36, 3e-40, -1e-45])]  # tiny rows, f32 subnormals included
    for row in rows:
        row = row.astype(np.float32)
        h, s = prepass(row)
        assert np.all(np.isfinite(h.astype(np.float32)))
        back = h.astype(np.float64) * s
        a = row.astype(np.float64)
        amax = np.max(np.abs(a))
        # 11 significant bits where the scaled value is a normal f16, an absolute
        # f16 subnormal step (2^-24 * s) below that: both well inside bf16's 2^-9
        err = np.abs(back - a)
        assert np.all(err <= np.maximum(2.0 ** -11 * np.abs(a), 2.0 ** -24 * s) * (1 + 1e-12))
        assert np.all(err <= 2.0 ** -9 * np.abs(a) + 2.0 ** -24 * s * 1.0001)
        assert np.max(np.abs(h.astype(np.float64))) < 2.0 ** 15
        assert amax / s >= 2.0 ** 14 or amax < 2.0 ** -112


def test_q8_0_codes_exact_and_one_rounding_in_range():
    rng = np.random.default_rng(1)
    scales = O.f32_to_f16_bits(np.float32(10.0) ** rng.uniform(-6, 0.2, 400).astype(np.float32))
    for d_bits in scales:
        d = float(np.uint16(d_bits).view(np.float16))
        for code in range(-128, 128):
            w256 = float(q8_weight_times_256(code, d_bits))
            exact = 256.0 * code * d
            if abs(exact) < 2.0 ** -14:      # beyond what the pins here address: f16 subnormals
                continue
            # one f16 rounding of 256 q d (plus the rounding of 256 d, exact for normal d)
            assert abs(w256 - exact) <= 2.0 ** -11 * abs(exact) * (1 + 1e-9), (code, d)


def test_q4_0_codes_exact_and_one_rounding_in_range():
    rng = np.random.default_rng(2)
    scales = O.f32_to_f16_bits(np.float32(10.0) ** rng.uniform(-6, 1.4, 400).astype(np.float32))
    for d_bits in scales:
        d = float(np.uint16(d_bits).view(np.float16))
        for nib in range(16):
            w256 = float(q4_weight_times_256(nib, d_bits))
            exact = 256.0 * (nib - 8) * d
            if exact != 0 and abs(exact) < 2.0 ** -14:
                continue
            assert abs(w256 - exact) <= 2.0 ** -11 * abs(exact) * (1 + 1e-9), (nib, d)


def test_weight_range_limit_of_the_tensor_core_route():
    """The documented limit: |w| below 256 stays finite, the largest Q8_0 block
    scale that keeps every code finite is just under 2, and larger weights
    overflow (the CUDA-core routes compute in f32 and have no such limit)."""
    ok = O.f32_to_f16_bits(np.float32(1.99))[()]
    assert np.isfinite(q8_weight_times_256(-128, ok)) and np.isfinite(q8_weight_times_256(127, ok))
    big = O.f32_to_f16_bits(np.float32(2.01))[()]
    assert not np.isfinite(q8_weight_times_256(-128, big))
    assert not np.isfinite(q8_weight_times_256(127, O.f32_to_f16_bits(np.float32(2.02))[()]))
    q4_ok = O.f32_to_f16_bits(np.float32(31.9))[()]
    assert np.isfinite(q4_weight_times_256(0, q4_ok))                 # q - 8 = -8: |w| = 255.2
    assert not np.isfinite(q4_weight_times_256(0, O.f32_to_f16_bits(np.float32(32.5))[()]))
    # the workloads' weights (~N(0, 0.02), outlier blocks x20) are orders of magnitude inside
    assert 256.0 * 0.02 * 20 * 5 < F16_MAX
