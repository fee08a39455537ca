"""Pins for the oracle's Q8_0 / Q4_0 packers and dequantisers.

Checked against hand-derived golden blocks (tests/golden), closed forms
(round-trip bounds, constant blocks, exact-scale blocks) and planted mistakes.
"""
import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _block_from_t(g):
    return (np.array(g["t"], dtype=np.float64) * g["x_scale"]).astype(np.float32)[None, :]


def test_q8_0_golden_exact_scale():
    g = _golden("q8_0_exact_scale.json")
    got = O.quantize_q8_0(_block_from_t(g))[0]
    assert list(got) == g["bytes"]


def test_q8_0_golden_half_away_from_zero():
    g = _golden("q8_0_half_away.json")
    got = O.quantize_q8_0(_block_from_t(g))[0]
    assert list(got) == g["bytes"]


def test_q4_0_golden_ramp_nibble_order():
    g = _golden("q4_0_ramp.json")
    x = (np.array(g["k"], dtype=np.float64) * g["x_scale"]).astype(np.float32)[None, :]
    got = O.quantize_q4_0(x)[0]
    assert list(got) == g["bytes"]


def test_q4_0_golden_positive_max_and_clamp():
    g = _golden("q4_0_positive_max.json")
    x = np.zeros((1, 32), dtype=np.float32)
    for i, v in g["x"].items():
        x[0, int(i)] = v
    got = O.quantize_q4_0(x)[0]
    assert list(got) == g["bytes"]


def test_zero_block_golden():
    g = _golden("zero_block.json")
    z = np.zeros((1, 32), dtype=np.float32)
    assert list(O.quantize_q8_0(z)[0]) == g["q8_0_bytes"]
    assert list(O.quantize_q4_0(z)[0]) == g["q4_0_bytes"]
    assert np.all(O.dequantize_q8_0(O.quantize_q8_0(z), 1, 32) == 0)
    assert np.all(O.dequantize_q4_0(O.quantize_q4_0(z), 1, 32) == 0)


def _f16_round(v):
    return O.f16_bits_to_f32(O.f32_to_f16_bits(np.asarray(v, dtype=np.float32)))


def test_q8_0_round_trip_bound_random():
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    W[3, 64:96] *= 20.0
    p = O.quantize_q8_0(W)
    What = O.dequantize_q8_0(p, 64, 1024)
    xb = W.reshape(64, 32, 32).astype(np.float64)
    d = (np.max(np.abs(W.reshape(64, 32, 32)), axis=2) / np.float32(127)).astype(np.float32)
    d16 = _f16_round(d).astype(np.float64)
    err = np.abs(xb - What.reshape(64, 32, 32).astype(np.float64))
    bound = d.astype(np.float64)[..., None] / 2 + 127 * np.abs(d.astype(np.float64) - d16)[..., None]
    assert np.all(err <= bound * (1 + 1e-6) + 1e-30)


def test_q8_0_exact_scale_reconstructs_within_half_step():
    # blocks with amax = 127 * 2^e: d = 2^e is exact in f16, so |x - w| <= d/2
    rng = np.random.default_rng(8)
    for e in range(-12, 3):
        d = 2.0 ** e
        x = rng.uniform(-127, 127, size=32)
        x[rng.integers(0, 32)] = 127 * (1 if rng.random() < 0.5 else -1)
        x = (x * d).astype(np.float32)[None, :]
        w = O.dequantize_q8_0(O.quantize_q8_0(x), 1, 32)
        assert np.all(np.abs(x.astype(np.float64) - w) <= d / 2)
        # multiples of d come back exactly
        t = rng.integers(-127, 128, size=32).astype(np.float64)
        t[0] = 127
        xm = (t * d).astype(np.float32)[None, :]
        assert np.array_equal(O.dequantize_q8_0(O.quantize_q8_0(xm), 1, 32), xm)


def test_q4_0_round_trip_bounds_random():
    rng = np.random.default_rng(9)
    for e in range(-10, 2):
        # d = m/-8 with m = -8 * 2^e * s: exact in f16
        for sign in (1, -1):
            m = -8 * sign * 2.0 ** e
            x = rng.uniform(-abs(m), abs(m), size=32)
            j = rng.integers(0, 32)
            x[j] = m
            x = x.astype(np.float32)[None, :]
            d = m / -8.0
            p = O.quantize_q4_0(x)
            w = O.dequantize_q4_0(p, 1, 32)[0].astype(np.float64)
            q = O.unpack_q4_0_codes(p, 1, 32)[0].astype(np.int64)
            r = x[0].astype(np.float64) / d
            err = np.abs(x[0] - w)
            inside = r <= 7.5
            assert np.all(err[inside] <= abs(d) / 2)
            assert np.all(err[~inside] <= abs(d))
            # the max-magnitude element reconstructs exactly
            assert w[j] == x[0, j]
            # q = 8 exactly when -0.5 <= x/d < 0.5 (away from the f32
            # rounding of x/d + 8.5 right at the edges)
            clear = (np.abs(r - 0.5) > 1e-5) & (np.abs(r + 0.5) > 1e-5)
            assert np.array_equal((q == 8)[clear], ((r >= -0.5) & (r < 0.5))[clear])


def test_constant_blocks_closed_form():
    for c in [0.37, -0.37, 1.0, -3.5e-3, 12345.0]:
        x = np.full((1, 32), c, dtype=np.float32)
        # Q8_0: q = 127*sign(c), w = f16(|c|/127) * 127 * sign(c)
        p8 = O.quantize_q8_0(x)
        q8 = p8[0, 2:].view(np.int8)
        assert np.all(q8 == 127 * np.sign(c))
        d = np.float32(abs(np.float32(c))) / np.float32(127)
        assert np.all(O.dequantize_q8_0(p8, 1, 32) == _f16_round(d) * np.float32(127 * np.sign(c)))
        # Q4_0: m = c, d = c/-8, x/d = -8 -> q = 0, w = -8 * f16(c/-8)
        p4 = O.quantize_q4_0(x)
        assert np.all(O.unpack_q4_0_codes(p4, 1, 32) == 0)
        w4 = O.dequantize_q4_0(p4, 1, 32)
        assert np.all(w4 == np.float32(-8) * _f16_round(np.float32(c) / np.float32(-8)))
    # c/8 exact in f16 -> reconstructs c exactly
    x = np.full((1, 32), 0.75, dtype=np.float32)
    assert np.all(O.dequantize_q4_0(O.quantize_q4_0(x), 1, 32) == 0.75)


def test_dequant_is_exact_f32_product():
    # d (11 significant bits) times q (<= 8 bits) fits in 24 bits: recompute
    # d*q in float64 and compare with the float32 result.
    rng = np.random.default_rng(10)
    W = (rng.standard_normal((16, 256)) * 0.05).astype(np.float32)
    for fmt in ("q8_0", "q4_0"):
        p = O.pack(fmt, W)
        bpb = O.Q8_0_BLOCK_BYTES if fmt == "q8_0" else O.Q4_0_BLOCK_BYTES
        b = p.reshape(16, 8, bpb)
        d = O.f16_bits_to_f32(b[..., 0].astype(np.uint16) | (b[..., 1].astype(np.uint16) << 8)).astype(np.float64)
        if fmt == "q8_0":
            q = b[..., 2:].view(np.int8).astype(np.float64)
        else:
            q = O.unpack_q4_0_codes(p, 16, 256).reshape(16, 8, 32).astype(np.float64) - 8
        exact = (d[..., None] * q).reshape(16, 256)
        assert np.array_equal(O.dequantize(fmt, p, 16, 256).astype(np.float64), exact)


def test_packers_reject_bad_input():
    with pytest.raises(ValueError):
        O.quantize_q8_0(np.zeros((2, 33), dtype=np.float32))
    with pytest.raises(ValueError):
        O.quantize_q4_0(np.full((1, 32), np.nan, dtype=np.float32))


def test_planted_half_even_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(O.oracle, "_round_half_away", lambda v: np.round(v.astype(np.float64)))
    with pytest.raises(AssertionError):
        test_q8_0_golden_half_away_from_zero()


def test_planted_interleaved_nibbles_are_caught(monkeypatch):
    """A dequantiser that reads the page's interleaved nibble order (byte j =
    elements 2j, 2j+1) must fail the ramp golden's round trip."""
    def interleaved(packed, N, K, interleaved=False):
        b = np.asarray(packed, dtype=np.uint8).reshape(N, K // 32, 18)[:, :, 2:]
        out = np.empty((N, K // 32, 32), dtype=np.uint8)
        out[:, :, 0::2] = b & 0xF
        out[:, :, 1::2] = b >> 4
        return out.reshape(N, K)

    g = _golden("q4_0_ramp.json")
    x = (np.array(g["k"], dtype=np.float64) * g["x_scale"]).astype(np.float32)[None, :]
    p = O.quantize_q4_0(x)
    assert np.array_equal(O.dequantize_q4_0(p, 1, 32), x)
    monkeypatch.setattr(O.oracle, "unpack_q4_0_codes", interleaved)
    assert not np.array_equal(O.dequantize_q4_0(p, 1, 32), x)


# ---- the pages' own layouts: interleaved Q4_0 nibbles, Q8_0 via 1/d --------
def test_q4_0i_golden_ramp_interleaved_nibbles():
    g = _golden("q4_0i_ramp.json")
    x = (np.array(g["k"], dtype=np.float64) * g["x_scale"]).astype(np.float32)[None, :]
    got = O.quantize_q4_0(x, interleaved=True)[0]
    assert list(got) == g["bytes"]
    assert list(O.pack("q4_0i", x)[0]) == g["bytes"]


def test_q4_0i_holds_the_same_values_as_q4_0():
    """The two layouts store the same codes and scale: dequantised they are
    identical element for element, while the bytes differ."""
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((9, 256)) * 0.05).astype(np.float32)
    a, b = O.pack("q4_0", W), O.pack("q4_0i", W)
    assert not np.array_equal(a, b)
    assert np.array_equal(O.dequantize("q4_0", a, 9, 256), O.dequantize("q4_0i", b, 9, 256))
    # a planted mistake: reading interleaved bytes in the standard order
    assert not np.array_equal(O.dequantize("q4_0", b, 9, 256), O.dequantize("q4_0i", b, 9, 256))


def test_q8_0_golden_reciprocal_rounding():
    g = _golden("q8_0_reciprocal.json")
    x = np.array(g["x_bits"], dtype=np.uint32).view(np.float32)[None, :]
    assert list(O.quantize_q8_0(x)[0]) == g["bytes_divide"]
    assert list(O.quantize_q8_0(x, reciprocal=True)[0]) == g["bytes_reciprocal"]


def test_q8_0_reciprocal_differs_from_divide_only_at_ties():
    """On random blocks the two rules agree except where x/d lies within an
    ulp of a half: the codes differ by one there."""
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((200, 1024)) * 0.02).astype(np.float32)
    a = O.quantize_q8_0(W).reshape(200, 32, 34)[:, :, 2:].view(np.int8).astype(int)
    b = O.quantize_q8_0(W, reciprocal=True).reshape(200, 32, 34)[:, :, 2:].view(np.int8).astype(int)
    diff = np.abs(a - b)
    assert diff.max() <= 1
    assert (diff > 0).mean() < 1e-3
