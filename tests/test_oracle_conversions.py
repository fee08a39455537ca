"""Pins for the oracle's f32<->f16 and f32->bf16 conversions.

The oracle restates the page's bit-level ``f32_to_f16`` (lattice-inference
0.1.2, metal_qwen35.rs). It is checked here against hand-derived binary16
encodings, against numpy's own float16 cast (an independent implementation of
IEEE round-to-nearest-even) over every f32 rounding class, and against
torch's bfloat16 cast.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _structured_f32_bits():
    """All 2^16 top halves (sign, exponent, 7 fraction bits) x the low halves
    that decide f16 rounding (0, 1, just below/at/above the f16 half-ulp at
    bit 12, all ones ...), plus random patterns."""
    hi = np.arange(1 << 16, dtype=np.uint64) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001,
                     0x3000, 0x5FFF, 0x6000, 0x6001, 0x7FFF, 0x8000, 0x8001, 0xA000,
                     0xBFFF, 0xC000, 0xE000, 0xEFFF, 0xF000, 0xFFFF], dtype=np.uint64)
    bits = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(1234)
    rnd = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64)
    return np.concatenate([bits, rnd]).astype(np.uint32)


def test_f16_golden_values():
    with open(os.path.join(GOLDEN, "f16_values.json")) as f:
        g = json.load(f)
    src = np.array([int(c[0], 16) for c in g["cases"]], dtype=np.uint32).view(np.float32)
    want = np.array([int(c[1], 16) for c in g["cases"]], dtype=np.uint16)
    got = O.f32_to_f16_bits(src)
    for s, w, gt, c in zip(src, want, got, g["cases"]):
        assert gt == w, f"{c[2]}: got {gt:#06x} want {w:#06x}"


def test_f32_to_f16_matches_numpy_cast():
    bits = _structured_f32_bits()
    f = bits.view(np.float32)
    got = O.f32_to_f16_bits(f)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    bad = np.nonzero((got != ref) & ~nan)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first f32 {bits[bad[0]]:#010x}"
    # NaN stays NaN (the page also sets the quiet bit)
    g_nan = got[nan]
    assert np.all((g_nan & 0x7C00) == 0x7C00) and np.all((g_nan & 0x03FF) != 0)
    assert np.all((g_nan & 0x0200) != 0)


def test_f16_to_f32_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = O.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    assert np.all(np.isnan(got[nan]))


def test_f16_round_trip_is_identity_on_f16_values():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.f16_bits_to_f32(h)
    finite = np.isfinite(v)
    back = O.f32_to_f16_bits(v[finite])
    assert np.array_equal(back, h[finite])


def test_f32_to_bf16_matches_torch_cast():
    bits = _structured_f32_bits()
    f = bits.view(np.float32)
    got = O.f32_to_bf16_rne(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(f)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    assert np.all(np.isnan(got[nan]))


def test_bf16_closed_forms():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even (1.0);
    # 1 + 3*2^-8 ties up to 1 + 2^-6; the largest finite f32 overflows.
    x = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20, -1.0, 0.0], dtype=np.float32)
    want = np.array([1.0, 1 + 2**-6, 1 + 2**-7, -1.0, 0.0], dtype=np.float32)
    assert np.array_equal(O.f32_to_bf16_rne(x), want)
    big = np.array([np.finfo(np.float32).max], dtype=np.float32)
    assert np.isinf(O.f32_to_bf16_rne(big)[0])


@pytest.mark.parametrize("mutant", ["truncate", "round_half_up"])
def test_planted_conversion_mistakes_are_caught(monkeypatch, mutant):
    """Plant a rounding mistake in the oracle's shift helper; the pins must fail."""
    orig = O.oracle._round_shift_right_even

    def truncate(value, shift):
        v = value.astype(np.uint64)
        s = np.minimum(shift.astype(np.uint64), 63)
        return np.where(shift >= 32, 0, v >> s)

    def half_up(value, shift):
        r = orig(value, shift)
        v = value.astype(np.uint64)
        s = np.maximum(shift.astype(np.uint64), 1)
        rem = v & ((np.uint64(1) << s) - np.uint64(1))
        tie = (rem == (np.uint64(1) << (s - np.uint64(1)))) & (shift > 0) & (shift < 32)
        return np.where(tie, (v >> s) + 1, r)

    monkeypatch.setattr(O.oracle, "_round_shift_right_even",
                        truncate if mutant == "truncate" else half_up)
    with pytest.raises(AssertionError):
        test_f16_golden_values()
