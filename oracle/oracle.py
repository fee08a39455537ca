"""CPU oracle for the weight-only mixed-precision matmul C = A @ W^T.

TEST INFRASTRUCTURE ONLY. Nothing in the product (the C-ABI library and its
Python binding) imports or calls this module; only the tests, the smoke check
and the CPU-baseline leg of the benchmark do. It shares no code with the CUDA
path.

It is deliberately plain and slow: the conversion and quantisation rules are
written out one step at a time in numpy float32 (the precision the host
packer on the source pages works in), and the matmul is a float64 library
matmul on the dequantised weights.

Sources (docs.rs source pages):

* lattice-inference 0.1.2, ``src/forward/metal_qwen35.rs``: the host helpers
  ``f32_to_f16`` / ``round_shift_right_even`` (IEEE round-to-nearest-even
  narrowing), ``f16_to_f32`` (exact widening), ``quantize_row_q8_0`` and the
  block constants ``Q8_0_BLOCK_SIZE = 34`` / ``Q4_0_BLOCK_SIZE = 18``; the MSL
  kernels ``gemv_q8_decode`` (x = d*q) and ``gemv_q4_decode`` (x = d*(q-8)).
* lattice-inference (latest), ``src/forward/metal_qwen35/inner/dispatch.rs``:
  ``dispatch_gemm_q8`` / ``dispatch_gemm_q4`` (C[M,N] = A[M,K] W[N,K]^T, M=1
  decode vs M>1 prefill).
* The matmul statement fixes the Q4_0 packer rule, which the pages import but
  do not print: m = the signed element of largest magnitude, d = m / -8,
  q = min(15, int(x/d + 8.5)), low nibbles hold elements 0-15 and high
  nibbles elements 16-31; and Q8_0 as d = max|x| / 127, q = round(x/d).

Readings taken where the sources are silent or disagree (each is listed with
its reason in the design notes):

* Q8_0 divides (x / d) as the matmul statement writes it; the page multiplies
  by the reciprocal. Both are computed from the float32 d, before it is
  narrowed to f16 for storage, as the page does.
* Rounding of halves is away from zero (Rust ``f32::round``); q is clamped to
  [-127, 127].
* Q4_0: the first index wins among elements of equal largest magnitude; an
  all-zero block stores q = 8 for every element (it dequantises to 0).
* The f16 scale is stored little-endian.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` to
closed forms, hand-derived golden bytes, library conversions and brute force
(the epilogues against scipy's logistic function and exact integer cases).
No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

QK = 32                 # elements per quantisation block
Q8_0_BLOCK_BYTES = 34   # f16 d + 32 x int8
Q4_0_BLOCK_BYTES = 18   # f16 d + 16 bytes of nibbles

GEMV_RTOL, GEMV_ATOL = 1e-4, 1e-6   # f32-accumulating GEMV / CUDA-core path
GEMM_RTOL, GEMM_ATOL = 5e-3, 1e-5   # tensor-core path (A rounded to bf16)


# --------------------------------------------------------------------------
# f32 <-> f16 (lattice-inference 0.1.2, metal_qwen35.rs, f32_to_f16)
# --------------------------------------------------------------------------
def _round_shift_right_even(value: np.ndarray, shift) -> np.ndarray:
    """value >> shift, rounded to nearest with ties to even (page's
    ``round_shift_right_even``): shift 0 keeps the value, shift >= 32 gives 0."""
    value = np.asarray(value).astype(np.uint64)
    shift = np.broadcast_to(np.asarray(shift, dtype=np.int64), value.shape)
    big = shift >= 32
    s = np.clip(shift, 1, 31).astype(np.uint64)
    base = value >> s
    rem = value & ((np.uint64(1) << s) - np.uint64(1))
    half = np.uint64(1) << (s - np.uint64(1))
    up = (rem > half) | ((rem == half) & ((base & np.uint64(1)) == 1))
    rounded = base + up.astype(np.uint64)
    out = np.where(shift == 0, value, rounded)
    return np.where(big, np.uint64(0), out)


_CHUNK = 1 << 22


def _f32_to_f16_chunk(bits: np.ndarray) -> np.ndarray:
    sign = ((bits >> 16) & 0x8000).astype(np.uint32)
    exp = ((bits >> 23) & 0xFF).astype(np.int32)
    frac = bits & np.uint32(0x7FFFFF)
    e = exp - 127
    out = sign.copy()                      # zero and f32 subnormals -> signed zero

    # normal f16 range: round the 23-bit fraction to 10 bits, a carry bumps
    # the exponent (possibly to infinity)
    normal = (exp != 0) & (exp != 0xFF) & (e >= -14) & (e <= 15)
    if normal.any():
        f = frac[normal]
        base = f >> 13
        rem = f & np.uint32(0x1FFF)
        up = (rem > 0x1000) | ((rem == 0x1000) & ((base & 1) == 1))
        frac16 = base + up.astype(np.uint32)
        exp16 = (e[normal] + 15).astype(np.uint32)
        carry = frac16 == 0x400
        exp16 = exp16 + carry.astype(np.uint32)
        frac16 = np.where(carry, np.uint32(0), frac16)
        val = np.where(exp16 >= 0x1F, np.uint32(0x7C00), (exp16 << 10) | frac16)
        out[normal] = sign[normal] | val

    # overflow to infinity
    over = (exp != 0) & (exp != 0xFF) & (e > 15)
    out[over] = sign[over] | 0x7C00

    # subnormal f16 range: shift the 24-bit significand right by (-e - 1)
    sub = (exp != 0) & (exp != 0xFF) & (e < -14)
    if sub.any():
        mant = frac[sub] | np.uint32(0x800000)
        v = _round_shift_right_even(mant, (-e[sub] - 1)).astype(np.uint32)
        # 0 stays signed zero; 0x400 is the smallest normal, both fit as-is
        out[sub] = sign[sub] | v

    # Inf / NaN (NaN keeps its top payload bits and gets the quiet bit)
    special = exp == 0xFF
    if special.any():
        f = frac[special]
        payload = (f >> 13) & 0x3FF
        payload = np.where(payload == 0, np.uint32(1), payload) | 0x200
        out[special] = sign[special] | 0x7C00 | np.where(f == 0, np.uint32(0), payload)
    return out.astype(np.uint16)


def f32_to_f16_bits(x) -> np.ndarray:
    """IEEE binary32 -> binary16 bits, round to nearest even.

    Step by step as the page's ``f32_to_f16``: Inf/NaN keep their class (NaN
    gets the quiet bit), f32 zero and subnormals become signed zero,
    exponents above 15 overflow to infinity, the normal range rounds the
    23-bit fraction to 10 bits (a carry bumps the exponent, possibly to
    infinity), and the subnormal range shifts the 24-bit significand right by
    (-e - 1) with round-to-nearest-even. Works through the input in chunks.
    """
    arr = np.ascontiguousarray(x, dtype=np.float32)
    bits = arr.view(np.uint32).reshape(-1)
    out = np.empty(bits.shape, dtype=np.uint16)
    for i in range(0, bits.size, _CHUNK):
        out[i:i + _CHUNK] = _f32_to_f16_chunk(bits[i:i + _CHUNK])
    return out.reshape(arr.shape)


def _f16_to_f32_codes(h: np.ndarray) -> np.ndarray:
    """binary16 bits -> binary32 bits, exact (page's ``f16_to_f32``)."""
    h = h.astype(np.uint32)
    sign = (h >> 15) & 1
    exp = (h >> 10) & 0x1F
    frac = h & 0x3FF
    out = np.zeros(h.shape, dtype=np.uint32)
    normal = (exp != 0) & (exp != 0x1F)
    out = np.where(normal, (sign << 31) | ((exp - 15 + 127) << 23) | (frac << 13), out)
    special = exp == 0x1F
    out = np.where(special, (sign << 31) | 0x7F800000 | (frac << 13), out)
    out = np.where((exp == 0) & (frac == 0), sign << 31, out)
    # subnormal: value = frac * 2^-24; normalise the leading one
    sub = (exp == 0) & (frac != 0)
    mant = frac.astype(np.int64)
    e = np.full(h.shape, -14, dtype=np.int64)
    for _ in range(10):
        need = sub & ((mant & 0x400) == 0)
        mant = np.where(need, mant << 1, mant)
        e = np.where(need, e - 1, e)
    sub_bits = (sign << 31) | (((e + 127).astype(np.uint32)) << 23) | ((mant & 0x3FF).astype(np.uint32) << 13)
    return np.where(sub, sub_bits, out)


# The widening evaluated once for every one of the 2^16 codes.
_F16_TABLE = _f16_to_f32_codes(np.arange(1 << 16, dtype=np.uint32)).view(np.float32)


def f16_bits_to_f32(h) -> np.ndarray:
    """binary16 bits -> binary32 value, exact (page's ``f16_to_f32``)."""
    return _F16_TABLE[np.asarray(h, dtype=np.uint16)]


def f32_to_bf16_rne(x) -> np.ndarray:
    """Round binary32 values to bfloat16 (nearest, ties to even), returned as f32.

    bfloat16 keeps the top 16 bits of the f32 encoding; rounding adds half an
    ulp of the kept part (0x7FFF plus the kept LSB for ties-to-even) before
    truncating. NaN stays NaN.
    """
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    isnan = ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x7FFFFF) != 0)
    rounded = np.where(isnan, (bits | 0x400000) & 0xFFFF0000, rounded)
    return (rounded & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


# --------------------------------------------------------------------------
# packers (W f32 [N, K] row-major -> bytes)
# --------------------------------------------------------------------------
def _check_finite(W: np.ndarray) -> None:
    if not np.all(np.isfinite(W)):
        raise ValueError("weights must be finite")


def pack_f16(W) -> np.ndarray:
    """W f32 [N,K] -> f16 bits [N,K] (make_buffer_f16: element-wise narrowing)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    return f32_to_f16_bits(W)


def _round_half_away(v32: np.ndarray) -> np.ndarray:
    """Nearest integer of float32 values, halves away from zero (f32::round).

    Done in float64 so that |v| + 0.5 is exact.
    """
    v = v32.astype(np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def quantize_q8_0(W, reciprocal: bool = False) -> np.ndarray:
    """Q8_0 packing of W f32 [N, K] (K % 32 == 0) -> uint8 [N, K/32*34].

    Per 32-element block (quantize_row_q8_0, with the division of the matmul
    statement):
      1. amax = max_i |x_i|                      (float32)
      2. d = amax / 127                          (float32)
      3. q_i = 0 if d == 0 else round(x_i / d)   (float32 divide, halves away
         from zero), clamped to [-127, 127]
      4. bytes 0-1: f16(d) little-endian; bytes 2..33: q_0..q_31 as int8.
    With ``reciprocal`` step 3 is the page's own expression: id = 1 / d
    (float32, 0 when d == 0), q_i = round(x_i * id) (float32 multiply).
    """
    W = np.ascontiguousarray(W, dtype=np.float32)
    _check_finite(W)
    N, K = W.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK
    x = W.reshape(N, nb, QK)
    amax = np.max(np.abs(x), axis=2)                          # f32
    d = (amax / np.float32(127.0)).astype(np.float32)         # f32
    with np.errstate(divide="ignore", invalid="ignore"):
        if reciprocal:
            inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
            v = (x * inv[:, :, None]).astype(np.float32)      # f32 multiply
        else:
            v = (x / d[:, :, None]).astype(np.float32)        # f32 divide
    q = _round_half_away(v)
    q = np.clip(q, -127, 127)
    q = np.where(d[:, :, None] == 0, 0, q).astype(np.int8)
    out = np.empty((N, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    d16 = f32_to_f16_bits(d)
    out[:, :, 0] = (d16 & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d16 >> 8).astype(np.uint8)
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(N, nb * Q8_0_BLOCK_BYTES)


def quantize_q4_0(W, interleaved: bool = False) -> np.ndarray:
    """Q4_0 packing of W f32 [N, K] (K % 32 == 0) -> uint8 [N, K/32*18].

    Per 32-element block:
      1. m = x_j for the first j with the largest |x_j|   (signed, float32)
      2. d = m / -8                                       (float32)
      3. q_i = 8 if d == 0 else min(15, trunc(x_i / d + 8.5))  (float32 math;
         the argument is >= 0.5 so truncation is floor)
      4. bytes 0-1: f16(d) little-endian; byte 2+j = q_j | q_{j+16} << 4 for
         j = 0..15 (low nibbles: elements 0-15, high nibbles: 16-31).
    With ``interleaved`` step 4 stores the order the pages' Q4 kernels read
    (gemv_q4_decode and gemm_q4: low nibble of byte j = element 2j, high
    nibble = element 2j+1): byte 2+j = q_{2j} | q_{2j+1} << 4.
    """
    W = np.ascontiguousarray(W, dtype=np.float32)
    _check_finite(W)
    N, K = W.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK
    x = W.reshape(N, nb, QK)
    j = np.argmax(np.abs(x), axis=2)                 # first index of the max
    m = np.take_along_axis(x, j[:, :, None], axis=2)[:, :, 0]
    d = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((x / d[:, :, None]).astype(np.float32) + np.float32(8.5)).astype(np.float32)
    qi = np.where(d[:, :, None] == 0, 8, np.minimum(15, np.trunc(np.nan_to_num(t)))).astype(np.uint8)
    out = np.empty((N, nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    d16 = f32_to_f16_bits(d)
    out[:, :, 0] = (d16 & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d16 >> 8).astype(np.uint8)
    if interleaved:
        out[:, :, 2:] = (qi[:, :, 0::2] & 0xF) | ((qi[:, :, 1::2] & 0xF) << 4)
    else:
        out[:, :, 2:] = (qi[:, :, :16] & 0xF) | ((qi[:, :, 16:] & 0xF) << 4)
    return out.reshape(N, nb * Q4_0_BLOCK_BYTES)


def pack(fmt: str, W) -> np.ndarray:
    if fmt == "f16":
        return pack_f16(W)
    if fmt == "q8_0":
        return quantize_q8_0(W)
    if fmt == "q4_0":
        return quantize_q4_0(W)
    if fmt == "q4_0i":
        return quantize_q4_0(W, interleaved=True)
    raise ValueError(fmt)


# --------------------------------------------------------------------------
# dequantisation (gemv_q8_decode: d*q; gemv_q4_decode: d*(q-8); f16: widen)
# --------------------------------------------------------------------------
def _scales(blocks: np.ndarray) -> np.ndarray:
    d16 = blocks[..., 0].astype(np.uint16) | (blocks[..., 1].astype(np.uint16) << 8)
    return f16_bits_to_f32(d16)


def dequantize_q8_0(packed, N: int, K: int) -> np.ndarray:
    """uint8 [N, K/32*34] -> f32 [N, K]; each value d*q is exact in float32."""
    b = np.asarray(packed, dtype=np.uint8).reshape(N, K // QK, Q8_0_BLOCK_BYTES)
    d = _scales(b)
    q = b[:, :, 2:].view(np.int8).astype(np.float32)
    return (d[:, :, None] * q).astype(np.float32).reshape(N, K)


def unpack_q4_0_codes(packed, N: int, K: int, interleaved: bool = False) -> np.ndarray:
    """uint8 [N, K/32*18] -> the 4-bit codes q in 0..15, shape [N, K]
    (``interleaved``: byte j holds elements 2j (low) and 2j+1 (high))."""
    b = np.asarray(packed, dtype=np.uint8).reshape(N, K // QK, Q4_0_BLOCK_BYTES)
    lo = b[:, :, 2:] & 0xF
    hi = b[:, :, 2:] >> 4
    if interleaved:
        return np.stack([lo, hi], axis=3).reshape(N, K)
    return np.concatenate([lo, hi], axis=2).reshape(N, K)


def dequantize_q4_0(packed, N: int, K: int, interleaved: bool = False) -> np.ndarray:
    """uint8 [N, K/32*18] -> f32 [N, K]; each value d*(q-8) is exact in float32."""
    b = np.asarray(packed, dtype=np.uint8).reshape(N, K // QK, Q4_0_BLOCK_BYTES)
    d = _scales(b)
    q = unpack_q4_0_codes(packed, N, K, interleaved).reshape(N, K // QK, QK).astype(np.float32) - np.float32(8)
    return (d[:, :, None] * q).astype(np.float32).reshape(N, K)


def dequantize_f16(packed, N: int, K: int) -> np.ndarray:
    return f16_bits_to_f32(np.asarray(packed, dtype=np.uint16).reshape(N, K))


def dequantize(fmt: str, packed, N: int, K: int) -> np.ndarray:
    if fmt == "f16":
        return dequantize_f16(packed, N, K)
    if fmt == "q8_0":
        return dequantize_q8_0(packed, N, K)
    if fmt == "q4_0":
        return dequantize_q4_0(packed, N, K)
    if fmt == "q4_0i":
        return dequantize_q4_0(packed, N, K, interleaved=True)
    raise ValueError(fmt)


def packed_row_bytes(fmt: str, K: int) -> int:
    if fmt == "f16":
        return 2 * K
    if fmt == "q8_0":
        return K // QK * Q8_0_BLOCK_BYTES
    if fmt in ("q4_0", "q4_0i"):
        return K // QK * Q4_0_BLOCK_BYTES
    raise ValueError(fmt)


# --------------------------------------------------------------------------
# the matmul and its error bound
# --------------------------------------------------------------------------
def matmul_ref(A, W_hat):
    """y_ref = A @ W_hat^T and B = |A| @ |W_hat|^T, both in float64.

    A f32 [M, K] activations, W_hat f32 [N, K] dequantised weights. B is the
    sum of |a_k * w_k| that scales the tolerance of every output element.
    """
    A64 = np.asarray(A, dtype=np.float32).astype(np.float64)
    W64 = np.asarray(W_hat, dtype=np.float32).astype(np.float64)
    y = A64 @ W64.T
    B = np.abs(A64) @ np.abs(W64).T
    return y, B


def reference(fmt: str, A, packed, N: int, K: int, tensor_core: bool = False):
    """(y_ref, tol) for C = A @ dequant(W)^T.

    With ``tensor_core`` the activations are first rounded to bf16 (the
    operand type of the tensor-core path) and the looser tolerance applies.
    """
    W_hat = dequantize(fmt, packed, N, K)
    A = np.asarray(A, dtype=np.float32)
    if tensor_core:
        A = f32_to_bf16_rne(A)
        rtol, atol = GEMM_RTOL, GEMM_ATOL
    else:
        rtol, atol = GEMV_RTOL, GEMV_ATOL
    y, B = matmul_ref(A, W_hat)
    return y, rtol * B + atol


# --------------------------------------------------------------------------
# epilogues: residual add and gate/up SwiGLU
# (oxibonsai-kernels 0.1.4, src/gpu_backend/metal_prefill/functions.rs:
# gemm_q1_v7_residual writes W x + hidden back into hidden;
# fused_gate_up_swiglu_gemm runs on the gate_up weight of 2 * inter rows and
# expands, without the fused kernel, to a GEMM with n_rows = 2 * inter and
# batched_swiglu. lattice-inference 0.1.2, metal_qwen35.rs: silu_mul, the
# product silu(gate) * up with silu(g) = g / (1 + exp(-g)); lattice-inference
# dispatch.rs: dispatch_silu_mul_fused over [gate | up] of one token, and
# dispatch_gemm_at, gate rows first and up rows after them in gate_up.)
# --------------------------------------------------------------------------
F32_EPS = 2.0 ** -24          # unit roundoff of float32
SILU_LIPSCHITZ = 1.0999       # max over x of |d silu(x) / dx| (1.0998 near x = 2.40)


def silu(x):
    """silu(x) = x / (1 + exp(-x)) in float64, as silu_mul writes it; for
    x below about -709 exp overflows and the quotient is -0, the limit."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def residual_reference(y, tol, R):
    """(c_ref, tol) for C = A W^T + R given the matmul's (y_ref, tol).

    The kernel adds R in float32 to its float32 sum: one more rounding, half
    an ulp of the result."""
    R64 = np.asarray(R, dtype=np.float32).astype(np.float64)
    c = y + R64
    return c, tol + F32_EPS * (np.abs(c) + tol)


def swiglu_reference(y, tol, I: int):
    """(h_ref, tol) for the gate/up SwiGLU over y = A [gate; up]^T (2I
    columns, gate first): h[m, j] = silu(g) * u with g = y[m, j] and
    u = y[m, I + j].

    Bound: the kernel's g' and u' are within tg and tu of g and u (the
    matmul tolerance of the two rows); silu is Lipschitz with constant
    SILU_LIPSCHITZ, so |silu(g') u' - silu(g) u| <= L tg (|u| + tu) +
    |silu(g)| tu. The float32 evaluation adds at most 3.5 ulp relative (exp
    within 2 ulp, then an add, a divide and a multiply of half an ulp each),
    taken as 8 F32_EPS of |h| plus that bound."""
    y = np.asarray(y, dtype=np.float64)
    tol = np.asarray(tol, dtype=np.float64)
    g, u = y[:, :I], y[:, I:2 * I]
    tg, tu = tol[:, :I], tol[:, I:2 * I]
    sg = silu(g)
    h = sg * u
    prop = SILU_LIPSCHITZ * tg * (np.abs(u) + tu) + np.abs(sg) * tu
    return h, prop + 8 * F32_EPS * (np.abs(h) + prop) + 1e-30


def topk_first(y, k: int):
    """The k best entries of y as (values, indices), best first: larger value
    first, equal values by the lower index, NaN never chosen (topk_better and
    the k candidates logits_topk_first_pass / logits_topk_merge_pass keep,
    lattice-inference 0.1.2, metal_qwen35.rs). Fewer than k non-NaN entries:
    the rest are the pages' sentinel, value -inf and index -1 (UINT_MAX)."""
    y = np.asarray(y, dtype=np.float64).reshape(-1)
    idx = [i for i in range(y.size) if not np.isnan(y[i])]
    # -0 and +0 compare equal, as the pages' float comparison does
    idx.sort(key=lambda i: (-(y[i] + 0.0), i))
    idx = idx[:k]
    vals = [float(y[i]) for i in idx] + [-np.inf] * (k - len(idx))
    return np.array(vals, dtype=np.float64), np.array(idx + [-1] * (k - len(idx)), dtype=np.int64)


def argmax_first(y) -> int:
    """Index of the largest value; ties go to the lowest index, NaN never wins."""
    y = np.asarray(y, dtype=np.float64)
    best, best_i = -np.inf, -1
    finite_or_inf = ~np.isnan(y)
    if not finite_or_inf.any():
        return -1
    vals = np.where(finite_or_inf, y, -np.inf)
    best = vals.max()
    cand = np.nonzero(finite_or_inf & (vals == best))[0]
    best_i = int(cand[0])
    return best_i
