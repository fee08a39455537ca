"""Host-side checks of the C-ABI library that need no GPU: the exported
symbols, the host packers (bit-exact against the oracle) and the argument
checks that return before any launch."""
import os
import re

import numpy as np
import pytest

import oracle as O
import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_declarations_are_all_exported(lq):
    with open(os.path.join(ROOT, "include", "lq.h")) as f:
        text = f.read()
    declared = set(re.findall(r"\b(lq_[a-z0-9_]+)\s*\(", text))
    assert declared == set(lq.EXPORTS)
    L = lq.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_version_and_status_strings(lq):
    assert "sm_103a" in lq.version()
    for s in range(6):
        assert lq.status_string(s).startswith("LQ_")


@pytest.mark.parametrize("fmt,N,K", [("f16", 3, 7), ("q8_0", 5, 64), ("q4_0", 2, 96)])
def test_packed_bytes(lq, fmt, N, K):
    assert lq.packed_bytes(fmt, N, K) == N * O.packed_row_bytes(fmt, K)
    assert lq.packed_bytes("q8_0", 1, 33) == 0
    assert lq.packed_bytes("q4_0", -1, 32) == 0


def _adversarial(K=256):
    rows = []
    z = np.zeros(K, np.float32)
    rows.append(z)                                   # all-zero blocks
    r = z.copy(); r[3] = 1.0; r[7] = -1.0            # +a/-a tie (first wins)
    rows.append(r)
    r = z.copy(); r[5] = -1.0; r[9] = 1.0
    rows.append(r)
    rows.append(np.full(K, 0.37, np.float32))        # constant blocks
    rows.append(np.full(K, -2.5e-3, np.float32))
    t = (np.arange(K) % 32 - 16).astype(np.float32) * np.float32(2**-6) * np.float32(127 / 16)
    rows.append(t.astype(np.float32))                # ramps
    rows.append((np.arange(K) % 32 - 16).astype(np.float32) * np.float32(0.5))  # exact halves
    rows.append(np.full(K, 1e-6, np.float32))        # d in the f16 subnormal range
    rows.append(np.full(K, 3e-9, np.float32))        # d underflows to 0 in f16
    r = np.full(K, 1e-3, np.float32); r[::32] = 1e7  # d overflows f16 (inf)
    rows.append(r)
    r = np.full(K, 0.01, np.float32); r[1::32] = -0.02
    rows.append(r)
    rng = np.random.default_rng(0)
    rows.append((rng.standard_normal(K) * 0.02).astype(np.float32))
    rows.append(-z)                                  # -0.0 everywhere
    return np.stack(rows)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
def test_packer_bit_exact_adversarial(lq, fmt):
    W = _adversarial()
    assert np.array_equal(lq.pack(fmt, W).view(np.uint8), O.pack(fmt, W).view(np.uint8))


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_packer_bit_exact_random(lq, fmt, seed):
    rng = np.random.default_rng(seed)
    N, K = 37, 32 * (1 + seed * 5)
    W = (rng.standard_normal((N, K)) * rng.choice([0.02, 1.0, 300.0])).astype(np.float32)
    W[rng.integers(0, N)] *= 20
    assert np.array_equal(lq.pack(fmt, W).view(np.uint8), O.pack(fmt, W).view(np.uint8))


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_packer_q8_0_reciprocal_bit_exact(lq, seed):
    """The pages' round(x * (1/d)): byte for byte with the oracle, on random
    weights and on the golden block where it differs from round(x / d)."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((64, 512)) * rng.choice([0.02, 1.0, 300.0])).astype(np.float32)
    W = np.concatenate([W, _adversarial(512)])
    got = lq.pack("q8_0", W, reciprocal=True)
    assert np.array_equal(got, O.quantize_q8_0(W, reciprocal=True))
    import json
    with open(os.path.join(ROOT, "tests", "golden", "q8_0_reciprocal.json")) as f:
        g = json.load(f)
    x = np.array(g["x_bits"], dtype=np.uint32).view(np.float32)[None, :]
    assert list(lq.pack("q8_0", x, reciprocal=True)[0]) == g["bytes_reciprocal"]
    assert list(lq.pack("q8_0", x)[0]) == g["bytes_divide"]


@pytest.mark.parametrize("name", ["gemv_q8_0_4096x4096", "gemv_q4_0_11008x4096_outliers",
                                  "gemm_q8_0_512x6144x2048", "gemm_q4_0_512x6144x2048",
                                  "gemm_f16_512x6144x2048"])
def test_packer_bit_exact_on_workload_weights(lq, name):
    w = synthetic.WORKLOADS[name]
    W, _ = synthetic.draw_workload(w, M=1)
    Wn = W.numpy()
    assert np.array_equal(lq.pack(w.fmt, Wn).view(np.uint8), O.pack(w.fmt, Wn).view(np.uint8))


def test_packer_rejects_bad_input(lq):
    with pytest.raises(lq.LQError):
        lq.pack("q8_0", np.zeros((2, 48), np.float32))
    bad = np.zeros((1, 32), np.float32)
    bad[0, 4] = np.inf
    for fmt in ("f16", "q8_0", "q4_0"):
        with pytest.raises(lq.LQError):
            lq.pack(fmt, bad)


def _raw(lq, name, A, W, C, M, N, K):
    return getattr(lq.lib(), name)(A, W, C, M, N, K, 0)


@pytest.mark.parametrize("kind", ["gemv", "gemm", "matmul"])
@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
def test_argument_errors_return_before_launch(lq, kind, fmt):
    name = f"lq_{kind}_{fmt}"
    # never dereferenced: every call below fails validation or is a no-op
    a, w, c = 0x10000, 0x20000, 0x30000
    assert _raw(lq, name, a, w, c, 0, 8, 64) == lq.LQ_OK
    assert _raw(lq, name, a, w, c, 1, 0, 64) == lq.LQ_OK
    assert _raw(lq, name, None, None, None, 0, 0, 64) == lq.LQ_OK
    assert _raw(lq, name, a, w, c, -1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a, w, c, 1, 8, -64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, None, w, c, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a, None, c, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a, w, None, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a, w, c, 1, 8, 0) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a + 2, w, c, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    assert _raw(lq, name, a, w, c + 1, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    if fmt == "f16":
        assert _raw(lq, name, a, w + 1, c, 1, 8, 64) == lq.LQ_ERR_INVALID_ARG
    else:
        assert _raw(lq, name, a, w, c, 1, 8, 48) == lq.LQ_ERR_INVALID_ARG
    if kind == "gemv":
        assert _raw(lq, name, a, w, c, 2, 8, 64) == lq.LQ_ERR_INVALID_ARG


def test_route_hooks(lq):
    for bad in (9, 4, -1):  # 4 counts the decode chain but is no route of its own
        with pytest.raises(lq.LQError):
            lq.force_route(bad)
    lq.force_route(lq.ROUTE_WARP_MMA)
    lq.force_route(0)
    lq.reset_counts()
    assert all(lq.route_count(r) == 0 for r in range(7))
    assert lq.route_count(7) == 0


def test_argmax_argument_errors_return_before_launch(lq):
    L = lq.lib()
    a, w, c, out = 0x10000, 0x20000, 0x30000, 0x40000
    # never dereferenced: every call below fails validation
    assert L.lq_gemv_argmax(0, a, w, c, 0, 64, out, 0) == lq.LQ_ERR_INVALID_ARG      # N == 0
    assert L.lq_gemv_argmax(0, a, w, c, 1 << 30, 64, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_argmax(7, a, w, c, 8, 64, out, 0) == lq.LQ_ERR_INVALID_ARG      # format
    assert L.lq_gemv_argmax(0, a, w, c, 8, 64, None, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_argmax(0, a, w, c, 8, 64, out + 4, 0) == lq.LQ_ERR_INVALID_ARG  # 8-byte alignment
    assert L.lq_gemv_argmax(1, a, w, c, 8, 48, out, 0) == lq.LQ_ERR_INVALID_ARG      # K % 32
    assert L.lq_gemv_argmax(0, None, w, c, 8, 64, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_argmax(0, a, w, c + 2, 8, 64, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_argmax_f32(c, 0, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_argmax_f32(c, 1 << 31, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_argmax_f32(None, 8, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_argmax_f32(c + 2, 8, out, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_argmax_f32(c, 8, out + 4, 0) == lq.LQ_ERR_INVALID_ARG


def test_epilogue_argument_errors_return_before_launch(lq):
    L = lq.lib()
    a, w, r, c = 0x10000, 0x20000, 0x30000, 0x40000
    for fmt in (0, 1, 2):
        # no-ops and refusals, never dereferenced
        assert L.lq_matmul_residual(fmt, a, w, r, c, 0, 8, 64, 0) == lq.LQ_OK
        assert L.lq_matmul_swiglu(fmt, a, w, c, 3, 0, 64, 0) == lq.LQ_OK
        assert L.lq_matmul_residual(fmt, a, w, None, c, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
        assert L.lq_matmul_residual(fmt, a, w, r + 2, c, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
        assert L.lq_matmul_residual(fmt, a, w, r, None, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
        assert L.lq_matmul_swiglu(fmt, a, None, c, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
        assert L.lq_matmul_swiglu(fmt, a, w, c, -1, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
        assert L.lq_matmul_swiglu(fmt, a, w, c, 2, 1 << 29, 64, 0) == lq.LQ_ERR_UNSUPPORTED
    assert L.lq_matmul_residual(5, a, w, r, c, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_matmul_swiglu(5, a, w, c, 2, 8, 64, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_matmul_swiglu(1, a, w, c, 2, 8, 48, 0) == lq.LQ_ERR_INVALID_ARG  # K % 32


def test_topk_argument_errors_return_before_launch(lq):
    L = lq.lib()
    x, v, i, w = 0x10000, 0x20000, 0x30000, 0x40000
    assert L.lq_topk_work_bytes(0, 5) == 0 and L.lq_topk_work_bytes(10, 0) == 0
    assert L.lq_topk_work_bytes(10, 65) == 0 and L.lq_topk_work_bytes(1 << 31, 5) == 0
    assert L.lq_topk_work_bytes(1, 1) == 16  # two regions of one key
    assert L.lq_topk_work_bytes(151936, 50) > 0
    assert L.lq_topk_f32(x, 0, 5, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_topk_f32(x, 10, 0, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_topk_f32(x, 10, 65, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_topk_f32(None, 10, 5, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_topk_f32(x, 10, 5, v, i, w + 4, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_topk_f32(x, 10, 5, None, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_topk(0, x, x, None, 10, 64, 5, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG  # C required
    assert L.lq_gemv_topk(9, x, x, x, 10, 64, 5, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_topk(0, x, x, x, 0, 64, 5, v, i, w, 0) == lq.LQ_ERR_INVALID_ARG


def test_chain_argument_errors_and_limits_return_before_launch(lq):
    """lq_gemv_chain refuses bad problem lists before touching the device,
    including the f16 K limit of its warp grid (16 chunks of 256 values)."""
    L = lq.lib()
    a, w, c = 0x10000, 0x20000, 0x30000

    def call(fmt, items):
        arr = lq.gemv_problems(items)
        return L.lq_gemv_chain(fmt, arr, len(items), 0)

    assert call(7, [(a, w, c, 8, 64, 0)]) == lq.LQ_ERR_INVALID_ARG           # format
    assert L.lq_gemv_chain(0, None, 1, 0) == lq.LQ_ERR_INVALID_ARG            # no list
    assert call(0, [(a, w, c, -1, 64, 0)]) == lq.LQ_ERR_INVALID_ARG          # N < 0
    assert call(1, [(a, w, c, 8, 48, 0)]) == lq.LQ_ERR_INVALID_ARG           # K % 32
    assert call(0, [(a, None, c, 8, 64, 0)]) == lq.LQ_ERR_INVALID_ARG        # null W
    assert call(0, [(a + 4, w, c, 8, 64, 0)]) == lq.LQ_ERR_UNSUPPORTED       # A not 16-byte aligned
    assert call(1, [(a, w, c, 8, 128, 0)]) == lq.LQ_ERR_UNSUPPORTED          # K % 256 (quantised)
    assert call(0, [(a, w, c, 8, 4096 + 8, 0)]) == lq.LQ_ERR_UNSUPPORTED     # f16 K > 4096
    assert call(0, [(a, w, c, 8, 64, 0)] * 65) == lq.LQ_ERR_UNSUPPORTED      # more than 64 problems


def test_chain_refuses_misaligned_outputs_before_launch(lq):
    """Each problem's A and C must be 4-byte aligned (f16 W 2-byte aligned),
    as for lq_gemv_<fmt>: refused before any launch."""
    L = lq.lib()
    a, w, c = 0x10000, 0x20000, 0x30000
    for fmt in (0, 1, 2, 3):
        arr = lq.gemv_problems([(a, w, c + 2, 8, 256, 0)])
        assert L.lq_gemv_chain(fmt, arr, 1, 0) == lq.LQ_ERR_INVALID_ARG
        arr = lq.gemv_problems([(a, w, c, 8, 256, 0), (a + 1, w, c, 8, 256, 1)])
        assert L.lq_gemv_chain(fmt, arr, 2, 0) == lq.LQ_ERR_INVALID_ARG
    arr = lq.gemv_problems([(a, w + 1, c, 8, 256, 0)])
    assert L.lq_gemv_chain(0, arr, 1, 0) == lq.LQ_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_noalloc_argument_errors_return_before_launch(lq, fmt):
    """lq_gemm_noalloc makes the same argument checks as lq_gemm_<fmt> before
    it looks at its workspace: never dereferenced here."""
    L = lq.lib()
    a, w, c = 0x10000, 0x20000, 0x30000
    assert L.lq_gemm_noalloc(fmt, a, w, c, 0, 8, 256, 0) == lq.LQ_OK          # no-op
    assert L.lq_gemm_noalloc(fmt, a, w, c, 8, 0, 256, 0) == lq.LQ_OK
    assert L.lq_gemm_noalloc(fmt, a, w, c, 8, 8, 0, 0) == lq.LQ_ERR_INVALID_ARG   # K == 0
    assert L.lq_gemm_noalloc(fmt, a, w, c, -1, 8, 256, 0) == lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemm_noalloc(fmt, a, w, c + 2, 8, 8, 256, 0) == lq.LQ_ERR_INVALID_ARG  # C alignment
    assert L.lq_gemm_noalloc(fmt, a + 2, w, c, 8, 8, 256, 0) == lq.LQ_ERR_INVALID_ARG  # A alignment
    assert L.lq_gemm_noalloc(fmt, a, w, None, 8, 8, 256, 0) == lq.LQ_ERR_INVALID_ARG
    if fmt != 0:
        assert L.lq_gemm_noalloc(fmt, a, w, c, 8, 8, 48, 0) == lq.LQ_ERR_INVALID_ARG  # K % 32
    assert L.lq_gemm_noalloc(3, a, w, c, 8, 8, 256, 0) == lq.LQ_ERR_INVALID_ARG  # Q4_0I not taken
