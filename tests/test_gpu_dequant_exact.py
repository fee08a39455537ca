"""Bit-exact dequantisation on the GPU, through the C-ABI.

A one-hot activation A = e_k makes every route return column k of the
dequantised weights: the product 1 * w is w itself and every other term is
a signed zero. On the CUDA-core routes (the decode GEMV, the batched decode
kernel for M = 2..8, whose five- to eight-row slices hold half a block per
lane, and the decode chain) the weights are dequantised exactly in f32 (f16
widened; Q8_0 d*q and Q4_0 d*(q-8), an 11-bit scale times a code of at most
8 bits), so C must equal the oracle's dequantise() of the same bytes bit for
bit. On the tensor-core route the weight operand is that
exact value rounded once to bf16 (round to nearest even), so C must equal
the oracle's bf16 rounding of it bit for bit. The only freedom is the sign
of a zero result: a weight of -0 may come back as +0 (the sum of the other
terms' +0), so zeros are compared as values.

Columns: the first and last of the row, both block parities, both nibble
halves of a Q4_0 byte, and blocks scaled x20 (the outlier blocks of the
workloads) or to large scales.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import to_dev

pytestmark = pytest.mark.gpu

N, K = 300, 1024
COLS = [0, 1, 15, 16, 31, 32, 33, 47, 63, 64 + 17, 511, 512, 1000, K - 1]


def _weights(fmt, seed):
    W, _ = synthetic.draw(1, N, K, seed=seed, outlier_frac=0.05)
    W = W.clone()
    # a few blocks with large scales and a row of zeros
    W[7, 32:64] *= 1000.0
    W[8, 0:32] *= 1e5
    W[9] = 0.0
    W[10, 960:992] = -W[10, 960:992].abs()
    # finite in f16 as well (an outlier block x20 x1e5 would round to inf there,
    # and 0 * inf = NaN is then the right product for every other column)
    return W.clamp_(-6.0e4, 6.0e4)


def _expected(fmt, W, cols, bf16=False):
    Wd = O.dequantize(fmt, O.pack(fmt, W.numpy()), N, K)[:, cols].T.astype(np.float32)
    if bf16:
        Wd = np.asarray(O.f32_to_bf16_rne(Wd), dtype=np.float32)
    return np.where(Wd == 0, np.float32(0.0), Wd)


def _bits(x):
    x = np.asarray(x, dtype=np.float32)
    return np.where(x == 0, np.float32(0.0), x).view(np.uint32)


def _onehot(cols):
    A = torch.zeros((len(cols), K), dtype=torch.float32)
    for i, k in enumerate(cols):
        A[i, k] = 1.0
    return A


def _pack(lq, fmt, W, dev):
    return to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
def test_gemv_dequantises_bit_exactly(lq, cuda_dev, fmt):
    W = _weights(fmt, 31)
    Wd = _pack(lq, fmt, W, cuda_dev)
    exp = _expected(fmt, W, COLS)
    lq.reset_counts()
    for i, k in enumerate(COLS):
        A = _onehot([k]).to(cuda_dev)
        C = torch.full((1, N), float("nan"), dtype=torch.float32, device=cuda_dev)
        getattr(lq, f"lq_gemv_{fmt}")(A, Wd, C, 1, N, K)
        torch.cuda.synchronize()
        got = C.cpu().numpy()[0]
        assert np.array_equal(_bits(got), _bits(exp[i])), f"{fmt} column {k}"
    assert lq.route_count(0) == len(COLS)  # the fast streaming kernel
    assert lq.last_device_error() == lq.LQ_OK


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8])
def test_batched_decode_dequantises_bit_exactly(lq, cuda_dev, fmt, M):
    W = _weights(fmt, 32 + M)
    Wd = _pack(lq, fmt, W, cuda_dev)
    for start in range(0, len(COLS), M):
        cols = (COLS[start:start + M] + COLS[:M])[:M]
        A = _onehot(cols).to(cuda_dev)
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device=cuda_dev)
        lq.reset_counts()
        lq.force_route(lq.ROUTE_STREAM)  # the router sends these rows to the tensor cores
        try:
            getattr(lq, f"lq_gemm_{fmt}")(A, Wd, C, M, N, K)
        finally:
            lq.force_route(0)
        torch.cuda.synchronize()
        assert lq.route_count(1) == 1
        got, exp = C.cpu().numpy(), _expected(fmt, W, cols)
        assert np.array_equal(_bits(got), _bits(exp)), f"{fmt} M={M} columns {cols}"
    assert lq.last_device_error() == lq.LQ_OK


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
def test_chain_dequantises_bit_exactly(lq, cuda_dev, fmt):
    W = _weights(fmt, 33)
    Wd = _pack(lq, fmt, W, cuda_dev)
    A = _onehot(COLS).to(cuda_dev)
    C = torch.full((len(COLS), N), float("nan"), dtype=torch.float32, device=cuda_dev)
    items = [(A[i], Wd, C[i], N, K, 0) for i in range(len(COLS))]
    lq.reset_counts()
    assert lq.lq_gemv_chain(fmt, items) == lq.LQ_OK
    torch.cuda.synchronize()
    assert lq.route_count(4) == 1
    assert np.array_equal(_bits(C.cpu().numpy()), _bits(_expected(fmt, W, COLS)))
    assert lq.last_device_error() == lq.LQ_OK


@pytest.mark.parametrize("fmt,route", [("f16", 2), ("q8_0", 2), ("q4_0", 2), ("q4_0i", 2),
                                       ("f16", 5), ("q8_0", 5), ("q4_0", 5)])
def test_tensor_core_operand_is_the_bf16_rounding_of_the_exact_weight(lq, cuda_dev, fmt, route):
    """Both tensor-core kernels: tcgen05 (route 2) and warp-level MMAs (5)."""
    W = _weights(fmt, 34)
    Wd = _pack(lq, fmt, W, cuda_dev)
    cols = COLS + COLS[:2]        # 16 tokens: one token tile
    A = _onehot(cols).to(cuda_dev)
    M = len(cols)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device=cuda_dev)
    lq.reset_counts()
    lq.force_route(route)
    try:
        getattr(lq, f"lq_gemm_{fmt}")(A, Wd, C, M, N, K)
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert lq.route_count(route) == 1
    assert np.array_equal(_bits(C.cpu().numpy()), _bits(_expected(fmt, W, cols, bf16=True)))
    assert lq.last_device_error() == lq.LQ_OK
