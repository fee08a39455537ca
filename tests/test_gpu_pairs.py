"""The tensor-core GEMM run as CTA pairs (route 2; W row tiles 2i and 2i + 1
on one 256-row cta_group::2 MMA, each CTA holding half of the token tile).

Pairs are opt-in (lq_debug_gemm_pairs(1); they measured slower than single
CTAs) and taken where A is streamed without a K split and the number of W
row tiles is even; the shapes below are such (ragged token tiles, a ragged
last W tile, both epilogues that pairs take, Q4_0I's reordered A). Each call
is checked against the oracle and, bit for bit, against the same GEMM with
pairs switched off: both hand the tensor cores the same bf16 operands in
the same K order.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu

PAIR_LAUNCHES = 7   # lq_debug_route_count: route-2 GEMMs launched as CTA pairs


def _call(lq, fmt, kind, Ad, Wd, R, M, N, K, dev):
    C = nan_filled(M, N, dev)
    if kind == "residual":
        C.copy_(R)
        lq.lq_matmul_residual(fmt, Ad, Wd, C, C, M, N, K)
    else:
        getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return C.cpu().numpy()


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
@pytest.mark.parametrize("M,N,K,kind", [(512, 2560, 2048, "gemm"), (1000, 1000, 1024, "gemm"),
                                        (700, 1280, 1024, "residual")])
def test_pairs_equal_oracle_and_unpaired(lq, cuda_dev, fmt, M, N, K, kind):
    W, A = synthetic.draw(M, N, K, seed=M + N + K, outlier_frac=0.05)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    Ad = A.to(cuda_dev)
    R = torch.randn(M, N, generator=torch.Generator().manual_seed(7)).to(cuda_dev)
    lq.reset_counts()
    C2 = _call(lq, fmt, kind, Ad, Wd, R, M, N, K, cuda_dev)
    assert lq.route_count(2) == 1 and lq.route_count(PAIR_LAUNCHES) == 0
    lq.gemm_pairs(True)
    try:
        C1 = _call(lq, fmt, kind, Ad, Wd, R, M, N, K, cuda_dev)
        assert lq.route_count(2) == 2 and lq.route_count(PAIR_LAUNCHES) == 1
    finally:
        lq.gemm_pairs(False)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    if kind == "residual":
        y, tol = O.residual_reference(y, tol, R.cpu().numpy())
    check(C1, y, tol, f"{fmt} {M}x{N}x{K} {kind} pairs")
    assert np.array_equal(C1, C2), f"{fmt} {M}x{N}x{K}: pairs and single CTAs differ"


def test_pairs_full_size_prefill(lq, cuda_dev):
    """The 512 x 6144 x 2048 Q8_0 prefill GEMM (token tiles of 176, 72 pairs)."""
    fmt, M, N, K = "q8_0", 512, 6144, 2048
    W, A = synthetic.draw(M, N, K, seed=9)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    lq.reset_counts()
    lq.gemm_pairs(True)
    try:
        C = _call(lq, fmt, "gemm", A.to(cuda_dev), Wd, None, M, N, K, cuda_dev)
    finally:
        lq.gemm_pairs(False)
    assert lq.route_count(PAIR_LAUNCHES) == 1
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C, y, tol, "q8_0 512x6144x2048 pairs")


def test_odd_tile_count_runs_unpaired(lq, cuda_dev):
    """Nine W row tiles: no pairs, the single-CTA kernel, even with pairs on."""
    fmt, M, N, K = "q8_0", 1000, 1100, 1024
    W, A = synthetic.draw(M, N, K, seed=3)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    lq.reset_counts()
    lq.gemm_pairs(True)
    try:
        C = _call(lq, fmt, "gemm", A.to(cuda_dev), Wd, None, M, N, K, cuda_dev)
    finally:
        lq.gemm_pairs(False)
    assert lq.route_count(2) == 1 and lq.route_count(PAIR_LAUNCHES) == 0
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C, y, tol, "q8_0 odd tiles")
