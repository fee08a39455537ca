"""The warp-MMA tensor-core GEMM for M = 2..48 (route 5) against the oracle.

W is streamed once as stages of 256 K; each lane dequantises 8 weights of a
row exactly and rounds them to bf16, A is rounded to bf16, mma.m16n8k16
accumulates in f32: the tensor-core tolerance (5e-3 * sum|a*w| + 1e-5)
applies. Shapes: ragged row counts per CTA (N not a multiple of 8 or of the
SM count), a single stage (K = 256), more stages than ring slots (K = 4096),
one to sixteen tokens (padding rows of the 16-token MMA), 17 to 48 tokens
(two or three token groups sharing each converted weight, CTAs of up to 64 or
48 W rows; single-piece stages where two pieces would not fit twice), the router's
choice, the residual epilogue (in place too), and the shapes the kernel
refuses. Output buffers start as NaN.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _run(lq, dev, fmt, W, A, force=True):
    N, K = W.shape
    M = A.shape[0]
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    C = nan_filled(M, N, dev)
    lq.reset_counts()
    if force:
        lq.force_route(lq.ROUTE_WARP_MMA)
    try:
        getattr(lq, f"lq_gemm_{fmt}")(A.to(dev), Wd, C, M, N, K)
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    assert lq.route_count(lq.ROUTE_WARP_MMA) == 1
    return C.cpu().numpy()


def _ref(fmt, W, A):
    N, K = W.shape
    return O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M,N,K", [(2, 1, 256), (5, 7, 256), (8, 300, 512), (9, 1000, 2048), (16, 6144, 2048),
                                   (16, 777, 4096), (3, 4097, 1024), (12, 19000, 256), (16, 153, 768),
                                   (7, 300, 16384), (17, 6144, 2048), (24, 1000, 768), (32, 4096, 4096),
                                   (31, 9727, 512), (20, 5, 256), (33, 6144, 2048), (48, 1000, 768),
                                   (48, 4096, 4096), (40, 7296, 512), (40, 300, 4096), (28, 6144, 2048)])
def test_warp_mma_gemm_matches_oracle(lq, cuda_dev, fmt, M, N, K):
    W, A = synthetic.draw(M, N, K, seed=M * 31 + N + K, outlier_frac=0.05)
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M", [2, 3, 8, 16, 17, 24, 40])
def test_router_sends_two_to_forty_eight_rows_to_warp_mmas(lq, cuda_dev, fmt, M):
    # (f16 at 6144 x 2048 with more than 24 rows needs stages larger than
    # half the shared memory, so the plan refuses and the tcgen05 kernel
    # takes it)
    w = synthetic.WORKLOADS[f"gemm_{fmt}_m16_6144x2048"]
    W, A = synthetic.draw(M, w.N, w.K, seed=M)
    C = _run(lq, cuda_dev, fmt, W, A, force=False)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} M={M} router")


def test_warp_mma_wide_range_token_rows(lq, cuda_dev):
    """Rows of A far beyond f16's range and f32 subnormals (A is rounded to
    bf16, which keeps f32's exponent range)."""
    M, N, K = 16, 256, 512
    W, A = synthetic.draw(M, N, K, seed=12)
    A = A.clone()
    A[0] *= 1e30
    A[1] = A[1] * 1e-38 * 1e-3
    A[2] = 0.0
    A[3, ::2] *= 1e20
    for fmt in ("f16", "q8_0", "q4_0"):
        C = _run(lq, cuda_dev, fmt, W, A)
        y, tol = _ref(fmt, W, A)
        check(C, y, tol, f"{fmt} wide rows")


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("M", [11, 27])
def test_warp_mma_residual(lq, cuda_dev, fmt, in_place, M):
    N, K = 1500, 2048
    W, A = synthetic.draw(M, N, K, seed=70)
    R = synthetic.rand_matrix(M, N, 71, scale=3.0)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    if in_place:
        C = R.to(cuda_dev).clone()
        Rd = C
    else:
        C = nan_filled(M, N, cuda_dev)
        Rd = R.to(cuda_dev)
    lq.reset_counts()
    lq.lq_matmul_residual(fmt, A.to(cuda_dev), Wd, Rd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    assert lq.route_count(lq.ROUTE_WARP_MMA) == 1
    y, tol = _ref(fmt, W, A)
    c, t = O.residual_reference(y, tol, R.numpy())
    check(C.cpu().numpy(), c, t, f"residual {fmt} in_place={in_place}")


@pytest.mark.parametrize("fmt,M,N,K", [("q8_0", 49, 512, 512),   # more than 48 rows
                                       ("q8_0", 33, 7297, 512),  # three token groups, more than 48 rows per SM
                                       ("q8_0", 17, 9729, 512),  # two token groups, more than 64 rows per SM
                                       ("q8_0", 8, 512, 320),    # K not a multiple of 256
                                       ("q4_0i", 8, 512, 512),   # interleaved nibbles
                                       ("f16", 1, 512, 512),     # a single row (the GEMV's)
                                       ("q8_0", 8, 19457, 256)])  # more than 128 rows per SM
def test_warp_mma_refuses_other_shapes(lq, cuda_dev, fmt, M, N, K):
    W, A = synthetic.draw(M, N, K, seed=5)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    C = nan_filled(M, N, cuda_dev)
    lq.force_route(lq.ROUTE_WARP_MMA)
    try:
        with pytest.raises(lq.LQError) as e:
            getattr(lq, f"lq_gemm_{fmt}")(A.to(cuda_dev), Wd, C, M, N, K)
        assert e.value.status == lq.LQ_ERR_UNSUPPORTED
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert torch.isnan(C).all()
