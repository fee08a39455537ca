"""lq_matmul_residual and lq_matmul_swiglu against the oracle, on every route.

Expected values: the oracle's matmul reference (GEMV tolerance on the
CUDA-core routes, the tensor-core tolerance with A rounded to bf16 on the
tensor-core route) carried through oracle.residual_reference /
oracle.swiglu_reference, whose tolerances add the epilogue's own float32
rounding. The route each case takes is checked with the launch counters.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu

ROUTE_GEMV, ROUTE_BATCH, ROUTE_TC, ROUTE_GENERIC, ROUTE_WARP = 0, 1, 2, 3, 5


def _pack_dev(lq, fmt, W, dev):
    return to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)


def _ref(fmt, A, W, tc):
    N, K = W.shape
    return O.reference(fmt, A, O.pack(fmt, W), N, K, tensor_core=tc)


def _swiglu(lq, dev, fmt, M, I, K, seed):
    W, A = synthetic.draw(M, 2 * I, K, seed=seed, outlier_frac=0.05 if K % 32 == 0 else 0.0)
    H = nan_filled(M, I, dev)
    lq.lq_matmul_swiglu(fmt, A.to(dev), _pack_dev(lq, fmt, W.numpy(), dev), H, M, I, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return W.numpy(), A.numpy(), H.cpu().numpy()


def _residual(lq, dev, fmt, M, N, K, seed, in_place=False):
    W, A = synthetic.draw(M, N, K, seed=seed, outlier_frac=0.05 if K % 32 == 0 else 0.0)
    R = synthetic.rand_matrix(M, N, seed + 1, scale=3.0)
    if in_place:
        C = R.to(dev).clone()
        Rd = C
    else:
        C = nan_filled(M, N, dev)
        Rd = R.to(dev)
    lq.lq_matmul_residual(fmt, A.to(dev), _pack_dev(lq, fmt, W.numpy(), dev), Rd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return W.numpy(), A.numpy(), R.numpy(), C.cpu().numpy()


CASES = [  # (M, rows, K, route, tensor-core tolerance)
    (1, 1000, 2048, ROUTE_GEMV, False),
    (1, 4133, 4096, ROUTE_GEMV, False),
    (2, 1000, 2048, ROUTE_BATCH, False),
    (4, 2437, 1024, ROUTE_BATCH, False),
    (6, 1000, 2048, ROUTE_BATCH, False),   # forced onto the batched kernel (residual: every M > 1; SwiGLU: from five)
    (8, 700, 1024, ROUTE_BATCH, False),
    (6, 1000, 2048, ROUTE_TC, True),       # ... where the router picks the tensor cores
    (16, 1000, 2048, ROUTE_TC, True),
    (24, 1000, 2048, ROUTE_TC, True),
    (40, 1000, 2048, ROUTE_TC, True),
    (64, 1000, 2048, ROUTE_TC, True),
    (300, 777, 1024, ROUTE_TC, True),
]


def _forced(lq, M, route, limit=1):
    """More rows than `limit` reach the batched kernel only by a forced route
    (the residual epilogue: every M > 1; SwiGLU, which the warp-MMA kernel
    does not take: five and more)."""
    if route == ROUTE_BATCH and M > limit:
        lq.force_route(lq.ROUTE_STREAM)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M,I,K,route,tc", CASES)
def test_swiglu_routes(lq, cuda_dev, fmt, M, I, K, route, tc):
    lq.reset_counts()
    _forced(lq, M, route, limit=4)
    try:
        W, A, H = _swiglu(lq, cuda_dev, fmt, M, I, K, seed=M + I + K)
    finally:
        lq.force_route(0)
    assert lq.route_count(route) == 1
    y, tol = _ref(fmt, A, W, tc)
    h, th = O.swiglu_reference(y, tol, I)
    check(H, h, th, f"swiglu {fmt} M={M} I={I} K={K}")


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M,N,K,route,tc", CASES)
def test_residual_routes(lq, cuda_dev, fmt, M, N, K, route, tc):
    lq.reset_counts()
    _forced(lq, M, route)
    try:
        W, A, R, C = _residual(lq, cuda_dev, fmt, M, N, K, seed=M + N + K)
    finally:
        lq.force_route(0)
    # up to 48 rows the tensor cores are reached by warp-level MMAs (swiglu:
    # by the tcgen05 kernel)
    assert lq.route_count(ROUTE_WARP if route == ROUTE_TC and M <= 48 else route) == 1
    y, tol = _ref(fmt, A, W, tc)
    c, tc_ = O.residual_reference(y, tol, R)
    check(C, c, tc_, f"residual {fmt} M={M} N={N} K={K}")


@pytest.mark.parametrize("M,route,tc", [(1, ROUTE_GEMV, False), (2, ROUTE_WARP, True), (40, ROUTE_WARP, True),
                                        (56, ROUTE_TC, True)])
def test_residual_in_place(lq, cuda_dev, M, route, tc):
    """R and C the same buffer: the residual stream updated in place."""
    fmt, N, K = "q8_0", 3000, 2048
    lq.reset_counts()
    W, A, R, C = _residual(lq, cuda_dev, fmt, M, N, K, seed=5, in_place=True)
    assert lq.route_count(route) == 1
    y, tol = _ref(fmt, A, W, tc)
    c, t = O.residual_reference(y, tol, R)
    check(C, c, t, "in place")


@pytest.mark.parametrize("fmt,K", [("q8_0", 96), ("f16", 20000), ("q4_0", 320)])
@pytest.mark.parametrize("M", [1, 3, 70])
def test_epilogues_outside_the_fast_paths(lq, cuda_dev, fmt, K, M):
    """Shapes no fast kernel takes (K, or K beyond the streaming limits) fall
    back to the generic kernel (or, for M > 1 where it fits, the tensor
    cores) with the same epilogue."""
    lq.reset_counts()
    I = 321
    W, A, H = _swiglu(lq, cuda_dev, fmt, M, I, K, seed=K + M)
    tc = lq.route_count(ROUTE_TC) == 1
    assert tc or lq.route_count(ROUTE_GENERIC) == 1 or lq.route_count(ROUTE_GEMV) == 1
    y, tol = _ref(fmt, A, W, tc)
    h, th = O.swiglu_reference(y, tol, I)
    check(H, h, th, f"swiglu fallback {fmt} M={M} K={K}")
    W, A, R, C = _residual(lq, cuda_dev, fmt, M, I, K, seed=K + M + 1)
    y, tol = _ref(fmt, A, W, tc)
    c, t = O.residual_reference(y, tol, R)
    check(C, c, t, f"residual fallback {fmt} M={M} K={K}")


@pytest.mark.parametrize("route", [ROUTE_GENERIC, ROUTE_BATCH])
def test_forced_routes(lq, cuda_dev, route):
    fmt, M, I, K = "q4_0", 4, 500, 1024
    try:
        lq.force_route(route)
        lq.reset_counts()
        W, A, H = _swiglu(lq, cuda_dev, fmt, M, I, K, seed=9)
        assert lq.route_count(route) == 1
    finally:
        lq.force_route(0)
    y, tol = _ref(fmt, A, W, False)
    h, th = O.swiglu_reference(y, tol, I)
    check(H, h, th, f"forced route {route}")


@pytest.mark.parametrize("I", [1, 7, 64, 65, 130])
def test_swiglu_small_and_ragged_I_on_the_tensor_cores(lq, cuda_dev, I):
    """Tiles of 64 outputs: I below, at and just past a tile boundary (the
    out-of-range gate and up rows of the last tile are zero-filled and never
    stored)."""
    fmt, M, K = "f16", 48, 512
    lq.reset_counts()
    W, A, H = _swiglu(lq, cuda_dev, fmt, M, I, K, seed=I)
    assert lq.route_count(ROUTE_TC) == 1
    y, tol = _ref(fmt, A, W, True)
    h, th = O.swiglu_reference(y, tol, I)
    check(H, h, th, f"I={I}")


def test_swiglu_equals_matmul_then_silu_mul(lq, cuda_dev):
    """The fused result agrees with the unfused one the pages run without a
    fused kernel (the GEMM into [gate | up], then silu_mul), within the
    swiglu tolerance of both."""
    fmt, M, I, K = "q8_0", 1, 2048, 2048
    W, A = synthetic.draw(M, 2 * I, K, seed=31)
    Wd = _pack_dev(lq, fmt, W.numpy(), cuda_dev)
    Ad = A.to(cuda_dev)
    H = nan_filled(M, I, cuda_dev)
    lq.lq_matmul_swiglu(fmt, Ad, Wd, H, M, I, K)
    G = nan_filled(M, 2 * I, cuda_dev)
    lq.lq_matmul_q8_0(Ad, Wd, G, M, 2 * I, K)
    torch.cuda.synchronize()
    g, u = G[:, :I].double(), G[:, I:].double()
    unfused = (g / (1 + torch.exp(-g)) * u).cpu().numpy()
    y, tol = _ref(fmt, A.numpy(), W.numpy(), False)
    _, th = O.swiglu_reference(y, tol, I)
    assert np.all(np.abs(H.cpu().numpy() - unfused) <= 2 * th)
