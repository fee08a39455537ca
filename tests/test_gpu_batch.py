"""The batched decode kernel (M = 2..8 rows of A, route 1) against the oracle.

The router sends M = 2..4 here; five to eight rows run here when the route is
forced (the tensor cores are faster there), which these tests do.

The kernel keeps f32 activations and dequantises W exactly, so every element
is held to the GEMV tolerance (1e-4 * sum|a*w| + 1e-6), not the tensor-core
one. Shapes cover several stages per CTA with a ragged last stage, fewer rows
than SMs, the K limits of the kernel and the fallbacks beyond them (shapes it
refuses go to the tensor-core or the generic kernel and still match). Five to
eight rows use the half-block slices (each lane holds half a quantised block
for every row).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _run(lq, dev, fmt, W, A, A_dev=None, force=None):
    """lq_gemm_<fmt> on the batched kernel (a forced route: the router sends
    these shapes to the warp-MMA kernel) unless force is False."""
    N, K = W.shape
    M = A.shape[0]
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    C = nan_filled(M, N, dev)
    if force if force is not None else True:
        lq.force_route(lq.ROUTE_STREAM)
    try:
        getattr(lq, f"lq_gemm_{fmt}")(A.to(dev) if A_dev is None else A_dev, Wd, C, M, N, K)
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return C.cpu().numpy()


def _ref(fmt, W, A):
    N, K = W.shape
    return O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(5, 512), (1000, 256), (4133, 2048), (2437, 1024)])
def test_batch_matches_oracle(lq, cuda_dev, fmt, M, N, K):
    W, A = synthetic.draw(M, N, K, seed=7 * M + N + K, outlier_frac=0.05)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} {M}x{N}x{K}")
    assert lq.route_count(1) == 1


@pytest.mark.parametrize("fmt,M,N,K", [("q8_0", 4, 20000, 2048), ("q4_0", 4, 16000, 4096),
                                       ("f16", 4, 20000, 2048), ("q8_0", 2, 8192, 8192),
                                       ("q4_0", 3, 30000, 1024), ("q8_0", 8, 20000, 2048),
                                       ("q4_0", 6, 16000, 2048), ("f16", 7, 20000, 2048),
                                       ("q4_0", 5, 30000, 1024)])
def test_batch_ring_refills(lq, cuda_dev, fmt, M, N, K):
    """More stages per CTA than ring slots: slots are refilled by the stage's
    finisher while other row-groups compute, and each refill's partials reuse
    the slot's reduction buffer."""
    W, A = synthetic.draw(M, N, K, seed=N + K, outlier_frac=0.05)
    lq.reset_counts()
    for _ in range(3):  # the same result on every run
        C = _run(lq, cuda_dev, fmt, W, A)
        y, tol = _ref(fmt, W, A)
        check(C, y, tol, f"{fmt} {M}x{N}x{K}")
    assert lq.route_count(1) == 3


@pytest.mark.parametrize("fmt,K", [("f16", 1000), ("f16", 2048), ("q8_0", 4096), ("q4_0", 4096),
                                   ("q8_0", 8192), ("q4_0", 8192)])
def test_batch_k_limits(lq, cuda_dev, fmt, K):
    # two and four rows of A fit up to the largest K of the warp grid (eight
    # K-groups: 2048 f16, 8192 quantised)
    for M in (2, 4):
        W, A = synthetic.draw(M, 1536, K, seed=K + M, outlier_frac=0.05 if K % 32 == 0 else 0.0)
        lq.reset_counts()
        C = _run(lq, cuda_dev, fmt, W, A)
        y, tol = _ref(fmt, W, A)
        assert lq.route_count(1) == 1
        check(C, y, tol, f"{fmt} {M}x1536x{K}")


@pytest.mark.parametrize("fmt,K", [("f16", 4096), ("q8_0", 16384), ("q4_0", 320)])
def test_batch_refused_shapes_fall_back(lq, cuda_dev, fmt, K):
    W, A = synthetic.draw(3, 640, K, seed=K, outlier_frac=0.0)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    N = W.shape[0]
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C, y, tol, f"{fmt} 3x640x{K}")
    assert lq.route_count(1) == 0


def test_batch_unaligned_a_falls_back(lq, cuda_dev):
    fmt, M, N, K = "q8_0", 2, 700, 1024
    W, A = synthetic.draw(M, N, K, seed=11)
    buf = torch.empty(M * K + 1, dtype=torch.float32, device=cuda_dev)
    buf[1:] = A.reshape(-1).to(cuda_dev)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A, A_dev=buf[1:])
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C, y, tol, "A at a 4-byte offset")
    assert lq.route_count(1) == 0


@pytest.mark.parametrize("fmt,K,fits", [("q8_0", 2048, True), ("q8_0", 4096, True), ("q8_0", 8192, False),
                                        ("q4_0", 3072, True), ("q4_0", 8192, False),
                                        ("f16", 2048, True), ("f16", 2304, False)])
def test_batch_eight_rows_k_limits(lq, cuda_dev, fmt, K, fits):
    """Eight rows of A up to K = 4096 quantised (half-block K-groups: four per
    64-block segment, eight at most) and 2048 f16; larger K goes to the
    tensor cores."""
    M, N = 8, 1536
    W, A = synthetic.draw(M, N, K, seed=K + 8, outlier_frac=0.05)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A, force=fits)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=not fits)
    check(C, y, tol, f"{fmt} 8x{N}x{K}")
    assert lq.route_count(1) == (1 if fits else 0)


@pytest.mark.parametrize("fmt", ["q4_0i", "q8_0"])
@pytest.mark.parametrize("M", [5, 8])
def test_batch_eight_row_slices_layouts_and_epilogues(lq, cuda_dev, fmt, M):
    """The half-block slices with the pages' interleaved nibbles, and the
    residual epilogue on them."""
    N, K = 3000, 2048
    W, A = synthetic.draw(M, N, K, seed=M + 40, outlier_frac=0.05)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} {M}x{N}x{K}")
    assert lq.route_count(1) == 1
    R = torch.randn(M, N, generator=torch.Generator().manual_seed(9))
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    Cd = R.to(cuda_dev)
    lq.reset_counts()
    lq.force_route(lq.ROUTE_STREAM)
    try:
        lq.lq_matmul_residual(fmt, A.to(cuda_dev), Wd, Cd, Cd, M, N, K)  # in place: C = A W^T + C
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert lq.route_count(1) == 1
    yr, tr = O.residual_reference(y, tol, R.numpy())
    check(Cd.cpu().numpy(), yr, tr, f"{fmt} residual {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_batch_crossover_config_m2(lq, cuda_dev, fmt):
    w = synthetic.WORKLOADS[f"gemm_{fmt}_m2_6144x2048"]
    W, A = synthetic.draw_workload(w)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, w.name)
    assert lq.route_count(1) == 1


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_batch_crossover_config_m8(lq, cuda_dev, fmt):
    """The eight-row workload on the batched kernel (forced route)."""
    w = synthetic.WORKLOADS[f"gemm_{fmt}_m8_6144x2048"]
    W, A = synthetic.draw_workload(w)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, w.name)
    assert lq.route_count(1) == 1


def test_batch_rows_equal_gemv(lq, cuda_dev):
    """Each row of the batched result agrees with the GEMV of that row of A
    within twice the GEMV tolerance (the two kernels add in different
    orders)."""
    fmt, M, N, K = "q4_0", 4, 1200, 2048
    W, A = synthetic.draw(M, N, K, seed=12)
    C = _run(lq, cuda_dev, fmt, W, A)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    _, tol = _ref(fmt, W, A)
    for m in range(M):
        g = nan_filled(1, N, cuda_dev)
        lq.lq_gemv_q4_0(A[m:m + 1].contiguous().to(cuda_dev), Wd, g, 1, N, K)
        torch.cuda.synchronize()
        assert np.all(np.abs(g.cpu().numpy()[0] - C[m]) <= 2 * tol[m])
