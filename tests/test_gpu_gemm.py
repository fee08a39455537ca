"""GPU parity of the prefill GEMM (M > 1) through the C-ABI, against the oracle.

The tensor-core route rounds A to bf16 and accumulates bf16 x bf16 products
in f32; the oracle rounds A to bf16 the same way and the tolerance is
5e-3 * sum|a*w| + 1e-5 per element. Output buffers start as NaN.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _run(lq, dev, fmt, W, A, kind="gemm"):
    N, K = W.shape
    M = A.shape[0]
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    C = nan_filled(M, N, dev)
    getattr(lq, f"lq_{kind}_{fmt}")(A.to(dev), Wd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return C.cpu().numpy()


def _ref(fmt, W, A):
    N, K = W.shape
    return O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_tc_single_tile_single_kstep(lq, cuda_dev, fmt):
    W, A = synthetic.draw(16, 128, 64, seed=1)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} 16x128x64")
    assert lq.route_count(2) == 1


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M,N,K", [(2, 128, 128), (5, 200, 512), (16, 1000, 1024), (33, 384, 256),
                                   (100, 130, 2048), (256, 256, 640), (300, 515, 512)])
def test_tc_shapes(lq, cuda_dev, fmt, M, N, K):
    W, A = synthetic.draw(M, N, K, seed=M + N + K, outlier_frac=0.05)
    lq.reset_counts()
    lq.force_route(lq.ROUTE_TENSOR_CORE)  # M <= 48 would take the warp-MMA or batched kernel
    try:
        C = _run(lq, cuda_dev, fmt, W, A)
    finally:
        lq.force_route(0)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} {M}x{N}x{K}")
    assert lq.route_count(2) == 1


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M,N,K", [(300, 6144, 1024), (400, 2048, 1024), (511, 1536, 512)])
def test_tc_shapes_that_fill_the_gpu(lq, cuda_dev, fmt, M, N, K):
    """Enough output tiles for every SM (K is not split), several token tiles
    of different heights; checked on every 97th W row against the oracle."""
    W, A = synthetic.draw(M, N, K, seed=M + N, outlier_frac=0.05)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    rows = np.arange(0, N, 97)
    Wr = W[rows]
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, Wr.numpy()), len(rows), K, tensor_core=True)
    check(C[:, rows], y, tol, f"{fmt} {M}x{N}x{K}")
    assert np.all(np.isfinite(C))
    assert lq.route_count(2) == 1


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_gemm_router_and_generic_route_agree(lq, cuda_dev, fmt):
    """Every route gives the oracle's answer (forced-route test hook)."""
    W, A = synthetic.draw(24, 192, 320, seed=3)
    y, tol = _ref(fmt, W, A)
    try:
        for route in (lq.ROUTE_AUTO, lq.ROUTE_TENSOR_CORE, lq.ROUTE_GENERIC, lq.ROUTE_STREAM):
            lq.force_route(route)
            C = _run(lq, cuda_dev, fmt, W, A, kind="matmul")
            check(C, y, tol, f"route {route}")
    finally:
        lq.force_route(0)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_gemm_k_not_multiple_of_64_uses_generic(lq, cuda_dev, fmt):
    W, A = synthetic.draw(8, 96, 96, seed=4)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol)
    assert lq.route_count(2) == 0


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
def test_gemm_config_512x6144x2048(lq, cuda_dev, fmt):
    w = synthetic.WORKLOADS[f"gemm_{fmt}_512x6144x2048"]
    W, A = synthetic.draw_workload(w)
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, w.name)


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0"])
@pytest.mark.parametrize("M", [2, 16, 64])
def test_gemm_config_crossover(lq, cuda_dev, fmt, M):
    w = synthetic.WORKLOADS[f"gemm_{fmt}_m{M}_6144x2048"]
    W, A = synthetic.draw_workload(w)
    C = _run(lq, cuda_dev, fmt, W, A)
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, w.name)


def test_gemm_row_equals_gemv(lq, cuda_dev):
    """Row m of the GEMM equals the GEMV on row m of A (within the GEMM
    tolerance)."""
    W, A = synthetic.draw(8, 512, 1024, seed=6)
    C = _run(lq, cuda_dev, "q8_0", W, A)
    Wd = to_dev(lq.pack("q8_0", W).reshape(-1).view(np.uint8), cuda_dev)
    _, tol = _ref("q8_0", W, A)
    for m in range(8):
        g = nan_filled(1, 512, cuda_dev)
        lq.lq_gemv_q8_0(A[m:m + 1].contiguous().to(cuda_dev), Wd, g, 1, 512, 1024)
        torch.cuda.synchronize()
        assert np.all(np.abs(g.cpu().numpy()[0] - C[m]) <= tol[m])


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
def test_tc_wide_range_token_rows(lq, cuda_dev, fmt):
    """Token rows far wider than f16's range, against the tolerance defined on
    A rounded to bf16: [1e6, 1e-4, 1e-4, ...] with w_0 = 0 and the other
    weights of one sign (every small term errs the same way if it is
    represented coarsely), rows near f32's largest and smallest values (f32
    subnormals included), an all-zero row, and a row mixing 1e30 with 1e-30."""
    M, N, K = 64, 256, 512
    W, A = synthetic.draw(M, N, K, seed=12)
    W, A = W.clone(), A.clone()
    W[:, 0] = 0.0
    W[:8, 1:] = 0.05 + 0.05 * torch.rand(8, K - 1, generator=torch.Generator().manual_seed(3))
    A[0] = 1e-4
    A[0, 0] = 1e6
    A[1] = -1e-4
    A[1, 0] = -3e7
    A[3] *= 1e-36
    A[7] = A[7] * 1e-38 * 1e-3   # f32 subnormals
    A[11] = 0.0
    A[13] *= 1e30
    A[17, ::2] *= 1e30
    A[17, 1::2] *= 1e-30
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    assert lq.route_count(2) == 1
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} wide rows")


@pytest.mark.parametrize("fmt,d", [("q8_0", 4.0), ("q8_0", 300.0), ("q8_0", 60000.0),
                                   ("q4_0", 40.0), ("q4_0", 4000.0), ("q4_0", 60000.0),
                                   ("q4_0i", 40.0), ("f16", 60000.0 / 127)])
@pytest.mark.parametrize("M,route", [(48, 5), (64, 2)])
def test_tc_large_block_scales(lq, cuda_dev, fmt, d, M, route):
    """Blocks whose f16 scale d is large (Q8_0 weights up to 127 d, Q4_0 up to
    8 d; f16 weights near f16's largest value): the dequantised weights are
    formed exactly and rounded to bf16, so any finite block scale stays within
    the tolerance. Here a tenth of the blocks, spread over the tiles, carry
    the large scale; the rest are the workloads' N(0, 0.02). Both tensor-core
    routes: 48 rows take the warp MMAs (Q4_0I, which reorders A, the tcgen05
    GEMM), 64 the tcgen05 GEMM."""
    N, K = 384, 1024
    W, A = synthetic.draw(M, N, K, seed=21)
    W = W.clone()
    g = torch.Generator().manual_seed(5)
    nb = N * K // 32
    pick = torch.randperm(nb, generator=g)[: nb // 10]
    Wb = W.view(nb, 32)
    amax = Wb[pick].abs().amax(dim=1, keepdim=True)
    peak = 127.0 * d if fmt in ("q8_0", "f16") else 8.0 * d
    Wb[pick] = Wb[pick] / amax * peak
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W, A)
    assert lq.route_count(2 if fmt == "q4_0i" else route) == 1
    y, tol = _ref(fmt, W, A)
    check(C, y, tol, f"{fmt} d={d}")


@pytest.mark.parametrize("fmt", ["f16", "q8_0", "q4_0", "q4_0i"])
@pytest.mark.parametrize("M,N,K,kind", [(5, 200, 512, "gemm"), (16, 1000, 1024, "gemm"),
                                        (33, 384, 2048, "gemm"), (64, 2048, 2048, "gemm"),
                                        (100, 130, 2048, "gemm"), (16, 300, 1024, "swiglu"),
                                        (40, 520, 512, "residual")])
def test_tc_resident_a_equals_streamed_a(lq, cuda_dev, fmt, M, N, K, kind):
    """For small token tiles the GEMM rounds its A slice to bf16 in shared
    memory itself (no pre-pass, no workspace); an explicit A-ring depth keeps
    the streamed copy. Both hand the tensor cores the same bf16 operands in
    the same order, so C must agree bit for bit, and with the oracle."""
    rows = 2 * N if kind == "swiglu" else N
    W, A = synthetic.draw(M, rows, K, seed=M * 7 + K, outlier_frac=0.05)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), cuda_dev)
    R = torch.randn(M, N, generator=torch.Generator().manual_seed(M))
    outs = []
    for a_stages in (0, 2):
        lq.gemm_rings(a_stages, 0)
        lq.force_route(lq.ROUTE_TENSOR_CORE)
        lq.reset_counts()
        try:
            if kind == "swiglu":
                C = nan_filled(M, N, cuda_dev)
                lq.lq_matmul_swiglu(fmt, A.to(cuda_dev), Wd, C, M, N, K)
            elif kind == "residual":
                C = R.to(cuda_dev)
                lq.lq_matmul_residual(fmt, A.to(cuda_dev), Wd, C, C, M, N, K)
            else:
                C = nan_filled(M, N, cuda_dev)
                getattr(lq, f"lq_gemm_{fmt}")(A.to(cuda_dev), Wd, C, M, N, K)
            torch.cuda.synchronize()
        finally:
            lq.gemm_rings(0, 0)
            lq.force_route(0)
        assert lq.route_count(2) == 1
        assert lq.last_device_error() == lq.LQ_OK
        outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), f"{fmt} {M}x{N}x{K} {kind}"
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), rows, K, tensor_core=True)
    if kind == "swiglu":
        y, tol = O.swiglu_reference(y, tol, N)
    elif kind == "residual":
        y, tol = O.residual_reference(y, tol, R.numpy())
    check(outs[0], y, tol, f"{fmt} {M}x{N}x{K} {kind}")
