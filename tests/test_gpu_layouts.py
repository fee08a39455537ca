"""The pages' own layouts on the GPU: Q4_0 with interleaved nibbles
(LQ_FMT_Q4_0I) on every route, with the epilogues and the fused argmax,
against the oracle's "q4_0i" reference; and Q8_0 packed through 1/d, which
the kernels read as any Q8_0.

Interleaved weights hold the same values as the standard layout, so the two
formats must also agree with each other within the route's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu

ROUTE_GEMV, ROUTE_BATCH, ROUTE_TC, ROUTE_GENERIC = 0, 1, 2, 3


def _run(lq, dev, fmt, W, A, kind="matmul"):
    N, K = W.shape
    M = A.shape[0]
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    C = nan_filled(M, N, dev)
    getattr(lq, f"lq_{kind}_{fmt}")(A.to(dev), Wd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K,route,tc", [
    (1, 4096, 4096, ROUTE_GEMV, False),
    (1, 1000, 256, ROUTE_GEMV, False),
    (1, 777, 96, ROUTE_GENERIC, False),
    (2, 3000, 2048, ROUTE_BATCH, False),
    (4, 1500, 8192 // 2, ROUTE_BATCH, False),
    (3, 640, 320, ROUTE_GENERIC, False),
    (64, 1000, 2048, ROUTE_TC, True),
    (300, 515, 512, ROUTE_TC, True),
])
def test_q4_0i_routes_match_oracle(lq, cuda_dev, M, N, K, route, tc):
    W, A = synthetic.draw(M, N, K, seed=M + N + K, outlier_frac=0.05)
    lq.reset_counts()
    C = _run(lq, cuda_dev, "q4_0i", W.numpy(), A)
    assert lq.route_count(route) == 1
    y, tol = O.reference("q4_0i", A.numpy(), O.pack("q4_0i", W.numpy()), N, K, tensor_core=tc)
    check(C, y, tol, f"q4_0i M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 3, 48])
def test_q4_0i_agrees_with_q4_0(lq, cuda_dev, M):
    """Same weights packed both ways: the same values, so the same results
    within the route's tolerance."""
    N, K = 2000, 1024
    W, A = synthetic.draw(M, N, K, seed=40 + M)
    c_std = _run(lq, cuda_dev, "q4_0", W.numpy(), A)
    c_il = _run(lq, cuda_dev, "q4_0i", W.numpy(), A)
    _, tol = O.reference("q4_0", A.numpy(), O.pack("q4_0", W.numpy()), N, K, tensor_core=M > 1)
    assert np.all(np.abs(c_std - c_il) <= 2 * tol)


@pytest.mark.parametrize("M,route,tc", [(1, ROUTE_GEMV, False), (3, ROUTE_BATCH, False), (64, ROUTE_TC, True)])
def test_q4_0i_epilogues(lq, cuda_dev, M, route, tc):
    I, K = 1200, 2048
    W, A = synthetic.draw(M, 2 * I, K, seed=50 + M)
    Wd = to_dev(lq.pack("q4_0i", W.numpy()).reshape(-1).view(np.uint8), cuda_dev)
    Ad = A.to(cuda_dev)
    H = nan_filled(M, I, cuda_dev)
    lq.reset_counts()
    lq.lq_matmul_swiglu("q4_0i", Ad, Wd, H, M, I, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    assert lq.route_count(route) == 1
    y, tol = O.reference("q4_0i", A.numpy(), O.pack("q4_0i", W.numpy()), 2 * I, K, tensor_core=tc)
    h, th = O.swiglu_reference(y, tol, I)
    check(H.cpu().numpy(), h, th, "q4_0i swiglu")
    R = synthetic.rand_matrix(M, 2 * I, 60 + M)
    C = nan_filled(M, 2 * I, cuda_dev)
    lq.lq_matmul_residual("q4_0i", Ad, Wd, R.to(cuda_dev), C, M, 2 * I, K)
    torch.cuda.synchronize()
    c, tc_ = O.residual_reference(y, tol, R.numpy())
    check(C.cpu().numpy(), c, tc_, "q4_0i residual")


def test_q4_0i_fused_argmax(lq, cuda_dev):
    N, K = 11008, 4096
    W, A = synthetic.draw(1, N, K, seed=70, outlier_frac=0.05)
    Wd = to_dev(lq.pack("q4_0i", W.numpy()).reshape(-1).view(np.uint8), cuda_dev)
    C = nan_filled(1, N, cuda_dev)[0]
    res = lq.argmax_result(cuda_dev)
    lq.lq_gemv_argmax("q4_0i", A.to(cuda_dev)[0], Wd, C, N, K, res)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    v, i = lq.read_argmax(res)
    c = C.cpu().numpy()
    assert i == O.argmax_first(c) and np.float32(v) == np.float32(c[i])
    y, tol = O.reference("q4_0i", A.numpy(), O.pack("q4_0i", W.numpy()), N, K)
    check(c[None, :], y, tol, "q4_0i argmax logits")


def test_q4_0i_in_the_decode_chain(lq, cuda_dev):
    """A dependent chain of interleaved-Q4_0 GEMVs, each against the oracle
    on the GPU's own previous output."""
    dims = [4096, 2048, 4096, 1024]
    torch.manual_seed(1)
    A0 = torch.randn(dims[0], dtype=torch.float32)
    items, Ws, Cs = [], [], []
    A = A0.to(cuda_dev)
    for j in range(len(dims) - 1):
        K, N = dims[j], dims[j + 1]
        W, _ = synthetic.draw(1, N, K, seed=90 + j, outlier_frac=0.05)
        Wd = to_dev(lq.pack("q4_0i", W.numpy()).reshape(-1).view(np.uint8), cuda_dev)
        C = nan_filled(1, N, cuda_dev)[0]
        items.append((A, Wd, C, N, K, 1 if j > 0 else 0))
        Ws.append((W.numpy(), Wd))
        Cs.append(C)
        A = C
    assert lq.lq_gemv_chain("q4_0i", items) == lq.LQ_OK
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    a_prev = A0.numpy()
    for (Wn, _), C in zip(Ws, Cs):
        N, K = Wn.shape
        c = C.cpu().numpy()
        y, tol = O.reference("q4_0i", a_prev[None, :], O.pack("q4_0i", Wn), N, K)
        check(c[None, :], y, tol, f"q4_0i chain N={N} K={K}")
        a_prev = c


def test_q4_0i_refused_by_the_fixed_workspace_gemm(lq, cuda_dev):
    N, K = 256, 256
    W, A = synthetic.draw(2, N, K, seed=80)
    Wd = to_dev(lq.pack("q4_0i", W.numpy()).reshape(-1).view(np.uint8), cuda_dev)
    C = nan_filled(2, N, cuda_dev)
    with pytest.raises(lq.LQError):
        lq.lq_gemm_noalloc(lq.FMT["q4_0i"], A.to(cuda_dev), Wd, C, 2, N, K)
    torch.cuda.synchronize()
    assert torch.isnan(C).all()


@pytest.mark.parametrize("M", [1, 4, 64])
def test_q8_0_packed_through_reciprocal(lq, cuda_dev, M):
    """Q8_0 bytes from the pages' rounding are ordinary Q8_0: every route
    reads them against the oracle's reference of the same bytes."""
    N, K = 1500, 2048
    W, A = synthetic.draw(M, N, K, seed=90 + M)
    packed = lq.pack("q8_0", W.numpy(), reciprocal=True)
    assert np.array_equal(packed, O.quantize_q8_0(W.numpy(), reciprocal=True))
    Wd = to_dev(packed.reshape(-1).view(np.uint8), cuda_dev)
    C = nan_filled(M, N, cuda_dev)
    lq.lq_matmul_q8_0(A.to(cuda_dev), Wd, C, M, N, K)
    torch.cuda.synchronize()
    y, tol = O.reference("q8_0", A.numpy(), packed, N, K, tensor_core=M > 1)
    check(C.cpu().numpy(), y, tol, f"q8_0 reciprocal M={M}")
