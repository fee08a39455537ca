"""Failure detection without a GPU fault, kernel by kernel: a wait limit of one
non-blocking poll (lq_debug_set_wait_limit_ns(1)) makes the bounded waits give
up at once; each kernel must record LQ_ERR_DEVICE_TIMEOUT in the status word,
let its own copies land, free what it holds and return, and the context must
compute correctly again with the default limit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _with_tiny_limit(lq, fn):
    try:
        lq.set_wait_limit_ns(1)
        _ = lq.last_device_error()
        fn()
        torch.cuda.synchronize()
        return lq.last_device_error()
    finally:
        lq.set_wait_limit_ns(0)


def _packed(lq, fmt, W, dev):
    return to_dev(lq.pack(fmt, W.numpy()).reshape(-1).view(np.uint8), dev)


@pytest.mark.parametrize("fmt,M,N,K", [("q8_0", 3, 20000, 2048), ("f16", 2, 8000, 1024),
                                       ("q4_0", 4, 16000, 4096), ("q8_0", 8, 20000, 2048),
                                       ("f16", 7, 8000, 1024)])
def test_batch_kernel_timeout(lq, cuda_dev, fmt, M, N, K):
    W, A = synthetic.draw(M, N, K, seed=N)
    Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)
    C = nan_filled(M, N, cuda_dev)
    lq.reset_counts()
    lq.force_route(lq.ROUTE_STREAM)  # the batched kernel, by a forced route
    try:
        st = _with_tiny_limit(lq, lambda: getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, C, M, N, K))
        assert lq.route_count(1) == 1
        assert st == lq.LQ_ERR_DEVICE_TIMEOUT
        C = nan_filled(M, N, cuda_dev)
        getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, C, M, N, K)
    finally:
        lq.force_route(0)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    check(C.cpu().numpy(), y, tol, "after the timeout")


@pytest.mark.parametrize("M,N,K,kind", [(64, 2048, 2048, "plain"), (16, 1024, 4096, "plain"),
                                        (96, 1000, 2048, "swiglu")])
def test_tensor_core_gemm_timeout(lq, cuda_dev, M, N, K, kind):
    """Includes a shape whose K is split over a cluster (the teardown's
    cluster barriers) and the SwiGLU epilogue (its named barrier)."""
    fmt = "q8_0"
    rows = 2 * N if kind == "swiglu" else N
    W, A = synthetic.draw(M, rows, K, seed=M + N)
    Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)
    C = nan_filled(M, N, cuda_dev)

    def go():
        lq.force_route(lq.ROUTE_TENSOR_CORE)  # sixteen rows would take the warp-MMA kernel
        try:
            if kind == "swiglu":
                lq.lq_matmul_swiglu(fmt, Ad, Wd, C, M, N, K)
            else:
                lq.lq_gemm_q8_0(Ad, Wd, C, M, N, K)
        finally:
            lq.force_route(0)
    lq.reset_counts()
    st = _with_tiny_limit(lq, go)
    assert lq.route_count(2) == 1
    assert st == lq.LQ_ERR_DEVICE_TIMEOUT
    C = nan_filled(M, N, cuda_dev)
    go()
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), rows, K, tensor_core=True)
    if kind == "swiglu":
        y, tol = O.swiglu_reference(y, tol, N)
    check(C.cpu().numpy(), y, tol, "after the timeout")


def test_chain_timeout(lq, cuda_dev):
    fmt, N, K = "q8_0", 8192, 4096
    W, A = synthetic.draw(1, N, K, seed=5)
    Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)[0]
    Cs = [nan_filled(1, N, cuda_dev)[0] for _ in range(3)]
    items = [(Ad, Wd, C, N, K, 0) for C in Cs]
    st = _with_tiny_limit(lq, lambda: lq.lq_gemv_chain(fmt, items))
    assert st == lq.LQ_ERR_DEVICE_TIMEOUT
    Cs = [nan_filled(1, N, cuda_dev)[0] for _ in range(3)]
    assert lq.lq_gemv_chain(fmt, [(Ad, Wd, C, N, K, 0) for C in Cs]) == lq.LQ_OK
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    for C in Cs:
        check(C.cpu().numpy()[None, :], y, tol, "chain after the timeout")


def test_fused_argmax_timeout_leaves_the_result_unwritten(lq, cuda_dev):
    fmt, N, K = "f16", 30000, 2048
    W, A = synthetic.draw(1, N, K, seed=6)
    Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)[0]
    res = lq.argmax_result(cuda_dev)
    marker = torch.tensor([7.0], dtype=torch.float32).view(torch.int32).item()
    res[0] = (7 << 32) | (marker & 0xFFFFFFFF)  # value bits 7.0, index 7
    st = _with_tiny_limit(lq, lambda: lq.lq_gemv_argmax(fmt, Ad, Wd, None, N, K, res))
    assert st == lq.LQ_ERR_DEVICE_TIMEOUT
    assert lq.read_argmax(res) == (7.0, 7)
    lq.lq_gemv_argmax(fmt, Ad, Wd, None, N, K, res)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    v, i = lq.read_argmax(res)
    i_ref = O.argmax_first(y[0])
    assert i == i_ref or y[0, i_ref] - y[0, i] <= tol[0, i_ref] + tol[0, i]


@pytest.mark.parametrize("fmt,M,N,K", [("q8_0", 16, 6144, 2048), ("f16", 5, 3000, 1024), ("q4_0", 9, 777, 4096)])
def test_warp_mma_gemm_timeout(lq, cuda_dev, fmt, M, N, K):
    """The warp-MMA kernel gives up on its stage waits, drains the copies it
    issued and leaves the context usable."""
    W, A = synthetic.draw(M, N, K, seed=N + 1)
    Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)
    C = nan_filled(M, N, cuda_dev)
    lq.reset_counts()
    st = _with_tiny_limit(lq, lambda: getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, C, M, N, K))
    assert lq.route_count(lq.ROUTE_WARP_MMA) == 1
    assert st == lq.LQ_ERR_DEVICE_TIMEOUT
    C = nan_filled(M, N, cuda_dev)
    getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, C, M, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C.cpu().numpy(), y, tol, "after the timeout")
