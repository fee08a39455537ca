"""GPU parity of the decode GEMV (M == 1) through the C-ABI, against the oracle.

Small shapes span several CTAs and stages and end in ragged tails; the full
workload shapes run in the launch configuration the benchmark times (the
library's own grid and ring). Every output buffer starts as NaN so that an
unwritten row shows up.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, reference_rows, to_dev

pytestmark = pytest.mark.gpu


def _run(lq, dev, fmt, W, A, kind="gemv", w_offset=0):
    N, K = W.shape
    packed = lq.pack(fmt, W)
    flat = packed.reshape(-1).view(np.uint8)
    if w_offset:
        buf = np.zeros(flat.size + w_offset, np.uint8)
        buf[w_offset:] = flat
        Wd = to_dev(buf, dev)[w_offset:]
    else:
        Wd = to_dev(flat, dev)
    Ad = A.to(dev)
    C = nan_filled(1, N, dev)
    getattr(lq, f"lq_{kind}_{fmt}")(Ad, Wd, C, 1, N, K)
    torch.cuda.synchronize()
    assert lq.last_device_error() == lq.LQ_OK
    return C.cpu().numpy()


FAST = [("f16", k) for k in (8, 264, 512, 2048, 4104, 16384)] + \
       [(f, k) for f in ("q8_0", "q4_0") for k in (256, 512, 1280, 2048, 4096, 4352, 11008)] + \
       [("q4_0", 16384)]
GENERIC = [("f16", 7), ("f16", 1023), ("f16", 16392), ("q8_0", 96), ("q8_0", 16416),
           ("q4_0", 32), ("q4_0", 20480)]


@pytest.mark.parametrize("fmt,K", FAST + GENERIC)
@pytest.mark.parametrize("N", [1, 7, 153, 1000])
def test_gemv_small_shapes(lq, cuda_dev, fmt, K, N):
    W, A = synthetic.draw(1, N, K, seed=N * 7 + K, outlier_frac=0.05 if K % 32 == 0 else 0.0)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W.numpy(), A)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    check(C, y, tol, f"{fmt} N={N} K={K}")
    fast = (fmt, K) in FAST
    assert lq.route_count(0) == (1 if fast else 0)
    assert lq.route_count(3) == (0 if fast else 1)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "f16"])
def test_gemv_misaligned_weights_take_generic_path(lq, cuda_dev, fmt):
    N, K = 64, 512
    W, A = synthetic.draw(1, N, K, seed=5)
    lq.reset_counts()
    C = _run(lq, cuda_dev, fmt, W.numpy(), A, w_offset=2)
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    check(C, y, tol, fmt)
    assert lq.route_count(3) == 1


@pytest.mark.parametrize("kind", ["gemv", "matmul"])
def test_router_sends_m1_to_gemv(lq, cuda_dev, kind):
    W, A = synthetic.draw(1, 300, 1024, seed=9)
    lq.reset_counts()
    C = _run(lq, cuda_dev, "q8_0", W.numpy(), A, kind=kind)
    y, tol = O.reference("q8_0", A.numpy(), O.pack("q8_0", W.numpy()), 300, 1024)
    check(C, y, tol)
    assert lq.route_count(0) == 1


def test_gemv_config_f16_256x512(lq, cuda_dev):
    w = synthetic.WORKLOADS["gemv_f16_256x512"]
    W, A = synthetic.draw_workload(w)
    C = _run(lq, cuda_dev, "f16", W.numpy(), A)
    y, tol = O.reference("f16", A.numpy(), O.pack("f16", W.numpy()), w.N, w.K)
    check(C, y, tol)


@pytest.mark.parametrize("seed", list(range(8)))
def test_gemv_config_q8_0_4096x4096(lq, cuda_dev, seed):
    w = synthetic.WORKLOADS["gemv_q8_0_4096x4096"]
    W, A = synthetic.draw_workload(w, seed=seed)
    C = _run(lq, cuda_dev, "q8_0", W.numpy(), A)
    y, tol = O.reference("q8_0", A.numpy(), O.pack("q8_0", W.numpy()), w.N, w.K)
    check(C, y, tol, f"seed {seed}")


def test_gemv_config_q4_0_11008x4096_outliers(lq, cuda_dev):
    w = synthetic.WORKLOADS["gemv_q4_0_11008x4096_outliers"]
    W, A = synthetic.draw_workload(w)
    C = _run(lq, cuda_dev, "q4_0", W.numpy(), A)
    y, tol = O.reference("q4_0", A.numpy(), O.pack("q4_0", W.numpy()), w.N, w.K)
    check(C, y, tol)


def test_gemv_config_f16_lmhead_argmax(lq, cuda_dev):
    """LM head: every row against the oracle, then the argmax row index."""
    w = synthetic.WORKLOADS["gemv_f16_lmhead_151936x2048"]
    W, A = synthetic.draw_workload(w)
    Wn = W.numpy()
    del W
    C = _run(lq, cuda_dev, "f16", Wn, A)[0]
    y, tol = reference_rows("f16", A.numpy(), Wn, np.arange(w.N))
    y, tol = y[0], tol[0]
    check(C[None, :], y[None, :], tol[None, :], "lm head")
    i_ref = O.argmax_first(y)
    j = O.argmax_first(C)
    # equal, or a near-tie that no f32 kernel can resolve
    assert j == i_ref or y[i_ref] - y[j] <= tol[i_ref] + tol[j], (j, i_ref)


def test_gemv_timeout_path_reports_error(lq, cuda_dev):
    """A tiny wait limit makes the kernel's bounded waits give up at once: it
    must return LQ_ERR_DEVICE_TIMEOUT through the status word, leave the
    context usable, and compute correctly again with the default limit."""
    N = 16384  # more stages per CTA than ring slots, so the producer waits too
    W, A = synthetic.draw(1, N, 4096, seed=11)
    try:
        lq.set_wait_limit_ns(1)
        _ = lq.last_device_error()
        packed = to_dev(lq.pack("q8_0", W.numpy()), cuda_dev)
        C = nan_filled(1, N, cuda_dev)
        lq.lq_gemv_q8_0(A.to(cuda_dev), packed, C, 1, N, 4096)
        torch.cuda.synchronize()
        st = lq.last_device_error()
    finally:
        lq.set_wait_limit_ns(0)
    assert st == lq.LQ_ERR_DEVICE_TIMEOUT
    C = _run(lq, cuda_dev, "q8_0", W.numpy(), A)
    y, tol = O.reference("q8_0", A.numpy(), O.pack("q8_0", W.numpy()), N, 4096)
    check(C, y, tol)
