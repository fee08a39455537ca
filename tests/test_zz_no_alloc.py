"""lq_gemm_noalloc: the tensor-core GEMM for callers that must not allocate
device memory (runtimes that own all device memory, fixed memory budgets,
real-time paths). It runs on a fixed workspace inside the
library; these tests check, through the C-ABI, on calls in a row, that
each output matches the CPU oracle element by element within the
tensor-core tolerance, that it is bit-identical to the regular
lq_gemm_<fmt> entry point (the same kernels on the same inputs), and that a
request larger than the workspace is refused without running anything.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _packed(lq, fmt, W, dev):
    return to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)


def _reference(fmt, W, A):
    N, K = W.shape
    return O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)


@pytest.mark.parametrize("fmt", ["q8_0", "f16", "q4_0"])
def test_noalloc_matches_oracle_and_regular_gemm_on_two_calls_in_a_row(lq, cuda_dev, fmt):
    # two different problems back to back on the shared workspace (token
    # tiles whose A slice is larger than shared memory); the second is
    # smaller, so leftovers of the first would show if they were read. Then
    # two small problems whose A the GEMM keeps in shared memory itself.
    cases = [(250, 1024, 4096, 20), (128, 4096, 4096, 23), (96, 384, 1024, 21), (56, 200, 512, 22)]
    lq.force_route(0)
    for M, N, K, seed in cases:
        W, A = synthetic.draw(M, N, K, seed=seed, outlier_frac=0.05)
        Wd, Ad = _packed(lq, fmt, W, cuda_dev), A.to(cuda_dev)
        ref = nan_filled(M, N, cuda_dev)
        lq.reset_counts()
        getattr(lq, f"lq_gemm_{fmt}")(Ad, Wd, ref, M, N, K)
        assert lq.route_count(2) == 1  # the regular call took the tensor-core route
        out = nan_filled(M, N, cuda_dev)
        lq.lq_gemm_noalloc(fmt, Ad, Wd, out, M, N, K)
        torch.cuda.synchronize()
        assert lq.last_device_error() == lq.LQ_OK
        ref_h, out_h = ref.cpu().numpy(), out.cpu().numpy()
        y, tol = _reference(fmt, W, A)
        check(out_h, y, tol, f"noalloc {fmt} {M}x{N}x{K}")
        check(ref_h, y, tol, f"lq_gemm_{fmt} {M}x{N}x{K}")
        # same kernels, same inputs: the workspace must not change a bit
        assert np.array_equal(out_h.view(np.uint32), ref_h.view(np.uint32)), f"{fmt} {M}x{N}x{K}"


def test_noalloc_refuses_requests_beyond_its_workspace(lq, cuda_dev):
    M, N, K = 4096, 256, 2048  # f16 copy of A alone needs 16 MiB > 8 MiB
    A = torch.zeros((M, K), dtype=torch.float32, device=cuda_dev)
    W = torch.zeros((N, K // 32 * 34,), dtype=torch.uint8, device=cuda_dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=cuda_dev)
    st = lq.lib().lq_gemm_noalloc(lq.FMT["q8_0"], A.data_ptr(), W.data_ptr(), C.data_ptr(), M, N, K,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == lq.LQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert float(C.abs().max()) == 0.0  # nothing ran
