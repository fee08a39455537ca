"""The bounds-checking build (liblq_debug.so, compiled with LQ_DEBUG_BOUNDS).

In that build every kernel checks the global indices it computes (and the
row ranges of its bulk weight copies) before the access; a failed check
records LQ_ERR_BOUNDS and skips the access instead of faulting. This test
builds it and, in a child process that loads only the debug library
(LQ_LIBRARY=debug), runs every route on small odd shapes (ragged row counts,
partial tiles and stages, K not a multiple of the fast paths' steps), and the
opt-in CTA pairs of the tensor-core GEMM on one ragged shape: each call must
leave the status word clean and match the CPU oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch
import gemm_gemv_f16w_gb300 as lq
import oracle as O, synthetic
from helpers import check, nan_filled, to_dev
assert lq.LIB_PATH.endswith("liblq_debug.so"), lq.LIB_PATH
assert "debug" in lq.version(), lq.version()
dev = torch.device("cuda:0")
torch.cuda.set_device(dev)

def clean(what):
    torch.cuda.synchronize()
    st = lq.last_device_error()
    assert st == lq.LQ_OK, f"{what}: {lq.status_string(st)}"

runs = 0
for fmt in ("f16", "q8_0", "q4_0", "q4_0i"):
    for (M, N, K, route) in [(1, 301, 512, 0), (1, 37, 1024, 3), (1, 1000, 96, 0),
                             (2, 519, 256, 0), (3, 1003, 1024, 0), (5, 777, 512, 0), (8, 130, 2048, 0),
                             (16, 200, 512, 0), (37, 129, 768, 0), (300, 515, 256, 0), (6, 77, 96, 0),
                             (24, 192, 320, 2), (7, 100, 160, 1), (9, 300, 512, 3), (6, 300, 512, 1),
                             (3, 257, 2048, 1), (11, 1000, 768, 5), (2, 19, 256, 5), (40, 300, 512, 5)]:
        if fmt == "f16" or K % 32 == 0:
            W, A = synthetic.draw(M, N, K, seed=M + N + K, outlier_frac=0.05 if K % 32 == 0 else 0.0)
            Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
            C = nan_filled(M, N, dev)
            lq.force_route(route)
            try:
                getattr(lq, f"lq_matmul_{fmt}")(A.to(dev), Wd, C, M, N, K)
            except lq.LQError as e:
                assert route in (2, 5) and e.status == lq.LQ_ERR_UNSUPPORTED
                continue
            finally:
                lq.force_route(0)
            clean(f"{fmt} {M}x{N}x{K} route {route}")
            y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=M > 1)
            check(C.cpu().numpy(), y, tol, f"{fmt} {M}x{N}x{K}")
            runs += 1
    # epilogues, the decode chain, the fused argmax and the no-allocation GEMM
    for M in (1, 3, 6, 40):
        N, K = 203, 512
        W, A = synthetic.draw(M, 2 * N, K, seed=M + 7)
        Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
        H = nan_filled(M, N, dev)
        lq.lq_matmul_swiglu(fmt, A.to(dev), Wd, H, M, N, K)
        clean(f"swiglu {fmt} M={M}")
        # SwiGLU on the tensor cores from five rows, the residual from two
        y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), 2 * N, K, tensor_core=M > 4)
        h, th = O.swiglu_reference(y, tol, N)
        check(H.cpu().numpy(), h, th, f"swiglu {fmt} M={M}")
        R = torch.randn(M, 2 * N)
        Cd = R.to(dev)
        lq.lq_matmul_residual(fmt, A.to(dev), Wd, Cd, Cd, M, 2 * N, K)
        clean(f"residual {fmt} M={M}")
        y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), 2 * N, K, tensor_core=M > 1)
        yr, tr = O.residual_reference(y, tol, R.numpy())
        check(Cd.cpu().numpy(), yr, tr, f"residual {fmt} M={M}")
        runs += 2
    dims = [512, 300, 768, 520]
    items, Ws, Cs = [], [], []
    for j in range(3):
        K, N = dims[j], dims[j + 1]
        K = K // 256 * 256 or 256 if fmt != "f16" else K // 8 * 8
        W, _ = synthetic.draw(1, N, K, seed=50 + j)
        Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
        A_j = torch.randn(K).to(dev)
        C = torch.full((N,), float("nan"), device=dev)
        items.append((A_j, Wd, C, N, K, 0))
        Ws.append((W, A_j))
        Cs.append(C)
    st = lq.lq_gemv_chain(fmt, items)
    clean(f"chain {fmt}")
    if st == lq.LQ_OK:
        for (W, A_j), C in zip(Ws, Cs):
            N, K = W.shape
            y, tol = O.reference(fmt, A_j.cpu().numpy()[None, :], O.pack(fmt, W.numpy()), N, K)
            check(C.cpu().numpy()[None, :], y, tol, f"chain {fmt}")
        runs += 1
    N, K = 1001, 512
    W, A = synthetic.draw(1, N, K, seed=3)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    res = lq.argmax_result(dev)
    lq.lq_gemv_argmax(fmt, A.to(dev), Wd, None, N, K, res)
    clean(f"argmax {fmt}")
    y, _ = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K)
    assert lq.read_argmax(res)[1] == int(np.argmax(y[0]))
    runs += 1
    if fmt != "q4_0i":
        M, N, K = 33, 300, 512
        W, A = synthetic.draw(M, N, K, seed=4)
        Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
        C = nan_filled(M, N, dev)
        lq.lq_gemm_noalloc(fmt, A.to(dev), Wd, C, M, N, K)
        clean(f"noalloc {fmt}")
        y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
        check(C.cpu().numpy(), y, tol, f"noalloc {fmt}")
        runs += 1
# the tensor-core GEMM as CTA pairs (opt-in): ragged token and W tiles
for fmt in ("f16", "q8_0", "q4_0"):
    M, N, K = 1000, 1000, 1024
    W, A = synthetic.draw(M, N, K, seed=11)
    Wd = to_dev(lq.pack(fmt, W).reshape(-1).view(np.uint8), dev)
    C = nan_filled(M, N, dev)
    lq.reset_counts()
    lq.gemm_pairs(True)
    try:
        getattr(lq, f"lq_gemm_{fmt}")(A.to(dev), Wd, C, M, N, K)
    finally:
        lq.gemm_pairs(False)
    clean(f"pairs {fmt}")
    assert lq.route_count(7) == 1
    y, tol = O.reference(fmt, A.numpy(), O.pack(fmt, W.numpy()), N, K, tensor_core=True)
    check(C.cpu().numpy(), y, tol, f"pairs {fmt}")
    runs += 1
x = torch.randn(5003).to(dev)
v, i, w = lq.topk_buffers(5003, 17, dev)
lq.lq_topk_f32(x, 5003, 17, v, i, w)
clean("topk")
assert list(i.cpu().numpy()) == list(np.argsort(-x.cpu().numpy(), kind="stable")[:17])
print("debug-bounds runs:", runs)
'''


def test_debug_bounds_build_runs_every_route_clean(lq, cuda_dev):
    from gemm_gemv_f16w_gb300 import build as b
    b.build(debug_bounds=True)
    env = dict(os.environ, LQ_LIBRARY="debug",
               PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                       stderr=subprocess.STDOUT, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:]
    assert "debug-bounds runs:" in r.stdout
