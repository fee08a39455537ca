"""lq_gemv_chain (the decode chain) against the oracle, problem by problem.

A dependent chain feeds every problem the previous problem's output (after
= 1), so each C_j is checked against the oracle on the GPU's own C_{j-1}
(read back), with the GEMV tolerance; both ways of running it are covered:
a new launch at each dependent problem (the default) and the in-kernel
device-wide wait (lq_debug_chain_waits). Independent problems, CTAs that own no
rows (N < number of SMs), N = 0 and the refusal of shapes outside the fast
path are covered as well.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from helpers import check, nan_filled, to_dev

pytestmark = pytest.mark.gpu


def _weights(lq, fmt, N, K, seed, dev):
    W, _ = synthetic.draw(1, N, K, seed=seed, outlier_frac=0.05 if K % 32 == 0 else 0.0)
    Wn = W.numpy()
    return Wn, to_dev(lq.pack(fmt, Wn).reshape(-1).view(np.uint8), dev)


def _run_chain(lq, fmt, items):
    st = lq.lq_gemv_chain(fmt, items)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("fmt,dims", [
    ("q8_0", [4096, 4096, 2048, 4096, 1024]),
    ("q4_0", [4096, 11008 // 256 * 256, 4096, 512]),
    ("f16", [2048, 1000 // 8 * 8, 2048, 256]),
])
@pytest.mark.parametrize("waits", [False, True])
def test_chain_dependent_matches_oracle_step_by_step(lq, cuda_dev, fmt, dims, waits):
    # problem j: K = dims[j], N = dims[j + 1]; A_j = C_{j-1} for j > 0
    torch.manual_seed(0)
    A0 = torch.randn(dims[0], dtype=torch.float32)
    Ws, items, Cs = [], [], []
    A = A0.to(cuda_dev)
    for j in range(len(dims) - 1):
        K, N = dims[j], dims[j + 1]
        Wn, Wd = _weights(lq, fmt, N, K, 100 + j, cuda_dev)
        C = nan_filled(1, N, cuda_dev)[0]
        items.append((A, Wd, C, N, K, 1 if j > 0 else 0))
        Ws.append(Wn)
        Cs.append(C)
        A = C
    lq.reset_counts()
    lq.chain_waits(waits)
    try:
        assert _run_chain(lq, fmt, items) == lq.LQ_OK
    finally:
        lq.chain_waits(False)
    assert lq.last_device_error() == lq.LQ_OK
    if waits:
        assert lq.route_count(4) == 1                 # one launch, in-kernel waits
    else:
        assert lq.route_count(0) == len(items)        # one streaming GEMV per dependent problem
    a_prev = A0.numpy()
    for j, (Wn, C) in enumerate(zip(Ws, Cs)):
        N, K = Wn.shape
        c = C.cpu().numpy()
        y, tol = O.reference(fmt, a_prev[None, :], O.pack(fmt, Wn), N, K)
        check(torch.from_numpy(c[None, :]), y, tol, f"{fmt} chain step {j} N={N} K={K}")
        a_prev = c


def test_chain_independent_problems_and_small_n(lq, cuda_dev):
    fmt = "q8_0"
    shapes = [(4096, 4096), (100, 2048), (7, 256), (0, 512), (3000, 4096), (152, 1024)]
    items, refs = [], []
    for j, (N, K) in enumerate(shapes):
        Wn, Wd = _weights(lq, fmt, max(N, 1), K, 200 + j, cuda_dev)
        Wn = Wn[:N]
        A = torch.randn(K, generator=torch.Generator().manual_seed(300 + j), dtype=torch.float32)
        C = nan_filled(1, max(N, 1), cuda_dev)[0]
        items.append((A.to(cuda_dev), Wd, C, N, K, 0))
        refs.append((Wn, A.numpy(), C, N, K))
    assert _run_chain(lq, fmt, items) == lq.LQ_OK
    assert lq.last_device_error() == lq.LQ_OK
    for Wn, a, C, N, K in refs:
        if N == 0:
            assert torch.isnan(C).all()  # nothing written
            continue
        y, tol = O.reference(fmt, a[None, :], O.pack(fmt, Wn), N, K)
        check(C[None, :N].cpu().numpy(), y, tol, f"independent N={N} K={K}")


@pytest.mark.parametrize("waits", [False, True])
def test_chain_runs_twice_in_a_row(lq, cuda_dev, waits):
    # the completion counter is reset for every call: the second call's
    # dependent problem must wait for its own first problem again
    fmt = "q4_0"
    lq.chain_waits(waits)
    K = N = 2048
    Wn, Wd = _weights(lq, fmt, N, K, 400, cuda_dev)
    A = torch.randn(K, generator=torch.Generator().manual_seed(401), dtype=torch.float32)
    Ad = A.to(cuda_dev)
    for _ in range(2):
        C1, C2 = nan_filled(1, N, cuda_dev)[0], nan_filled(1, N, cuda_dev)[0]
        assert lq.lq_gemv_chain(fmt, [(Ad, Wd, C1, N, K, 0), (C1, Wd, C2, N, N, 1)]) == lq.LQ_OK
        torch.cuda.synchronize()
        assert lq.last_device_error() == lq.LQ_OK
        c1 = C1.cpu().numpy()
        y1, tol1 = O.reference(fmt, A.numpy()[None, :], O.pack(fmt, Wn), N, K)
        check(c1[None, :], y1, tol1, "first problem")
        y2, tol2 = O.reference(fmt, c1[None, :], O.pack(fmt, Wn), N, N)
        check(C2.cpu().numpy()[None, :], y2, tol2, "second problem (reads the first's output)")
    lq.chain_waits(False)


def test_chain_runs_of_independent_problems_between_dependent_ones(lq, cuda_dev):
    """Runs of independent problems (one chain launch each) separated by
    dependent ones: every output checked on the GPU's own inputs."""
    fmt, K = "q8_0", 2048
    Ws = [_weights(lq, fmt, K, K, 600 + j, cuda_dev) for j in range(6)]
    A0 = torch.randn(K, generator=torch.Generator().manual_seed(7), dtype=torch.float32).to(cuda_dev)
    Cs = [nan_filled(1, K, cuda_dev)[0] for _ in range(6)]
    # 0, 1 independent; 2 reads C1; 3, 4 independent of each other (read C2); 5 reads C4
    srcs = [A0, A0, Cs[1], Cs[2], Cs[2], Cs[4]]
    after = [0, 0, 1, 1, 0, 1]
    items = [(srcs[j], Ws[j][1], Cs[j], K, K, after[j]) for j in range(6)]
    lq.reset_counts()
    assert _run_chain(lq, fmt, items) == lq.LQ_OK
    assert lq.last_device_error() == lq.LQ_OK
    assert lq.route_count(4) == 2 and lq.route_count(0) == 2   # runs {0, 1}, {2}, {3, 4}, {5}
    for j in range(6):
        a = srcs[j].cpu().numpy()
        y, tol = O.reference(fmt, a[None, :], O.pack(fmt, Ws[j][0]), K, K)
        check(Cs[j].cpu().numpy()[None, :], y, tol, f"problem {j}")


def test_chain_calls_back_to_back_read_and_overwrite_earlier_data(lq, cuda_dev):
    """A launch of independent problems may start while the previous kernel
    on the stream runs (its weights stream at once; A is read, and C
    written, after that kernel has completed). Three calls with no
    synchronisation between them: the second reads the first's outputs, the
    third overwrites what the second read, and a streaming GEMV then reads
    the third's output. The kernels are deterministic, so every output must
    equal, bit for bit, the same calls run with a synchronisation after
    each; that run is checked against the oracle."""
    fmt, K = "q8_0", 4096
    Ws = [_weights(lq, fmt, K, K, 700 + j, cuda_dev) for j in range(4)]
    A0 = torch.randn(K, generator=torch.Generator().manual_seed(9), dtype=torch.float32).to(cuda_dev)

    def run(sync):
        C = [nan_filled(1, K, cuda_dev)[0] for _ in range(5)]
        calls = [
            [(A0, Ws[0][1], C[0], K, K, 0), (A0, Ws[1][1], C[1], K, K, 0)],
            [(C[0], Ws[2][1], C[2], K, K, 0), (C[1], Ws[3][1], C[3], K, K, 0)],
            [(C[2], Ws[0][1], C[0], K, K, 0), (C[3], Ws[1][1], C[1], K, K, 0)],
        ]
        seen = []
        for items in calls:
            assert lq.lq_gemv_chain(fmt, items) == lq.LQ_OK
            if sync:
                torch.cuda.synchronize()
                seen.append([c.clone() for c in C])
        lq.lq_gemv_q8_0(C[0], Ws[3][1], C[4], 1, K, K)
        torch.cuda.synchronize()
        assert lq.last_device_error() == lq.LQ_OK
        return [c.cpu() for c in C], seen

    ref, seen = run(True)
    out, _ = run(False)
    for j in range(5):
        assert torch.equal(out[j].view(torch.int32), ref[j].view(torch.int32)), f"output {j}"
    # the synchronised run against the oracle, call by call on its own inputs
    after1, after2 = seen[0], seen[1]
    for src, w, dst, tag in [(A0.cpu(), 0, after1[0].cpu(), "C0"), (after1[0].cpu(), 2, after2[2].cpu(), "C2"),
                             (after2[2].cpu(), 0, ref[0], "C0 again"), (ref[0], 3, ref[4], "GEMV")]:
        y, tol = O.reference(fmt, src.numpy()[None, :], O.pack(fmt, Ws[w][0]), K, K)
        check(dst.numpy()[None, :], y, tol, tag)


def test_chain_refuses_shapes_outside_its_path(lq, cuda_dev):
    fmt = "q8_0"
    K, N = 96, 64  # K % 256 != 0
    Wn, Wd = _weights(lq, fmt, N, K, 500, cuda_dev)
    A = torch.randn(K, dtype=torch.float32, device=cuda_dev)
    C = nan_filled(1, N, cuda_dev)[0]
    assert lq.lq_gemv_chain(fmt, [(A, Wd, C, N, K, 0)]) == lq.LQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(C).all()


@pytest.mark.parametrize("K", [2304, 4096])
def test_chain_f16_single_row_group(lq, cuda_dev, K):
    """f16 beyond K = 2048 (up to 4096, the chain's f16 limit): one row-group
    of consumer warps, whose ring the plan keeps at three slots or more for
    independent problems; every problem against the oracle. Then a dependent
    pair (its second problem starts a new launch)."""
    fmt = "f16"
    items, refs = [], []
    for j, N in enumerate([4096, 1000, 152, 2048]):
        Wn, Wd = _weights(lq, fmt, N, K, 300 + j, cuda_dev)
        A = torch.randn(K, generator=torch.Generator().manual_seed(j))
        C = nan_filled(1, N, cuda_dev)[0]
        items.append((A.to(cuda_dev), Wd, C, N, K, 0))
        refs.append((Wn, A.numpy(), C))
    lq.reset_counts()
    assert _run_chain(lq, fmt, items) == lq.LQ_OK
    assert lq.last_device_error() == lq.LQ_OK and lq.route_count(4) == 1
    for Wn, a, C in refs:
        N = Wn.shape[0]
        y, tol = O.reference(fmt, a[None, :], O.pack(fmt, Wn), N, K)
        check(torch.from_numpy(C.cpu().numpy()[None, :]), y, tol, f"f16 chain N={N} K={K}")
    # a dependent pair: the second problem reads the first one's output
    Wn0, Wd0 = _weights(lq, fmt, K, K, 400, cuda_dev)
    Wn1, Wd1 = _weights(lq, fmt, 512, K, 401, cuda_dev)
    A = torch.randn(K, generator=torch.Generator().manual_seed(9))
    C0, C1 = nan_filled(1, K, cuda_dev)[0], nan_filled(1, 512, cuda_dev)[0]
    assert _run_chain(lq, fmt, [(A.to(cuda_dev), Wd0, C0, K, K, 0), (C0, Wd1, C1, 512, K, 1)]) == lq.LQ_OK
    assert lq.last_device_error() == lq.LQ_OK
    c0 = C0.cpu().numpy()
    y0, t0 = O.reference(fmt, A.numpy()[None, :], O.pack(fmt, Wn0), K, K)
    check(torch.from_numpy(c0[None, :]), y0, t0, "f16 dependent step 0")
    y1, t1 = O.reference(fmt, c0[None, :], O.pack(fmt, Wn1), 512, K)
    check(torch.from_numpy(C1.cpu().numpy()[None, :]), y1, t1, "f16 dependent step 1")
