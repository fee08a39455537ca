"""Python binding of liblq, the GB300 weight-only matmul library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``liblq.so`` (built in-tree by ``gemm_gemv_f16w_gb300.build``).
The names match the C-ABI in ``include/lq.h``:

    lq_gemv_{f16,q8_0,q4_0}, lq_gemm_{f16,q8_0,q4_0}, lq_matmul_{f16,q8_0,q4_0}
    lq_pack_{f16,q8_0,q4_0}, lq_packed_bytes, lq_last_device_error, ...

Compute calls take torch CUDA tensors (A float32 [M,K], W packed bytes,
C float32 [M,N]) or raw device addresses; the stream defaults to torch's
current stream. A non-OK status raises ``LQError``. If the library is
missing, the first call fails loudly: there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# LQ_LIBRARY=debug loads the bounds-checking build (liblq_debug.so, see build.py)
LIB_PATH = os.path.join(_PKG, "liblq_debug.so" if os.environ.get("LQ_LIBRARY") == "debug" else "liblq.so")

LQ_OK, LQ_ERR_INVALID_ARG, LQ_ERR_UNSUPPORTED, LQ_ERR_CUDA, LQ_ERR_DEVICE_TIMEOUT, LQ_ERR_BOUNDS = range(6)
FMT = {"f16": 0, "q8_0": 1, "q4_0": 2, "q4_0i": 3}  # q4_0i: the pages' interleaved nibbles
ROUTE_AUTO, ROUTE_STREAM, ROUTE_TENSOR_CORE, ROUTE_GENERIC = range(4)
ROUTE_WARP_MMA = 5         # tensor cores, warp-level MMAs, M = 2..48
COUNT_CHAIN, COUNT_PREPASS = 4, 6  # route_count(): decode-chain launches, route 2's A pre-pass launches

# every symbol include/lq.h declares
EXPORTS = [
    "lq_gemv_f16", "lq_gemv_q8_0", "lq_gemv_q4_0",
    "lq_gemm_f16", "lq_gemm_q8_0", "lq_gemm_q4_0",
    "lq_matmul_f16", "lq_matmul_q8_0", "lq_matmul_q4_0",
    "lq_packed_bytes", "lq_pack_f16", "lq_pack_q8_0", "lq_pack_q4_0",
    "lq_status_string", "lq_last_device_error", "lq_version",
    "lq_debug_force_route", "lq_debug_route_count", "lq_debug_reset_counts",
    "lq_debug_set_wait_limit_ns", "lq_gemm_noalloc", "lq_debug_gemv_plan", "lq_gemv_chain", "lq_debug_gemm_rings",
    "lq_debug_gemm_pairs",
    "lq_gemv_argmax", "lq_argmax_f32", "lq_matmul_residual", "lq_matmul_swiglu",
    "lq_gemv_q4_0i", "lq_gemm_q4_0i", "lq_matmul_q4_0i", "lq_pack_q4_0i", "lq_pack_q8_0_rcp",
    "lq_topk_work_bytes", "lq_topk_f32", "lq_gemv_topk", "lq_debug_chain_waits",
]
_COMPUTE = [n for n in EXPORTS if n.split("_")[1] in ("gemv", "gemm", "matmul")]


class LQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded liblq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        for n in _COMPUTE:
            f = getattr(L, n)
            f.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            f.restype = st
        L.lq_packed_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.lq_packed_bytes.restype = ctypes.c_size_t
        for n in ("lq_pack_f16", "lq_pack_q8_0", "lq_pack_q4_0", "lq_pack_q4_0i", "lq_pack_q8_0_rcp"):
            f = getattr(L, n)
            f.argtypes = [vp, i64, i64, vp]
            f.restype = st
        L.lq_status_string.argtypes = [st]
        L.lq_status_string.restype = ctypes.c_char_p
        L.lq_last_device_error.argtypes = []
        L.lq_last_device_error.restype = st
        L.lq_version.restype = ctypes.c_char_p
        L.lq_debug_force_route.argtypes = [st]
        L.lq_debug_force_route.restype = st
        L.lq_debug_route_count.argtypes = [st]
        L.lq_debug_route_count.restype = ctypes.c_uint64
        L.lq_debug_reset_counts.argtypes = []
        L.lq_debug_reset_counts.restype = None
        L.lq_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.lq_debug_set_wait_limit_ns.restype = None
        L.lq_gemv_chain.argtypes = [st, ctypes.POINTER(GemvProblem), ctypes.c_int, vp]
        L.lq_gemv_chain.restype = st
        L.lq_debug_gemm_rings.argtypes = [ctypes.c_int, ctypes.c_int]
        L.lq_debug_gemm_rings.restype = st
        L.lq_debug_gemm_pairs.argtypes = [ctypes.c_int]
        L.lq_debug_gemm_pairs.restype = None
        L.lq_debug_chain_waits.argtypes = [ctypes.c_int]
        L.lq_debug_chain_waits.restype = None
        L.lq_debug_gemv_plan.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.lq_debug_gemv_plan.restype = st
        L.lq_gemm_noalloc.argtypes = [st, vp, vp, vp, i64, i64, i64, vp]
        L.lq_gemm_noalloc.restype = st
        L.lq_gemv_argmax.argtypes = [st, vp, vp, vp, i64, i64, vp, vp]
        L.lq_gemv_argmax.restype = st
        L.lq_argmax_f32.argtypes = [vp, i64, vp, vp]
        L.lq_argmax_f32.restype = st
        L.lq_matmul_residual.argtypes = [st, vp, vp, vp, vp, i64, i64, i64, vp]
        L.lq_matmul_residual.restype = st
        L.lq_matmul_swiglu.argtypes = [st, vp, vp, vp, i64, i64, i64, vp]
        L.lq_matmul_swiglu.restype = st
        L.lq_topk_work_bytes.argtypes = [i64, ctypes.c_int]
        L.lq_topk_work_bytes.restype = ctypes.c_size_t
        L.lq_topk_f32.argtypes = [vp, i64, ctypes.c_int, vp, vp, vp, vp]
        L.lq_topk_f32.restype = st
        L.lq_gemv_topk.argtypes = [st, vp, vp, vp, i64, i64, ctypes.c_int, vp, vp, vp, vp]
        L.lq_gemv_topk.restype = st
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().lq_status_string(int(s)).decode()


def _check(s: int, what: str) -> None:
    if s != LQ_OK:
        raise LQError(s, what)


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, A, W, C, M, N, K, stream=None) -> None:
    _check(getattr(lib(), name)(_ptr(A), _ptr(W), _ptr(C), int(M), int(N), int(K), _stream(stream)),
           name)


def _make(name):
    def f(A, W, C, M, N, K, stream=None):
        _call(name, A, W, C, M, N, K, stream)
    f.__name__ = name
    f.__doc__ = f"{name}(A, W, C, M, N, K, stream=None): see include/lq.h."
    return f


for _n in _COMPUTE:
    globals()[_n] = _make(_n)


def matmul(fmt: str, A, W, N: int, K: int, out=None, kind: str = "matmul", stream=None):
    """C = A @ W^T for packed W of format ``fmt``; A is float32 CUDA [M, K].

    ``kind`` picks the entry point: "matmul" (router), "gemv" or "gemm".
    """
    import torch
    M = A.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _call(f"lq_{kind}_{fmt}", A, W, out, M, N, K, stream)
    return out


class GemvProblem(ctypes.Structure):
    """One problem of lq_gemv_chain (the lq_gemv_problem struct of lq.h)."""
    _fields_ = [("A", ctypes.c_void_p), ("W", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("after", ctypes.c_int32)]


def gemv_problems(items):
    """ctypes array of lq_gemv_problem from (A, W, C, N, K, after) tuples."""
    arr = (GemvProblem * len(items))()
    for i, (A, W, C, N, K, after) in enumerate(items):
        arr[i] = GemvProblem(_ptr(A), _ptr(W), _ptr(C), int(N), int(K), int(after))
    return arr


def lq_gemv_chain(fmt, problems, stream=None) -> int:
    """Runs lq_gemv_chain on a ctypes array from gemv_problems (or a list of
    tuples); returns the lq_status (LQ_ERR_UNSUPPORTED is not an exception:
    the caller falls back to one lq_gemv_<fmt> per problem)."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    arr = problems if isinstance(problems, ctypes.Array) else gemv_problems(problems)
    st = lib().lq_gemv_chain(f, arr, len(arr), _stream(stream))
    if st not in (LQ_OK, LQ_ERR_UNSUPPORTED):
        _check(st, "lq_gemv_chain")
    return st


def lq_gemm_noalloc(fmt, A, W, C, M, N, K, stream=None):
    """Tensor-core GEMM on the library's fixed workspace (no device
    allocation during the call); see include/lq.h for the limits."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().lq_gemm_noalloc(f, _ptr(A), _ptr(W), _ptr(C), int(M), int(N), int(K),
                                 _stream(stream)), "lq_gemm_noalloc")


# ---- argmax ---------------------------------------------------------------
ARGMAX_RESULT_BYTES = 24  # sizeof(lq_argmax_result): value, index, 16 bytes of work


def argmax_result(dev=None):
    """A device buffer for one lq_argmax_result (int64 x 3, 8-byte aligned)."""
    import torch
    return torch.zeros(3, dtype=torch.int64, device=dev or "cuda")


def read_argmax(res):
    """(value, index) of an lq_argmax_result buffer (synchronises)."""
    raw = res.detach().cpu().numpy().view(np.uint8)
    return float(raw[0:4].view(np.float32)[0]), int(raw[4:8].view(np.int32)[0])


def lq_gemv_argmax(fmt, A, W, C, N, K, out, stream=None):
    """Fused GEMV (M = 1) + argmax into the device lq_argmax_result `out`
    (argmax_result()); C may be None. See include/lq.h."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().lq_gemv_argmax(f, _ptr(A), _ptr(W), _ptr(C), int(N), int(K), _ptr(out),
                                _stream(stream)), "lq_gemv_argmax")


def lq_argmax_f32(x, n, out, stream=None):
    """Argmax of n device floats into the device lq_argmax_result `out`."""
    _check(lib().lq_argmax_f32(_ptr(x), int(n), _ptr(out), _stream(stream)), "lq_argmax_f32")


# ---- top-k ----------------------------------------------------------------
def topk_buffers(n, k, dev=None):
    """(values, indices, work) device buffers for a top-k of n entries."""
    import torch
    dev = dev or "cuda"
    nbytes = int(lib().lq_topk_work_bytes(int(n), int(k)))
    if nbytes == 0:
        raise LQError(LQ_ERR_INVALID_ARG, "lq_topk_work_bytes")
    return (torch.empty(k, dtype=torch.float32, device=dev), torch.empty(k, dtype=torch.int32, device=dev),
            torch.empty(nbytes // 8, dtype=torch.int64, device=dev))


def lq_topk_f32(x, n, k, values, indices, work, stream=None):
    _check(lib().lq_topk_f32(_ptr(x), int(n), int(k), _ptr(values), _ptr(indices), _ptr(work),
                             _stream(stream)), "lq_topk_f32")


def lq_gemv_topk(fmt, A, W, C, N, K, k, values, indices, work, stream=None):
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().lq_gemv_topk(f, _ptr(A), _ptr(W), _ptr(C), int(N), int(K), int(k), _ptr(values),
                              _ptr(indices), _ptr(work), _stream(stream)), "lq_gemv_topk")


# ---- epilogue fusions ----------------------------------------------------
def lq_matmul_residual(fmt, A, W, R, C, M, N, K, stream=None):
    """C = A W^T + R (R may be C); see include/lq.h."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().lq_matmul_residual(f, _ptr(A), _ptr(W), _ptr(R), _ptr(C), int(M), int(N), int(K),
                                    _stream(stream)), "lq_matmul_residual")


def lq_matmul_swiglu(fmt, A, W, H, M, I, K, stream=None):
    """H = silu(A gate^T) * (A up^T) for W = [gate; up] (2I rows); see
    include/lq.h."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib().lq_matmul_swiglu(f, _ptr(A), _ptr(W), _ptr(H), int(M), int(I), int(K), _stream(stream)),
           "lq_matmul_swiglu")


# ---- host packers --------------------------------------------------------
def packed_bytes(fmt: str, N: int, K: int) -> int:
    return int(lib().lq_packed_bytes(FMT[fmt], int(N), int(K)))


def pack(fmt: str, W, reciprocal: bool = False) -> np.ndarray:
    """Pack f32 weights [N, K] (numpy or CPU torch) on the host.

    Returns uint16 [N, K] for f16 and uint8 [N, K/32*34 or *18] otherwise.
    fmt "q4_0i" stores the pages' interleaved nibble order; reciprocal=True
    packs Q8_0 with the pages' q = round(x * (1/d)).
    """
    if hasattr(W, "detach"):
        W = W.detach().cpu().numpy()
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    nbytes = packed_bytes(fmt, N, K)
    if nbytes == 0 and N * K > 0:
        raise LQError(LQ_ERR_INVALID_ARG, f"lq_pack_{fmt}")
    if fmt == "f16":
        out = np.empty((N, K), dtype=np.uint16)
    else:
        out = np.empty((N, nbytes // max(N, 1)), dtype=np.uint8)
    name = "lq_pack_q8_0_rcp" if (reciprocal and fmt == "q8_0") else f"lq_pack_{fmt}"
    _check(getattr(lib(), name)(W.ctypes.data, N, K, out.ctypes.data), name)
    return out


def lq_pack_f16(W) -> np.ndarray:
    return pack("f16", W)


def lq_pack_q4_0i(W) -> np.ndarray:
    return pack("q4_0i", W)


def lq_pack_q8_0_rcp(W) -> np.ndarray:
    return pack("q8_0", W, reciprocal=True)


def lq_pack_q8_0(W) -> np.ndarray:
    return pack("q8_0", W)


def lq_pack_q4_0(W) -> np.ndarray:
    return pack("q4_0", W)


# ---- status and test hooks -----------------------------------------------
def last_device_error() -> int:
    return int(lib().lq_last_device_error())


def version() -> str:
    return lib().lq_version().decode()


def force_route(route: int) -> None:
    _check(lib().lq_debug_force_route(int(route)), "lq_debug_force_route")


def route_count(route: int) -> int:
    return int(lib().lq_debug_route_count(int(route)))


def reset_counts() -> None:
    lib().lq_debug_reset_counts()


def set_wait_limit_ns(ns: int) -> None:
    lib().lq_debug_set_wait_limit_ns(int(ns))


def gemv_plan(ctas_per_sm: int = 0, rows_per_stage: int = 0, smem_bytes: int = 0) -> None:
    """Override the decode GEMV's launch plan (0 = automatic); tuning only."""
    _check(lib().lq_debug_gemv_plan(int(ctas_per_sm), int(rows_per_stage), int(smem_bytes)),
           "lq_debug_gemv_plan")


def chain_waits(on: bool) -> None:
    """Dependent problems of lq_gemv_chain wait inside one launch (True) or
    start a new launch (False, the default); for comparisons."""
    lib().lq_debug_chain_waits(1 if on else 0)


def gemm_pairs(on: bool) -> None:
    """Let the tensor-core GEMM pair CTAs on 256-row MMAs where they fit
    (True) or never (False, the default); for comparisons."""
    lib().lq_debug_gemm_pairs(1 if on else 0)


def gemm_rings(a_stages: int = 0, raw_stages: int = 0) -> None:
    """Override the tensor-core GEMM's ring depths (0 = automatic); tuning only."""
    _check(lib().lq_debug_gemm_rings(int(a_stages), int(raw_stages)), "lq_debug_gemm_rings")
