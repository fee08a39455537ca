"""Seeded synthetic inputs for the weight-only matmul C[M,N] = A[M,K] @ W[N,K]^T.

This module only draws random numbers and names the workload shapes. It holds
none of the method's arithmetic (no rounding, no quantisation, no matmul), so
both the CPU oracle and the CUDA path can take their inputs from it.

Recipe (fixed for every workload):

* ``g = torch.Generator().manual_seed(seed)`` on the CPU.
* ``W = torch.randn(N, K, generator=g) * 0.02`` (float32), drawn first.
* ``A = torch.randn(M, K, generator=g)`` (float32, N(0, 1)), drawn second.
* Outlier workloads then draw ``torch.randperm(N*K/32, generator=g)`` and
  multiply the first ``round(frac * N*K/32)`` 32-element blocks of W (blocks
  counted row-major along K) by ``outlier_scale`` before any packing.

The shapes are the ones the source pages use for decode and prefill of a
Qwen-style model: a small f16 GEMV, a 4096x4096 Q8_0 projection, the
11008x4096 FFN up-projection in Q4_0 with outlier blocks, the 151936x2048 f16
LM head, and a 512-token prefill GEMM over a 6144x2048 weight.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

FORMATS = ("f16", "q8_0", "q4_0")


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str
    M: int
    N: int
    K: int
    seeds: tuple = (0,)
    outlier_frac: float = 0.0
    outlier_scale: float = 20.0
    notes: str = ""

    @property
    def kind(self) -> str:
        return "gemv" if self.M == 1 else "gemm"


def _wl(*a, **k) -> Workload:
    return Workload(*a, **k)


# The five workload families, by shape. The first one is small enough for the
# oracle to finish in milliseconds.
WORKLOADS = {
    w.name: w
    for w in [
        _wl("gemv_f16_256x512", "f16", 1, 256, 512),
        _wl("gemv_q8_0_4096x4096", "q8_0", 1, 4096, 4096, seeds=tuple(range(8))),
        _wl("gemv_q4_0_11008x4096_outliers", "q4_0", 1, 11008, 4096,
            outlier_frac=0.05, outlier_scale=20.0),
        _wl("gemv_f16_lmhead_151936x2048", "f16", 1, 151936, 2048,
            notes="argmax of C[0,:] is checked"),
    ]
    + [_wl(f"gemm_{f}_512x6144x2048", f, 512, 6144, 2048) for f in FORMATS]
    + [_wl(f"gemm_{f}_m{m}_6144x2048", f, m, 6144, 2048)
       for m in (2, 4, 8, 16, 32, 64) for f in FORMATS]
}


def n_outlier_blocks(N: int, K: int, frac: float) -> int:
    """Exact count of outlier blocks: round(frac * N*K/32), half away from zero."""
    nb = N * K // 32
    x = frac * nb
    return int(x + 0.5)


def draw(M: int, N: int, K: int, seed: int, outlier_frac: float = 0.0,
         outlier_scale: float = 20.0):
    """Draw (W f32 [N,K], A f32 [M,K]) on the CPU with the fixed recipe."""
    g = torch.Generator().manual_seed(int(seed))
    W = torch.randn(N, K, generator=g, dtype=torch.float32) * 0.02
    A = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outlier_frac > 0.0:
        if K % 32:
            raise ValueError("outlier blocks need K % 32 == 0")
        nb = N * K // 32
        pick = torch.randperm(nb, generator=g)[: n_outlier_blocks(N, K, outlier_frac)]
        Wb = W.view(nb, 32)
        Wb[pick] *= outlier_scale
    return W.contiguous(), A.contiguous()


def draw_workload(w: Workload, seed: int | None = None, M: int | None = None):
    """Inputs of a named workload (optionally with another M, e.g. for a sample)."""
    s = w.seeds[0] if seed is None else seed
    return draw(w.M if M is None else M, w.N, w.K, s, w.outlier_frac, w.outlier_scale)


def rand_matrix(rows: int, cols: int, seed: int, scale: float = 1.0):
    """A plain N(0, scale^2) float32 matrix (for edge-case tests)."""
    g = torch.Generator().manual_seed(int(seed))
    return (torch.randn(rows, cols, generator=g, dtype=torch.float32) * scale).contiguous()
