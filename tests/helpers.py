"""Shared helpers for the GPU parity tests (inputs from synthetic.py, expected
values from the oracle only)."""
import numpy as np
import torch

import oracle as O


def to_dev(packed: np.ndarray, dev):
    return torch.from_numpy(np.ascontiguousarray(packed)).to(dev)


def nan_filled(M, N, dev):
    """Output buffer pre-filled with NaN so that an unwritten element shows."""
    return torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)


def check(C, y_ref, tol, what=""):
    """Element-wise |C - y_ref| <= tol, every element written and finite."""
    C = np.asarray(C, dtype=np.float64)
    assert C.shape == y_ref.shape, (C.shape, y_ref.shape)
    assert np.all(np.isfinite(C)), f"{what}: {np.count_nonzero(~np.isfinite(C))} unwritten/non-finite"
    err = np.abs(C - y_ref)
    ratio = err / tol
    bad = np.count_nonzero(ratio > 1.0)
    assert bad == 0, (f"{what}: {bad} of {C.size} outside tolerance; worst err/tol "
                      f"{ratio.max():.3g} at {np.unravel_index(ratio.argmax(), ratio.shape)}")
    return float(ratio.max())


def reference_rows(fmt, A, W, rows, tensor_core=False, chunk=16384):
    """Oracle reference for the given rows of W (packed with the oracle's own
    packer), processed in chunks of rows."""
    K = W.shape[1]
    ys, tols = [], []
    for i in range(0, len(rows), chunk):
        r = rows[i:i + chunk]
        Wr = np.ascontiguousarray(W[r])
        y, t = O.reference(fmt, A, O.pack(fmt, Wr), len(r), K, tensor_core=tensor_core)
        ys.append(y)
        tols.append(t)
    return np.concatenate(ys, axis=1), np.concatenate(tols, axis=1)
