"""Shared helpers of the GPU parity tests (not a test module)."""
import numpy as np
import torch

import oracle as O


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> contiguous CUDA tensor; uint32 arrays travel as int32 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if a.dtype == np.int32:
        a = a.view(np.uint32)
    return a


def assert_linear_close(y_gpu: np.ndarray, X16, qw, sc, zs, inv_s, rows=None, cols=None):
    """Per-element bound |y_gpu - y_ref| <= 4e-3 * sum_k |x~ w^| + 1 fp16 ulp of y_ref.

    ``rows`` selects output channels (columns of Y) to check, ``cols`` tokens.
    """
    Xs = X16 if cols is None else X16[cols]
    if rows is not None:
        qw, sc, zs = qw[rows], sc[rows], zs[rows]
    y_ref, base = O.linear(Xs, qw, sc, zs, inv_s)
    y = y_gpu.astype(np.float64)
    if cols is not None:
        y = y[cols]
    if rows is not None:
        y = y[:, rows]
    tol = O.tolerance(y_ref, base)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not np.any(~np.isfinite(y)), "non-finite output"
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside the bound; worst ratio "
                           f"{float((err / tol).max()):.3f}")
    return float((err / tol).max())
