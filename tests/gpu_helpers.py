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


def row_sq_error_bound(X16, W16, s_c, inv_s, rows, e_ref, token_chunk=4096, **cfg):
    """Rigorous bound on |e_gpu - e_ref| per row for the squared-error pass.

    The tensor cores multiply x~ and w^ rounded to fp16 (relative error
    <= 2^-11 each) and accumulate K products in fp32; the reference output
    X W^T is accumulated in fp32 too.  So every residual is off by at most
    delta_t = u * (sum_k |x~ w^| + sum_k |x w|) with u = 2^-10 + K 2^-23, and
    by Cauchy-Schwarz  |sum (r + d)^2 - sum r^2| <= 2 sqrt(e D) + D  with
    D = sum_t delta_t^2.  The fp32 partial sums of squares (128 tokens each)
    add at most 1e-5 e.
    """
    import oracle as O
    W16 = np.asarray(W16, dtype=np.float16)
    K = W16.shape[1]
    qw, sc, zs = O.awq_pack(W16[rows], s_c, **cfg)
    aw = np.abs(O.dequant(qw, sc, zs, cfg.get("group", O.GROUP),
                          cfg.get("w_bit", O.W_BIT)).astype(np.float64))
    ww = np.abs(W16[rows].astype(np.float64))
    u = 2.0 ** -10 + K * 2.0 ** -23
    D = np.zeros(len(rows))
    for t0 in range(0, X16.shape[0], token_chunk):
        xs = X16[t0:t0 + token_chunk]
        b = np.abs(O.scaled_activations(xs, inv_s).astype(np.float64)) @ aw.T
        b += np.abs(xs.astype(np.float64)) @ ww.T
        D += ((u * b) ** 2).sum(axis=0)
    return 2 * np.sqrt(e_ref * D) + D + 1e-5 * e_ref
