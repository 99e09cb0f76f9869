"""Python binding of ``libawq.so``: the B300 AWQ W4A16 group-quantized linear.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch provides device memory and streams.  The library must have been built
(``python weight_only_bit_05_b300/build.py``); importing this module without it
raises, there is no fallback path.

Functions take and return CUDA tensors on the current device and enqueue on
the current torch stream:

* ``absmean(X)``                      -> a fp32 [K]
* ``channel_scales(a, alpha)``        -> (s_c, inv_s) fp32 [K]
* ``pack(W, s_c=None)``               -> (qweight int32 [N, K/8], scales fp16 [N, K/128],
                                          zeros int32 [N, ceil(G/8)])
* ``gemv(X, qweight, scales, zeros, inv_s=None)``  M <= 8, CUDA cores
* ``gemm(X, qweight, scales, zeros, inv_s=None)``  any M, tensor cores
* ``search(X_cal, W, n_grid=20)``     -> dict(best, alpha, mse, s_c, inv_s, row_err)

Packed integer tensors are int32 tensors holding the uint32 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

__all__ = ["lib", "LIB_PATH", "AwqError", "exported_symbols", "absmean", "channel_scales", "pack",
           "gemv", "gemm", "search", "check_device_error", "gemm_workspace_bytes",
           "gemv_silu_mul", "gemm_silu_mul", "fold_inv_scales", "clip_search", "pack_clipped",
           "measure_stream_read", "debug_stall"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libawq.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "awq.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python weight_only_bit_05_b300/build.py` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)


class AwqConfig(ctypes.Structure):
    _fields_ = [("w_bit", ctypes.c_int32), ("group", ctypes.c_int32),
                ("zero_point", ctypes.c_int32), ("n_grid", ctypes.c_int32)]


_p, _i32, _i64, _sz, _f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_double
_SIGS = {
    "awq_default_config": (AwqConfig, []),
    "awq_last_error_string": (ctypes.c_char_p, []),
    "awq_check_device_error": (ctypes.c_int, [_p]),
    "awq_absmean_workspace_size": (_sz, [_i64, _i32]),
    "awq_absmean": (ctypes.c_int, [_p, _i64, _i32, _p, _p, _sz, _p]),
    "awq_channel_scales": (ctypes.c_int, [_p, _i32, _f64, _p, _p, _p]),
    "awq_pack": (ctypes.c_int, [_p, _p, _i32, _i32, ctypes.POINTER(AwqConfig), _p, _p, _p, _p]),
    "awq_gemv": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p, _i32, _i32, _p, _p]),
    "awq_gemm_workspace_size": (_sz, [_i32, _i32, _i32]),
    "awq_gemm": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p, _i32, _i32, _p, _p, _sz, _p]),
    "awq_gemv_silu_mul": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p, _i32, _i32, _p, _p]),
    "awq_gemm_silu_mul": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p, _i32, _i32, _p, _p, _sz, _p]),
    "awq_gemv_ex": (ctypes.c_int, [ctypes.POINTER(AwqConfig), _p, _i32, _p, _p, _p, _p, _i32,
                                   _i32, _p, _p]),
    "awq_gemm_ex": (ctypes.c_int, [ctypes.POINTER(AwqConfig), _p, _i32, _p, _p, _p, _p, _i32,
                                   _i32, _p, _p, _sz, _p]),
    "awq_fold_inv_scales": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _p]),
    "awq_clip_search_workspace_size": (_sz, [_i64, _i32, ctypes.POINTER(AwqConfig)]),
    "awq_clip_search": (ctypes.c_int, [_p, _i64, _p, _i32, _i32, _p, _p,
                                       ctypes.POINTER(AwqConfig), _i32, _p, _sz, _p, _p, _p]),
    "awq_pack_clipped": (ctypes.c_int, [_p, _p, _i32, _i32, ctypes.POINTER(AwqConfig), _p, _i32,
                                        _p, _p, _p, _p]),
    "awq_measure_stream_read": (ctypes.c_int, [_p, _sz, _i32, _p, _p]),
    "awq_debug_stall": (ctypes.c_int, [_i32, _i64]),
    "awq_search_workspace_size": (_sz, [_i64, _i32, _i32]),
    "awq_search_scales": (ctypes.c_int, [_p, _i64, _p, _i32, _i32, ctypes.POINTER(AwqConfig), _p,
                                         _sz, _p, _p, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_double), _p, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

STATUS = {0: "AWQ_OK", 1: "AWQ_ERR_SHAPE", 2: "AWQ_ERR_NULL", 3: "AWQ_ERR_ALIGN",
          4: "AWQ_ERR_CUDA", 5: "AWQ_ERR_UNSUPPORTED", 6: "AWQ_ERR_WORKSPACE",
          7: "AWQ_ERR_DEVICE"}


class AwqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def exported_symbols():
    """Function names declared in include/awq.h."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(awq_\w+)\s*\(", txt, re.M)))


def _check(code: int):
    if code != 0:
        raise AwqError(code, lib.awq_last_error_string().decode())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def check_device_error():
    _check(lib.awq_check_device_error(_stream()))


def absmean(X: torch.Tensor) -> torch.Tensor:
    _dev(X, torch.float16, "X")
    T, K = X.shape
    a = torch.empty(K, dtype=torch.float32, device=X.device)
    ws = torch.empty(max(16, lib.awq_absmean_workspace_size(T, K)), dtype=torch.uint8, device=X.device)
    _check(lib.awq_absmean(_ptr(X), T, K, _ptr(a), _ptr(ws), ws.numel(), _stream()))
    return a


def channel_scales(a: torch.Tensor, alpha: float):
    _dev(a, torch.float32, "a")
    K = a.numel()
    s = torch.empty_like(a)
    inv = torch.empty_like(a)
    _check(lib.awq_channel_scales(_ptr(a), K, float(alpha), _ptr(s), _ptr(inv), _stream()))
    return s, inv


def _cfg(w_bit=4, group=128, zero_point=True, n_grid=20):
    c = lib.awq_default_config()
    c.w_bit, c.group, c.zero_point, c.n_grid = w_bit, group, int(bool(zero_point)), n_grid
    return c


def pack(W: torch.Tensor, s_c: torch.Tensor | None = None, w_bit: int = 4, group: int = 128,
         zero_point: bool = True, out=None):
    """(qweight, scales, zeros) of W; ``out`` = existing (qweight, scales, zeros)
    buffers to write into."""
    _dev(W, torch.float16, "W")
    if s_c is not None:
        _dev(s_c, torch.float32, "s_c")
    N, K = W.shape
    c = 32 // w_bit
    G = K // group
    if out is not None:
        qweight, scales, zeros = out
        _dev(qweight, torch.int32, "qweight")
        _dev(scales, torch.float16, "scales")
        _dev(zeros, torch.int32, "zeros")
        if (tuple(qweight.shape), tuple(scales.shape), tuple(zeros.shape)) != \
                ((N, K // c), (N, G), (N, (G + c - 1) // c)):
            raise ValueError("pack: out buffers have the wrong shapes")
    else:
        qweight = torch.empty((N, K // c), dtype=torch.int32, device=W.device)
        scales = torch.empty((N, G), dtype=torch.float16, device=W.device)
        zeros = torch.empty((N, (G + c - 1) // c), dtype=torch.int32, device=W.device)
    cfg = _cfg(w_bit, group, zero_point)
    _check(lib.awq_pack(_ptr(W), _ptr(s_c), N, K, ctypes.byref(cfg), _ptr(qweight), _ptr(scales),
                        _ptr(zeros), _stream()))
    return qweight, scales, zeros


def _linear_args(X, qweight, scales, zeros, inv_s):
    _dev(X, torch.float16, "X")
    _dev(qweight, torch.int32, "qweight")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.int32, "zeros")
    if inv_s is not None:
        _dev(inv_s, torch.float32, "inv_s")
    M, K = X.shape
    N = qweight.shape[0]
    return M, N, K


def _layout(K, qweight, scales):
    """(w_bit, group) of a packed weight, from its shapes."""
    w_bit = 32 * qweight.shape[1] // K
    group = K // scales.shape[1]
    return w_bit, group


def gemv(X, qweight, scales, zeros, inv_s=None, out=None):
    M, N, K = _linear_args(X, qweight, scales, zeros, inv_s)
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    w_bit, group = _layout(K, qweight, scales)
    if (w_bit, group) == (4, 128):
        _check(lib.awq_gemv(_ptr(X), M, _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(inv_s), N,
                            K, _ptr(Y), _stream()))
    else:
        cfg = _cfg(w_bit, group)
        _check(lib.awq_gemv_ex(ctypes.byref(cfg), _ptr(X), M, _ptr(qweight), _ptr(scales),
                               _ptr(zeros), _ptr(inv_s), N, K, _ptr(Y), _stream()))
    return Y


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib.awq_gemm_workspace_size(M, N, K))


def gemm(X, qweight, scales, zeros, inv_s=None, out=None, workspace=None):
    M, N, K = _linear_args(X, qweight, scales, zeros, inv_s)
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    if inv_s is not None and workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=X.device)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    w_bit, group = _layout(K, qweight, scales)
    if (w_bit, group) == (4, 128):
        _check(lib.awq_gemm(_ptr(X), M, _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(inv_s), N,
                            K, _ptr(Y), _ptr(workspace), nbytes, _stream()))
    else:
        cfg = _cfg(w_bit, group)
        _check(lib.awq_gemm_ex(ctypes.byref(cfg), _ptr(X), M, _ptr(qweight), _ptr(scales),
                               _ptr(zeros), _ptr(inv_s), N, K, _ptr(Y), _ptr(workspace), nbytes,
                               _stream()))
    return Y


def gemv_silu_mul(X, qweight, scales, zeros, inv_s=None, out=None):
    """silu(gate) * up for a stacked [gate; up] weight of 2I rows: Y [M][I]."""
    M, N, K = _linear_args(X, qweight, scales, zeros, inv_s)
    Y = out if out is not None else torch.empty((M, N // 2), dtype=torch.float16, device=X.device)
    _check(lib.awq_gemv_silu_mul(_ptr(X), M, _ptr(qweight), _ptr(scales), _ptr(zeros),
                                 _ptr(inv_s), N // 2, K, _ptr(Y), _stream()))
    return Y


def gemm_silu_mul(X, qweight, scales, zeros, inv_s=None, out=None, workspace=None):
    """Tensor-core form of :func:`gemv_silu_mul`, any M."""
    M, N, K = _linear_args(X, qweight, scales, zeros, inv_s)
    Y = out if out is not None else torch.empty((M, N // 2), dtype=torch.float16, device=X.device)
    if inv_s is not None and workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=X.device)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.awq_gemm_silu_mul(_ptr(X), M, _ptr(qweight), _ptr(scales), _ptr(zeros),
                                 _ptr(inv_s), N // 2, K, _ptr(Y), _ptr(workspace), nbytes,
                                 _stream()))
    return Y


def fold_inv_scales(W: torch.Tensor, inv_s: torch.Tensor, out=None):
    """Row r of W (fp16, one row per input channel: a norm weight [K] or the
    previous linear's output rows [K][C]) times inv_s[r], rounded to fp16."""
    _dev(W, torch.float16, "W")
    _dev(inv_s, torch.float32, "inv_s")
    rows = W.shape[0]
    cols = W.numel() // rows if rows else 0
    Y = out if out is not None else torch.empty_like(W)
    _check(lib.awq_fold_inv_scales(_ptr(W), rows, cols, _ptr(inv_s), _ptr(Y), _stream()))
    return Y


def clip_search(X_cal: torch.Tensor, W: torch.Tensor, s_c=None, inv_s=None, n_clip: int = 20,
                w_bit: int = 4, group: int = 128, zero_point: bool = True, err: bool = False):
    """Per-group clipping ratio index (uint8 [N][K/group]) and, with err=True,
    every candidate's error (fp32 [N][G][n_clip])."""
    _dev(X_cal, torch.float16, "X_cal")
    _dev(W, torch.float16, "W")
    for t, nm in ((s_c, "s_c"), (inv_s, "inv_s")):
        if t is not None:
            _dev(t, torch.float32, nm)
    T, K = X_cal.shape
    N = W.shape[0]
    G = K // group
    cfg = _cfg(w_bit, group, zero_point)
    ws = torch.empty(lib.awq_clip_search_workspace_size(T, K, ctypes.byref(cfg)),
                     dtype=torch.uint8, device=W.device)
    idx = torch.empty((N, G), dtype=torch.uint8, device=W.device)
    e = torch.empty((N, G, n_clip), dtype=torch.float32, device=W.device) if err else None
    _check(lib.awq_clip_search(_ptr(X_cal), T, _ptr(W), N, K, _ptr(s_c), _ptr(inv_s),
                               ctypes.byref(cfg), n_clip, _ptr(ws), ws.numel(), _ptr(idx), _ptr(e),
                               _stream()))
    return (idx, e) if err else idx


def pack_clipped(W: torch.Tensor, s_c, clip_idx: torch.Tensor, n_clip: int = 20, w_bit: int = 4,
                 group: int = 128, zero_point: bool = True):
    _dev(W, torch.float16, "W")
    if s_c is not None:
        _dev(s_c, torch.float32, "s_c")
    _dev(clip_idx, torch.uint8, "clip_idx")
    N, K = W.shape
    c = 32 // w_bit
    G = K // group
    qweight = torch.empty((N, K // c), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, G), dtype=torch.float16, device=W.device)
    zeros = torch.empty((N, (G + c - 1) // c), dtype=torch.int32, device=W.device)
    cfg = _cfg(w_bit, group, zero_point)
    _check(lib.awq_pack_clipped(_ptr(W), _ptr(s_c), N, K, ctypes.byref(cfg), _ptr(clip_idx),
                                n_clip, _ptr(qweight), _ptr(scales), _ptr(zeros), _stream()))
    return qweight, scales, zeros


def search(X_cal: torch.Tensor, W: torch.Tensor, n_grid: int = 20, row_err: bool = False,
           w_bit: int = 4, group: int = 128, zero_point: bool = True):
    _dev(X_cal, torch.float16, "X_cal")
    _dev(W, torch.float16, "W")
    T, K = X_cal.shape
    N = W.shape[0]
    ws = torch.empty(lib.awq_search_workspace_size(T, N, K), dtype=torch.uint8, device=W.device)
    s_c = torch.empty(K, dtype=torch.float32, device=W.device)
    inv_s = torch.empty(K, dtype=torch.float32, device=W.device)
    rerr = torch.empty((n_grid, N), dtype=torch.float64, device=W.device) if row_err else None
    best = ctypes.c_int32(-1)
    mse = (ctypes.c_double * n_grid)()
    cfg = _cfg(w_bit, group, zero_point, n_grid)
    _check(lib.awq_search_scales(_ptr(X_cal), T, _ptr(W), N, K, ctypes.byref(cfg), _ptr(ws),
                                 ws.numel(), _ptr(s_c), _ptr(inv_s), ctypes.byref(best), mse,
                                 _ptr(rerr), _stream()))
    return {"best": best.value, "alpha": best.value / n_grid, "mse": list(mse), "s_c": s_c,
            "inv_s": inv_s, "row_err": rerr}


def measure_stream_read(buf: torch.Tensor, read_first: bool, out: torch.Tensor):
    """Measurement aid: one streaming read of ``buf`` (any contiguous CUDA
    tensor, size a multiple of 16 bytes) launched like :func:`gemv`; ``out``
    is an int32 CUDA tensor with one element per SM."""
    if not (buf.is_cuda and buf.is_contiguous() and out.is_cuda and out.dtype == torch.int32):
        raise ValueError("buf and out must be contiguous CUDA tensors, out int32")
    _check(lib.awq_measure_stream_read(_ptr(buf), buf.numel() * buf.element_size(),
                                       int(bool(read_first)), _ptr(out), _stream()))


def debug_stall(which: int, wait_limit_ns: int = 1_000_000_000):
    """Test hook: ``which`` 1 (awq_gemv), 2 (awq_gemm, M > 128) or 3 makes the
    next launches of those kernels lose one stage's copy, so that a bounded
    wait runs out after ``wait_limit_ns`` (see awq.h); ``debug_stall(0)``
    restores the defaults."""
    _check(lib.awq_debug_stall(int(which), int(wait_limit_ns)))
