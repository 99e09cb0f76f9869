"""awq_absmean_noalloc: the activation statistics for callers that cannot
provide device memory (runtimes that plan every buffer ahead of execution,
real-time loops that must not allocate, plugins whose host owns all device
memory).  The partial sums live in a fixed 4 MiB array inside the library.

Checked through the C ABI against the regular entry point awq_absmean (which
takes a caller workspace), on two calls in a row with different inputs, with
the statistics tolerance used elsewhere (2e-6 relative); sizes beyond the
fixed array are rejected.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")

lib = awq.lib
lib.awq_absmean_noalloc.restype = ctypes.c_int
lib.awq_absmean_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_void_p, ctypes.c_void_p]


def _noalloc(X):
    T, K = X.shape
    a = torch.empty(K, dtype=torch.float32, device=X.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.awq_absmean_noalloc(ctypes.c_void_p(X.data_ptr()), T, K, ctypes.c_void_p(a.data_ptr()),
                                 stream)
    assert rc == 0, lib.awq_last_error_string().decode()
    return a


def _inputs(seed, T, K):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float32) * rng.uniform(0.1, 20.0, size=K).astype(np.float32)
    return torch.from_numpy(x.astype(np.float16)).cuda()


@pytest.mark.parametrize("T,K", [(4096, 4096), (257, 11008), (65536, 8192)])
def test_noalloc_matches_workspace_entry_point_twice(T, K):
    for call, seed in enumerate((T + K, T + K + 1)):
        X = _inputs(seed, T, K)
        ref = awq.absmean(X)                 # existing entry point, caller workspace
        got = _noalloc(X)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy().astype(np.float64), got.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - r) <= 2e-6 * np.abs(r)), f"call {call}"


def test_noalloc_rejects_too_large_and_bad_arguments():
    X = torch.zeros((2, 128), dtype=torch.float16, device="cuda")
    a = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big_k = 524288 + 128
    assert lib.awq_absmean_noalloc(ctypes.c_void_p(X.data_ptr()), 2, big_k,
                                   ctypes.c_void_p(a.data_ptr()), s) == 1
    assert "scratch limit" in lib.awq_last_error_string().decode()
    assert lib.awq_absmean_noalloc(None, 2, 128, ctypes.c_void_p(a.data_ptr()), s) == 2
    assert lib.awq_absmean_noalloc(ctypes.c_void_p(X.data_ptr()), 0, 128,
                                   ctypes.c_void_p(a.data_ptr()), s) == 1
