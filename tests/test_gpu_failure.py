"""Failure detection of the matmuls' bounded waits, without a GPU fault.

A test hook makes one CTA of awq_gemv (decode matmul) or awq_gemm (wide
tensor-core matmul) withhold the copy of one stage, so that the wait for it
cannot complete; with the limit lowered to 20 ms the wait runs out, the
kernel records it in the device's error word, stops its other roles, lets
its copies and MMAs in flight finish (bounded), frees its tensor memory and
returns.  The host learns of it through awq_check_device_error
(AWQ_ERR_DEVICE), the context stays usable, and the next call is correct.
Nothing here faults, traps or hangs the GPU: the only "failure" is a wait on
a copy that was never requested.
"""
import time

import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import assert_linear_close, dev, host  # noqa: E402


def test_gemv_wait_runs_out_is_reported_and_the_next_call_is_correct():
    N, K = 1096, 2304
    rng = np.random.default_rng(11)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    qw, sc, zs = O.awq_pack(W16, None)
    X = awq_inputs.timed_tokens(1, K, 77)
    gX, gq, gs, gz = dev(X), dev(qw), dev(sc), dev(zs)
    awq.check_device_error()                     # nothing pending
    awq.debug_stall(1, 20_000_000)               # 20 ms limit, one stage withheld
    try:
        t0 = time.monotonic()
        awq.gemv(gX, gq, gs, gz, None)
        with pytest.raises(awq.AwqError) as err:
            awq.check_device_error()
        assert err.value.code == 7               # AWQ_ERR_DEVICE
        assert time.monotonic() - t0 < 10.0      # the call returned; nothing hung
    finally:
        awq.debug_stall(0)
    y = host(awq.gemv(gX, gq, gs, gz, None))
    awq.check_device_error()                     # the error word was cleared
    assert_linear_close(y, X, qw, sc, zs, None)


def test_gemm_wait_runs_out_is_reported_tensor_memory_freed_and_next_call_correct():
    M, N, K = 256, 264, 1152      # M > 128: the wide persistent tcgen05 kernel
    rng = np.random.default_rng(12)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    qw, sc, zs = O.awq_pack(W16, None)
    X = awq_inputs.timed_tokens(M, K, 78)
    gX, gq, gs, gz = dev(X), dev(qw), dev(sc), dev(zs)
    awq.check_device_error()
    awq.debug_stall(2, 20_000_000)
    try:
        t0 = time.monotonic()
        awq.gemm(gX, gq, gs, gz, None)
        with pytest.raises(awq.AwqError) as err:
            awq.check_device_error()
        assert err.value.code == 7
        assert time.monotonic() - t0 < 10.0
    finally:
        awq.debug_stall(0)
    # tensor memory was released: new launches allocate it and finish
    for _ in range(3):
        y = host(awq.gemm(gX, gq, gs, gz, None))
    awq.check_device_error()
    assert_linear_close(y, X, qw, sc, zs, None)
