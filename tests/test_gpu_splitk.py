"""Split-K launches of the tensor-core matmul (chosen when a layer has too few
128-row tiles to fill the GPU): per-element parity with the oracle, the same
result as the launch without split-K within the bound, and bitwise
determinism (the splits are added in a fixed order)."""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import assert_linear_close, dev, host  # noqa: E402


def _layer(seed, N, K, w_bit=4, group=128):
    rng = np.random.default_rng(seed)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.5, size=K)).astype(np.float32)
    qw, sc, zs = O.awq_pack(W16, s_c, group, w_bit, True)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32)
    return rng, qw, sc, zs, inv_s


def _split_bytes(M, N, K):
    return awq.gemm_workspace_bytes(M, N, K) - ((M * K * 2 + 255) // 256) * 256


@pytest.mark.parametrize("M,N,K", [(16, 256, 4096), (48, 640, 8192), (100, 384, 11008),
                                   (130, 1024, 4096), (9, 2048, 4096)])
def test_splitk_matches_oracle_and_is_deterministic(M, N, K):
    assert _split_bytes(M, N, K) > 0, "the plan is expected to split K for this shape"
    rng, qw, sc, zs, inv_s = _layer(M + N + K, N, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    args = (dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    y1 = host(awq.gemm(*args))
    y2 = host(awq.gemm(*args))
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))
    assert_linear_close(y1, X16, qw, sc, zs, inv_s)
    # without room for the partial sums the launch runs unsplit
    ws = torch.empty(((M * K * 2 + 255) // 256) * 256, dtype=torch.uint8, device="cuda")
    y0 = host(awq.gemm(*args, workspace=ws))
    assert_linear_close(y0, X16, qw, sc, zs, inv_s)


def test_splitk_unscaled_activations_with_workspace():
    # inv_s NULL: the workspace holds only the partial sums
    M, N, K = 32, 512, 8192
    rng, qw, sc, zs, _ = _layer(7, N, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    nbytes = _split_bytes(M, N, K)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = host(awq.gemm(dev(X16), dev(qw), dev(sc), dev(zs), None, workspace=ws))
    assert_linear_close(y, X16, qw, sc, zs, None)


@pytest.mark.parametrize("w_bit,group", [(8, 128), (4, 32)])
def test_splitk_variants(w_bit, group):
    M, N, K = 24, 384, 8192
    rng, qw, sc, zs, inv_s = _layer(11 + w_bit, N, K, w_bit, group)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = host(awq.gemm(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s)))
    y_ref, base = O.linear(X16, qw, sc, zs, inv_s, group, w_bit)
    err = np.abs(y.astype(np.float64) - y_ref)
    assert np.all(err <= O.tolerance(y_ref, base))


def _tiles(M, N):
    bn = 160 if M > 128 else max(16, 1 << (M - 1).bit_length())
    return -(-N // 128) * -(-M // bn)


@pytest.mark.parametrize("M,N,K", [(300, 9736, 4096), (2048, 3584, 4096), (2048, 3584, 11008)])
def test_ragged_round_split(M, N, K):
    """More tiles than SMs with a ragged last round: only that round's tiles
    are split over K.  (300, 9736): the split tiles are the ragged last token
    tile and include the ragged last row tile; the other two have 364 tiles
    of 160 tokens at 2048 tokens (2.5 rounds of 148 SMs).  Every output of
    the last token tile and a sample of the other tokens are checked;
    repeated calls are bitwise equal."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = _tiles(M, N)
    assert tiles > sms and tiles % sms != 0
    assert _split_bytes(M, N, K) > 0, "the plan is expected to split the last round"
    rng, qw, sc, zs, inv_s = _layer(M + N + K, N, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    args = (dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    y1 = host(awq.gemm(*args))
    y2 = host(awq.gemm(*args))
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))
    last = np.arange(((M - 1) // 160) * 160, M)
    sample = np.unique(np.concatenate([last, np.arange(0, M, 61)]))
    assert_linear_close(y1, X16, qw, sc, zs, inv_s, cols=sample)
