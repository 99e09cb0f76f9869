"""GPU parity: every kernel of the C ABI against the CPU oracle.

Packed codes, zero points and steps are compared bit for bit; the matmuls per
element against |y_gpu - y_ref| <= 4e-3 * sum_k |x~ w^| + 1 fp16 ulp(y_ref);
the statistics against a 2e-6 relative bound (fp32 runs of 16 tokens folded
into fp64); the search by its chosen alpha and its per-row errors.
Inputs are the seeded synthetic ones of ``awq_inputs`` (or constructed
closed-form cases); the matmul tests feed the oracle's own packed weights to
the GPU, so that they do not depend on the GPU quantizer.
"""
import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import assert_linear_close, dev, host, row_sq_error_bound  # noqa: E402


def _rand_layer(seed, N, K, outliers=True):
    rng = np.random.default_rng(seed)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.5, size=K)).astype(np.float32) if outliers else None
    return rng, W16, s_c


# ------------------------------------------------------------------ quantizer
@pytest.mark.parametrize("N,K", [(8, 128), (136, 384), (24, 11008), (512, 512), (40, 1152)])
@pytest.mark.parametrize("with_sc", [False, True])
def test_pack_bit_exact(N, K, with_sc):
    _, W16, s_c = _rand_layer(N * 7 + K, N, K)
    s_c = s_c if with_sc else None
    qw, sc, zs = O.awq_pack(W16, s_c)
    gq, gs, gz = awq.pack(dev(W16), dev(s_c) if s_c is not None else None)
    torch.cuda.synchronize()
    assert np.array_equal(host(gq), qw)
    assert np.array_equal(host(gs).view(np.uint16), sc.view(np.uint16))
    assert np.array_equal(host(gz), zs)


def test_pack_hand_derived_golden_row():
    import test_oracle_pins as P
    g = P._load_golden("hand_derived_groups.txt")
    k = np.arange(384)
    w = np.empty(384)
    w[:128] = ((k[:128] % 16) - 3) / 4.0
    i = np.arange(128)
    w[128:256] = np.where(i == 0, 0.0, np.where(i == 1, 15.0, 0.5 + ((i - 2) % 15))) / 4.0
    w[256:] = 1.0
    W16 = np.repeat(w.astype(np.float16)[None, :], 8, axis=0)
    gq, gs, gz = awq.pack(dev(W16))
    assert [int(v) for v in host(gq)[3]] == g["qweight"]
    assert [int(v) for v in host(gs).view(np.uint16)[5]] == g["scales"]
    assert [int(v) for v in host(gz)[7]] == g["zeros"]


def test_pack_degenerate_groups():
    W16 = np.zeros((8, 256), dtype=np.float16)
    W16[1] = -2.0
    W16[2, :64], W16[2, 64:128] = -65000.0, 65000.0
    W16[3, ::2] = np.float16(6e-8)          # fp16 subnormals
    s_c = np.full(256, 8.0, dtype=np.float32)
    for sc_arg in (None, s_c):
        qw, sc, zs = O.awq_pack(W16, sc_arg)
        gq, gs, gz = awq.pack(dev(W16), dev(sc_arg) if sc_arg is not None else None)
        assert np.array_equal(host(gq), qw)
        assert np.array_equal(host(gs).view(np.uint16), sc.view(np.uint16))
        assert np.array_equal(host(gz), zs)


# ---------------------------------------------------------------- statistics
@pytest.mark.parametrize("T,K", [(1, 128), (255, 512), (256, 512), (4097, 384), (20000, 128)])
def test_absmean(T, K):
    rng = np.random.default_rng(T + K)
    X16 = (rng.standard_normal((T, K)) * rng.uniform(0.1, 20, size=K)).astype(np.float16)
    a_ref = O.absmean(X16).astype(np.float64)
    a = host(awq.absmean(dev(X16))).astype(np.float64)
    assert np.all(np.abs(a - a_ref) <= 2e-6 * np.abs(a_ref) + 1e-30)


def test_channel_scales_all_grid_points():
    X16 = awq_inputs.calib_tokens(256, 512, 0)
    a = O.absmean(X16)
    a[:3] = [0.0, 1e-12, 3.5]   # the floor and an exact value
    ga = dev(a)
    for al in O.alpha_grid():
        s_ref, inv_ref = O.channel_scales(a, al)
        s, inv = awq.channel_scales(ga, al)
        s, inv = host(s), host(inv)
        ulp = np.abs(s.view(np.int32).astype(np.int64) - s_ref.view(np.int32).astype(np.int64))
        assert ulp.max() <= 1
        assert np.array_equal(inv, (np.float32(1) / s).astype(np.float32))


# ------------------------------------------------------------------- matmuls
def _packed(seed, N, K):
    rng, W16, s_c = _rand_layer(seed, N, K)
    qw, sc, zs = O.awq_pack(W16, s_c)
    inv_s = (np.float32(1) / s_c).astype(np.float32)
    return rng, qw, sc, zs, inv_s


def _x(rng, M, K):
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, rng.choice(K, size=max(1, K // 100), replace=False)] *= 20
    return x.astype(np.float16)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("N,K", [(512, 512), (8, 128), (24, 1152), (136, 2048), (40, 11008)])
def test_gemv_parity(M, N, K):
    rng, qw, sc, zs, inv_s = _packed(M * 1000 + N + K, N, K)
    X16 = _x(rng, M, K)
    y = awq.gemv(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    assert_linear_close(host(y), X16, qw, sc, zs, inv_s)
    y0 = awq.gemv(dev(X16), dev(qw), dev(sc), dev(zs), None)
    assert_linear_close(host(y0), X16, qw, sc, zs, None)


@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64, 100, 128, 129, 160, 161, 192, 193, 256, 300, 320, 384, 513])
@pytest.mark.parametrize("N,K", [(512, 512), (136, 384), (8, 128), (264, 1152)])
def test_gemm_parity(M, N, K):
    rng, qw, sc, zs, inv_s = _packed(M * 7 + N * 3 + K, N, K)
    X16 = _x(rng, M, K)
    y = awq.gemm(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    awq.check_device_error()
    assert_linear_close(host(y), X16, qw, sc, zs, inv_s)


def test_gemm_without_channel_scales():
    rng, qw, sc, zs, _ = _packed(5, 256, 640)
    X16 = _x(rng, 40, 640)
    y = awq.gemm(dev(X16), dev(qw), dev(sc), dev(zs), None)
    awq.check_device_error()
    assert_linear_close(host(y), X16, qw, sc, zs, None)


@pytest.mark.parametrize("fn", ["gemv", "gemm"])
def test_closed_form_row_sums_and_single_code(fn):
    """s = 1, q = z + 1 -> Y = row sums of X; one extra code at (n0, k0) on top
    of q = z -> column n0 is X[:, k0] * inv_s[k0], all others zero."""
    rng = np.random.default_rng(11)
    M, N, K = (4 if fn == "gemv" else 20), 136, 512
    z = rng.integers(0, 15, size=(N, K // 128)).astype(np.uint8)
    s16 = np.ones((N, K // 128), dtype=np.float16)
    X16 = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
    f = getattr(awq, fn)
    q = (np.repeat(z, 128, axis=1) + 1).astype(np.uint8)
    y = host(f(dev(X16), dev(O.pack_codes(q)), dev(s16), dev(O.pack_zeros(z)), None))
    assert np.array_equal(y.astype(np.float64), np.repeat(X16.astype(np.float64).sum(1, keepdims=True), N, 1))
    q = np.repeat(z, 128, axis=1).astype(np.uint8)
    n0, k0 = 77, 300
    q[n0, k0] += 1
    inv_s = np.exp2(rng.integers(-2, 3, size=K)).astype(np.float32)
    y = host(f(dev(X16), dev(O.pack_codes(q)), dev(s16), dev(O.pack_zeros(z)), dev(inv_s))).astype(np.float64)
    assert np.array_equal(y[:, n0], X16[:, k0].astype(np.float64) * inv_s[k0])
    y[:, n0] = 0
    assert np.all(y == 0)


# -------------------------------------------------------------------- search
def test_search_toy_matches_oracle():
    """Toy layer (K = N = 512, T = 256 calibration tokens with 1% outlier
    channels).  The chosen alpha equals the oracle's, or the oracle's MSE at
    the GPU's alpha is within 1e-4 of the best.  Each row's squared error for
    every alpha lies within the rigorous fp16-operand bound of
    ``row_sq_error_bound`` of the oracle's, and each alpha's MSE within 1e-3:
    the tensor cores see x~ and w^ rounded to fp16, and when a few outlier
    channels carry most of the output that moves the squared error by ~1e-4
    of the MSE (observed up to 1.5e-4 on this layer)."""
    K, N, lid = awq_inputs.layer("toy", "linear")
    X16 = awq_inputs.calib_tokens(256, K, lid)
    W16 = awq_inputs.weight(N, K, lid)
    ref = O.search(X16, W16)
    res = awq.search(dev(X16), dev(W16), row_err=True)
    mse_gpu = np.array(res["mse"])
    b = res["best"]
    assert b == ref["best"] or ref["mse"][b] <= ref["mse"][ref["best"]] * (1 + O.MSE_REL)
    assert np.allclose(mse_gpu, ref["mse"], rtol=1e-3, atol=0)
    assert mse_gpu[b] < mse_gpu[0]
    rerr = host(res["row_err"])
    rows = np.arange(N)
    for i, al in enumerate(O.alpha_grid()):
        s_c, inv_s = O.channel_scales(ref["a"], al)
        bound = row_sq_error_bound(X16, W16, s_c, inv_s, rows, ref["row_err"][i])
        assert np.all(np.abs(rerr[i] - ref["row_err"][i]) <= bound), i
