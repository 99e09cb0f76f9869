"""GPU parity of the quantization variants against the oracle: 4- and 8-bit
codes, groups of 128, 64 and 32 channels, zero point on and off.

Packing is compared bit for bit; the GEMV and the tensor-core GEMM per element
within |y_gpu - y_ref| <= 4e-3 sum_k |x~ w^| + 1 fp16 ulp (the matmuls are fed
the oracle's own packed weights); the search by its chosen alpha.
"""
import itertools

import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import dev, host, row_sq_error_bound  # noqa: E402

VARIANTS = [v for v in itertools.product((4, 8), (128, 64, 32), (True, False))]
IDS = [f"w{b}g{g}{'a' if z else 's'}" for b, g, z in VARIANTS]


def _layer(seed, N, K, with_sc=True):
    rng = np.random.default_rng(seed)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.5, size=K)).astype(np.float32) if with_sc else None
    return rng, W16, s_c


def _check(y_gpu, X16, qw, sc, zs, inv_s, group, w_bit):
    y_ref, base = O.linear(X16, qw, sc, zs, inv_s, group, w_bit)
    tol = O.tolerance(y_ref, base)
    y = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside the bound; worst ratio "
                           f"{float((err / tol).max()):.3f}")


@pytest.mark.parametrize("w_bit,group,zp", VARIANTS, ids=IDS)
@pytest.mark.parametrize("N,K", [(8, 128), (136, 384), (40, 1152), (24, 11008)])
def test_pack_variants_bit_exact(w_bit, group, zp, N, K):
    _, W16, s_c = _layer(N + K + w_bit + group, N, K)
    qw, sc, zs = O.awq_pack(W16, s_c, group, w_bit, zp)
    gq, gs, gz = awq.pack(dev(W16), dev(s_c), w_bit=w_bit, group=group, zero_point=zp)
    torch.cuda.synchronize()
    assert np.array_equal(host(gq), qw)
    assert np.array_equal(host(gs).view(np.uint16), sc.view(np.uint16))
    assert np.array_equal(host(gz), zs)


@pytest.mark.parametrize("w_bit,group,zp", VARIANTS, ids=IDS)
@pytest.mark.parametrize("N,K", [(256, 1152), (40, 384), (512, 11008)])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_gemv_variants_match_oracle(w_bit, group, zp, N, K, M):
    rng, W16, s_c = _layer(N * 3 + K + M, N, K)
    qw, sc, zs = O.awq_pack(W16, s_c, group, w_bit, zp)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = awq.gemv(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    _check(host(y), X16, qw, sc, zs, inv_s, group, w_bit)


@pytest.mark.parametrize("w_bit,group,zp", VARIANTS, ids=IDS)
@pytest.mark.parametrize("M", [1, 33, 300])
@pytest.mark.parametrize("scaled", [True, False])
def test_gemm_variants_match_oracle(w_bit, group, zp, M, scaled):
    # scaled: k-permuted activations written by the prescale pass; else the
    # caller's activations in natural order
    N, K = 200, 1152
    rng, W16, s_c = _layer(M * 7 + w_bit + group, N, K, with_sc=scaled)
    qw, sc, zs = O.awq_pack(W16, s_c, group, w_bit, zp)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32) if scaled else None
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = awq.gemm(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s) if scaled else None)
    _check(host(y), X16, qw, sc, zs, inv_s, group, w_bit)


@pytest.mark.parametrize("w_bit,group,zp", [(4, 64, True), (4, 32, False), (8, 128, True),
                                            (8, 32, False)])
def test_search_variants_match_oracle(w_bit, group, zp):
    rng = np.random.default_rng(w_bit + group)
    T, N, K = 256, 64, 512
    X = rng.standard_normal((T, K))
    X[:, rng.choice(K, 5, replace=False)] *= 20
    X16 = X.astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    cfg = dict(group=group, w_bit=w_bit, zero_point=zp)
    res = awq.search(dev(X16), dev(W16), row_err=True, w_bit=w_bit, group=group, zero_point=zp)
    ref = O.search(X16, W16, **cfg)
    best = int(res["best"])
    assert best == ref["best"] or ref["mse"][best] <= ref["mse"][ref["best"]] * (1 + O.MSE_REL)
    # each row's squared error, for every alpha, within the rigorous bound for
    # fp16 tensor-core operands (8-bit codes leave so little quantization error
    # that the fp16 rounding of x~ moves the mse by about 1%)
    rerr = host(res["row_err"])
    for i, al in enumerate(O.alpha_grid()):
        s_c, inv_s = O.channel_scales(ref["a"], al)
        bound = row_sq_error_bound(X16, W16, s_c, inv_s, np.arange(N), ref["row_err"][i], **cfg)
        assert np.all(np.abs(rerr[i] - ref["row_err"][i]) <= bound), i


@pytest.mark.parametrize("w_bit,group,zp", [(8, 128, True), (4, 32, False)])
def test_variants_full_size_sampled(w_bit, group, zp):
    # Llama-2-7B qkv 4096 -> 12288 at decode (GEMV, M = 1) and prefill
    # (GEMM, M = 2048) on sampled output channels and tokens
    K, N, lid = awq_inputs.layer("llama2-7b", "qkv")
    W16 = awq_inputs.weight(N, K, lid)
    Xc = awq_inputs.calib_tokens(256, K, lid)
    s_c, inv_s = O.channel_scales(O.absmean(Xc), 0.5)
    qw, sc, zs = awq.pack(dev(W16), dev(s_c), w_bit=w_bit, group=group, zero_point=zp)
    rows = np.unique(np.concatenate([np.arange(8), np.linspace(0, N - 1, 56).astype(np.int64)]))
    hq, hs, hz = host(qw)[rows], host(sc)[rows], host(zs)[rows]
    # the GPU quantizer agrees with the oracle on these rows
    oq, os_, oz = O.awq_pack(W16[rows], s_c, group, w_bit, zp)
    assert np.array_equal(hq, oq) and np.array_equal(hz, oz)
    X1 = awq_inputs.timed_tokens(1, K, lid)
    y1 = host(awq.gemv(dev(X1), qw, sc, zs, dev(inv_s)))
    _check(y1[:, rows], X1, hq, hs, hz, inv_s, group, w_bit)
    X2 = awq_inputs.timed_tokens(2048, K, lid)
    y2 = host(awq.gemm(dev(X2), qw, sc, zs, dev(inv_s)))
    tok = np.linspace(0, 2047, 24).astype(np.int64)
    _check(y2[np.ix_(tok, rows)], X2[tok], hq, hs, hz, inv_s, group, w_bit)
