"""GPU parity of the fused projections and the scale fold against the oracle.

* silu(gate) * up for a stacked [gate; up] weight: awq_gemv_silu_mul (M <= 8,
  CUDA cores) and awq_gemm_silu_mul (any M, tensor cores), per element
  within the oracle's propagated bound (``oracle.silu_mul_linear``), at sizes
  that span several tiles and a ragged tail, and at the Llama-2 gate/up shapes
  on sampled output columns;
* awq_fold_inv_scales bit for bit (one fp16 rounding of an fp32 product);
* one activation-aware search over stacked q/k/v projections.
"""
import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import dev, host  # noqa: E402


def _fused(seed, I, K, with_sc=True):
    rng = np.random.default_rng(seed)
    W16 = (rng.standard_normal((2 * I, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.5, size=K)).astype(np.float32) if with_sc else None
    qw, sc, zs = O.awq_pack(W16, s_c)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32) if with_sc else None
    return rng, qw, sc, zs, inv_s


def _check(y_gpu, X16, qw, sc, zs, inv_s):
    y_ref, tol = O.silu_mul_linear(X16, qw, sc, zs, inv_s)
    y = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside the bound; worst ratio "
                           f"{float((err / tol).max()):.3f}")


def _sub(qw, sc, zs, I, cols):
    """The stacked rows of the sampled output columns: gate rows, then up rows."""
    rows = np.concatenate([cols, I + cols])
    return qw[rows], sc[rows], zs[rows]


# ------------------------------------------------------- gemv (M <= 8)
@pytest.mark.parametrize("I,K", [(256, 512), (100, 384), (36, 1152), (1024, 11008)])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_gemv_silu_mul_matches_oracle(I, K, M):
    rng, qw, sc, zs, inv_s = _fused(I * 13 + K + M, I, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = awq.gemv_silu_mul(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))
    _check(host(y), X16, qw, sc, zs, inv_s)


def test_gemv_silu_mul_without_inv_s():
    rng, qw, sc, zs, _ = _fused(5, 200, 640, with_sc=False)
    X16 = rng.standard_normal((2, 640)).astype(np.float16)
    y = awq.gemv_silu_mul(dev(X16), dev(qw), dev(sc), dev(zs))
    _check(host(y), X16, qw, sc, zs, None)


# --------------------------------------------------- gemm (any M, tcgen05)
@pytest.mark.parametrize("I,K", [(256, 512), (100, 384), (36, 1152)])
@pytest.mark.parametrize("M", [1, 16, 100, 300])
@pytest.mark.parametrize("scaled", [True, False])
def test_gemm_silu_mul_matches_oracle(I, K, M, scaled):
    # scaled: the prescale pass writes k-permuted activations; otherwise the
    # caller's activations are read in natural order
    rng, qw, sc, zs, inv_s = _fused(I * 7 + K + M, I, K, with_sc=scaled)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = awq.gemm_silu_mul(dev(X16), dev(qw), dev(sc), dev(zs),
                          dev(inv_s) if scaled else None)
    _check(host(y), X16, qw, sc, zs, inv_s if scaled else None)


def test_gemm_and_gemv_silu_mul_agree_with_unfused_products():
    # the fused kernels equal silu of the gate layer times the up layer, each
    # computed by the plain kernels in fp32 (here compared through fp16)
    rng, qw, sc, zs, inv_s = _fused(11, 128, 1024)
    X16 = rng.standard_normal((4, 1024)).astype(np.float16)
    g = awq.gemm(dev(X16), dev(qw[:128]), dev(sc[:128]), dev(zs[:128]), dev(inv_s))
    u = awq.gemm(dev(X16), dev(qw[128:]), dev(sc[128:]), dev(zs[128:]), dev(inv_s))
    ref = torch.nn.functional.silu(g.float()) * u.float()
    for y in (awq.gemm_silu_mul(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s)),
              awq.gemv_silu_mul(dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s))):
        # both sides round g and u (or the product) to fp16 once
        assert torch.allclose(y.float(), ref, rtol=4e-3, atol=1e-3)


# ------------------------------------- Llama-2 gate/up shapes, sampled columns
@pytest.mark.parametrize("model", ["llama2-7b", "llama2-13b"])
def test_fused_gate_up_full_size_sampled(model):
    K, N, lid = awq_inputs.layer(model, "gate_up")
    I = N // 2
    W16 = awq_inputs.weight(N, K, lid)
    Xc = awq_inputs.calib_tokens(256, K, lid)
    s_c, inv_s = O.channel_scales(O.absmean(Xc), 0.5)
    qw, sc, zs = awq.pack(dev(W16), dev(s_c))
    g_inv = dev(inv_s)
    cols = np.unique(np.concatenate([np.arange(8), np.linspace(0, I - 1, 56).astype(np.int64),
                                     [I - 1]]))
    hq, hs, hz = host(qw), host(sc), host(zs)
    sq, ss, sz = _sub(hq, hs, hz, I, cols)
    # decode (M = 1, the launch shape the GEMV runs) and prefill (M = 2048)
    X1 = awq_inputs.timed_tokens(1, K, lid)
    y1 = host(awq.gemv_silu_mul(dev(X1), qw, sc, zs, g_inv))
    _check(y1[:, cols], X1, sq, ss, sz, inv_s)
    X2 = awq_inputs.timed_tokens(2048, K, lid)
    y2 = host(awq.gemm_silu_mul(dev(X2), qw, sc, zs, g_inv))
    tok = np.linspace(0, 2047, 24).astype(np.int64)
    _check(y2[np.ix_(tok, cols)], X2[tok], sq, ss, sz, inv_s)


# ------------------------------------------------------------ scale fold
@pytest.mark.parametrize("shape", [(4096,), (512, 1), (256, 96), (1000, 13), (11008, 4096)])
def test_fold_inv_scales_bit_exact(shape):
    rng = np.random.default_rng(sum(shape))
    W16 = rng.standard_normal(shape).astype(np.float16)
    inv_s = np.exp(rng.uniform(-2.0, 2.0, size=shape[0])).astype(np.float32)
    out = host(awq.fold_inv_scales(dev(W16), dev(inv_s)))
    assert np.array_equal(out.view(np.uint16), O.fold_inv_scales(W16, inv_s).view(np.uint16))


def test_fold_inv_scales_in_place_and_gemv_equivalence():
    # folding 1/s_c into the previous linear's output rows and calling the
    # layer with inv_s = NULL matches the runtime-scaled call up to fp16 roundings
    rng = np.random.default_rng(3)
    C, K, N = 256, 512, 64
    Wp = (rng.standard_normal((K, C)) * 0.05).astype(np.float16)
    x = rng.standard_normal((1, C)).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.0, size=K)).astype(np.float32)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32)
    t = dev(Wp)
    awq.fold_inv_scales(t, dev(inv_s), out=t)
    assert np.array_equal(host(t).view(np.uint16), O.fold_inv_scales(Wp, inv_s).view(np.uint16))
    y_prev = (x.astype(np.float64) @ Wp.astype(np.float64).T).astype(np.float16)
    y_fold = (x.astype(np.float64) @ host(t).astype(np.float64).T).astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    qw, sc, zs = O.awq_pack(W16, s_c)
    a = host(awq.gemv(dev(y_prev), dev(qw), dev(sc), dev(zs), dev(inv_s))).astype(np.float64)
    b = host(awq.gemv(dev(y_fold), dev(qw), dev(sc), dev(zs))).astype(np.float64)
    _, base = O.linear(y_prev, qw, sc, zs, inv_s)
    assert np.all(np.abs(a - b) <= 4 * 2.0 ** -11 * base + 2 * O.ulp_fp16(a))


# ---------------------------------------- one search over stacked q, k, v
def test_search_on_stacked_qkv_matches_oracle():
    rng = np.random.default_rng(21)
    T, K = 256, 512
    X = rng.standard_normal((T, K))
    X[:, rng.choice(K, 5, replace=False)] *= 20
    X16 = X.astype(np.float16)
    parts = [(rng.standard_normal((n, K)) * 0.02).astype(np.float16) for n in (64, 32, 32)]
    W16 = np.concatenate(parts, axis=0)
    res = awq.search(dev(X16), dev(W16), row_err=True)
    ref = O.search(X16, W16)
    # alpha: the oracle's, or one whose oracle mse is within 1e-4 of its best
    best = int(res["best"])
    assert best == ref["best"] or ref["mse"][best] <= ref["mse"][ref["best"]] * (1 + O.MSE_REL)
    # the stacked layer's per-row errors are the parts' rows, in order
    each = np.concatenate([O.search(X16, p)["row_err"] for p in parts], axis=1)
    assert np.allclose(ref["row_err"], each, rtol=1e-12, atol=0)
