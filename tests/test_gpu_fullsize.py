"""GPU parity at the full layer sizes of the Llama-2 configurations.

The kernels run on whole layers, in the launch configuration the benchmark
uses; the oracle checks sampled output rows one by one:

* pack: the sampled rows' codes, steps and zero points bit for bit;
* GEMV / GEMM: the sampled rows of Y within 4e-3 * sum|x~ w^| + 1 fp16 ulp,
  the oracle computing them from the GPU's own packed rows;
* search: per-row squared errors of sampled rows for every alpha, with the
  oracle given the GPU's activation statistics (themselves checked to 2e-6),
  so that both sides quantize with the same s_c; the subset sums within 1e-4.
"""
import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import assert_linear_close, dev, host, row_sq_error_bound  # noqa: E402

_CACHE = {}


def _layer(model, name, T_cal=256):
    key = (model, name, T_cal)
    if key not in _CACHE:
        _CACHE.clear()
        K, N, lid = awq_inputs.layer(model, name)
        W = awq_inputs.weight(N, K, lid)
        Xc = awq_inputs.calib_tokens(T_cal, K, lid)
        _CACHE[key] = (K, N, lid, W, Xc)
    return _CACHE[key]


def _rows(N, n=48, seed=0):
    rng = np.random.default_rng(seed + N)
    r = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=n, replace=False)]))
    return r


def _pack_and_check(W, Xc, rows):
    """GPU statistics, scales (alpha = 0.5) and pack of the whole layer; the
    sampled rows are checked bit for bit against the oracle."""
    a = awq.absmean(dev(Xc))
    a_ref = O.absmean(Xc).astype(np.float64)
    assert np.all(np.abs(host(a).astype(np.float64) - a_ref) <= 2e-6 * a_ref)
    s_c, inv_s = awq.channel_scales(a, 0.5)
    gW = dev(W)
    qw, sc, zs = awq.pack(gW, s_c)
    del gW
    s_c_h, inv_h = host(s_c), host(inv_s)
    rq, rs, rz = O.awq_pack(W[rows], s_c_h)
    hq, hs, hz = host(qw[rows]), host(sc[rows]), host(zs[rows])
    assert np.array_equal(hq, rq)
    assert np.array_equal(hs.view(np.uint16), rs.view(np.uint16))
    assert np.array_equal(hz, rz)
    return qw, sc, zs, inv_s, (rq, rs, rz, inv_h)


DECODE = [("llama2-7b", "qkv"), ("llama2-7b", "o"), ("llama2-7b", "gate_up"),
          ("llama2-7b", "down"), ("llama2-70b", "qkv"), ("llama2-70b", "o"),
          ("llama2-70b", "gate_up"), ("llama2-70b", "down")]


@pytest.mark.parametrize("model,name", DECODE)
def test_decode_gemv_full_layer(model, name):
    K, N, lid, W, Xc = _layer(model, name)
    rows = _rows(N)
    qw, sc, zs, inv_s, (rq, rs, rz, inv_h) = _pack_and_check(W, Xc, rows)
    for M in (1, 4, 8) if model == "llama2-7b" else (1,):
        X = awq_inputs.timed_tokens(M, K, lid)
        y = host(awq.gemv(dev(X), qw, sc, zs, inv_s))
        assert np.all(np.isfinite(y))
        assert_linear_close(y[:, rows], X, rq, rs, rz, inv_h)


BATCHED = [("llama2-7b", n, M) for n in ("qkv", "o", "gate_up", "down") for M in (8, 32, 128)] + \
    [("llama2-7b", "gate_up", 2048), ("llama2-13b", "qkv", 2048), ("llama2-13b", "gate_up", 4096),
     ("llama2-13b", "down", 4096), ("llama2-70b", "qkv", 4096), ("llama2-70b", "down", 512),
     ("llama2-70b", "gate_up", 1024)]


@pytest.mark.parametrize("model,name,M", BATCHED)
def test_gemm_full_layer(model, name, M):
    K, N, lid, W, Xc = _layer(model, name)
    rows = _rows(N, n=24)
    qw, sc, zs, inv_s, (rq, rs, rz, inv_h) = _pack_and_check(W, Xc, rows)
    X = awq_inputs.timed_tokens(M, K, lid)
    y = host(awq.gemm(dev(X), qw, sc, zs, inv_s))
    awq.check_device_error()
    assert np.all(np.isfinite(y))
    tok = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(M).choice(M, size=min(M, 64), replace=False)]))
    assert_linear_close(y[:, rows], X, rq, rs, rz, inv_h, cols=tok)


def _search_case(model, name, T, nrows):
    K, N, lid = awq_inputs.layer(model, name)
    W = awq_inputs.weight(N, K, lid)
    X = awq_inputs.calib_tokens(T, K, lid)
    gX = dev(X)
    res = awq.search(gX, dev(W), row_err=True)
    a = host(awq.absmean(gX))
    a_ref = O.absmean(X).astype(np.float64)
    assert np.all(np.abs(a.astype(np.float64) - a_ref) <= 2e-6 * a_ref)
    rows = _rows(N, n=nrows, seed=7)
    ref = O.search(X, W, rows=rows, a=a)
    g = host(res["row_err"])[:, rows]
    return X, W, a, rows, res, ref, g


def _check_search(X, W, a, rows, res, ref, g):
    """The GPU's own MSE picks its alpha; the sampled rows' squared errors lie
    within the rigorous fp16-operand bound of the oracle's (both sides use the
    same statistics, hence the same s_c), and their sums within 1e-3."""
    mse = np.array(res["mse"])
    assert np.argmin(mse) == res["best"]
    assert np.all(np.isfinite(mse)) and mse[res["best"]] < mse[0]
    for i, al in enumerate(O.alpha_grid()):
        s_c, inv_s = O.channel_scales(a, al)
        bound = row_sq_error_bound(X, W, s_c, inv_s, rows, ref["row_err"][i])
        assert np.all(np.abs(g[i] - ref["row_err"][i]) <= bound), i
    assert np.allclose(g.sum(axis=1), ref["row_err"].sum(axis=1), rtol=1e-3, atol=0)


def test_search_7b_o_4096_tokens():
    """7B o-projection, 4096 calibration tokens (the batched configuration's
    scale search)."""
    _check_search(*_search_case("llama2-7b", "o", 4096, 40))


def test_search_70b_gate_up_65536_tokens():
    """70B gate_up (8192 -> 57344), 128 x 512 = 65536 calibration tokens; the
    oracle scores 10 sampled rows for all 20 alphas."""
    _check_search(*_search_case("llama2-70b", "gate_up", 65536, 8))
