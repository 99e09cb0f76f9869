"""GPU parity of the weight-clipping search and the clipped pack.

* awq_pack_clipped: codes, steps and zero points bit for bit against the
  oracle's quantize_clipped, for every variant and random ratio indices;
* awq_clip_search: every candidate's error within fp32-summation distance of
  the oracle's fp64 error, and the chosen ratio the oracle's or one whose
  oracle error is within 1e-4 of the best (the rule the scale search uses);
* at the Llama-2-7B qkv shape with 4096 calibration tokens, on sampled rows.
"""
import itertools

import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import dev, host  # noqa: E402

VARIANTS = list(itertools.product((4, 8), (128, 64, 32), (True, False)))
IDS = [f"w{b}g{g}{'a' if z else 's'}" for b, g, z in VARIANTS]


@pytest.mark.parametrize("w_bit,group,zp", VARIANTS, ids=IDS)
def test_pack_clipped_bit_exact(w_bit, group, zp):
    rng = np.random.default_rng(w_bit * 7 + group)
    N, K, n_clip = 40, 1152, 20
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1, 1.5, size=K)).astype(np.float32)
    idx = rng.integers(0, n_clip, size=(N, K // group)).astype(np.uint8)
    q, z, s16 = O.quantize_clipped(W16, s_c, idx, n_clip, group, w_bit, zp)
    gq, gs, gz = awq.pack_clipped(dev(W16), dev(s_c), dev(idx), n_clip, w_bit, group, zp)
    assert np.array_equal(host(gq), O.pack_codes(q, w_bit))
    assert np.array_equal(host(gs).view(np.uint16), s16.view(np.uint16))
    assert np.array_equal(host(gz), O.pack_zeros(z, w_bit))


def _check_search(idx_gpu, err_gpu, idx_ref, err_ref):
    # the candidates' errors: fp32 Gram and quadratic form vs fp64
    scale = err_ref.max(axis=2, keepdims=True)
    assert np.all(np.abs(err_gpu - err_ref) <= 1e-4 * err_ref + 1e-6 * scale)
    # the choice: the oracle's, or within 1e-4 of the oracle's best
    N, G = idx_ref.shape
    e_at_gpu = np.take_along_axis(err_ref, idx_gpu[:, :, None].astype(np.int64), axis=2)[:, :, 0]
    e_best = np.take_along_axis(err_ref, idx_ref[:, :, None].astype(np.int64), axis=2)[:, :, 0]
    assert np.all((idx_gpu == idx_ref) | (e_at_gpu <= e_best * (1 + 1e-4)))


@pytest.mark.parametrize("w_bit,group,zp", [(4, 128, True), (4, 64, False), (4, 32, True),
                                            (8, 128, True), (8, 32, False)])
def test_clip_search_matches_oracle(w_bit, group, zp):
    rng = np.random.default_rng(3 + w_bit + group)
    T, N, K = 256, 64, 512
    X = rng.standard_normal((T, K))
    X[:, rng.choice(K, 5, replace=False)] *= 20
    X16 = X.astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c, inv_s = O.channel_scales(O.absmean(X16), 0.5)
    idx_ref, err_ref = O.clip_search(X16, W16, s_c, inv_s, 20, group, w_bit, zp)
    idx, err = awq.clip_search(dev(X16), dev(W16), dev(s_c), dev(inv_s), 20, w_bit, group, zp,
                               err=True)
    _check_search(host(idx), host(err).astype(np.float64), idx_ref, err_ref)


def test_clip_search_full_size_sampled():
    K, N, lid = awq_inputs.layer("llama2-7b", "qkv")
    W16 = awq_inputs.weight(N, K, lid)
    X16 = awq_inputs.calib_tokens(4096, K, lid)
    s_c, inv_s = O.channel_scales(O.absmean(X16), 0.5)
    idx, err = awq.clip_search(dev(X16), dev(W16), dev(s_c), dev(inv_s), 20, err=True)
    rows = np.linspace(0, N - 1, 12).astype(np.int64)
    idx_ref, err_ref = O.clip_search(X16, W16[rows], s_c, inv_s, 20)
    _check_search(host(idx)[rows], host(err)[rows].astype(np.float64), idx_ref, err_ref)
    # clipping never raises a group's error above no clipping
    e = host(err).astype(np.float64)
    chosen = np.take_along_axis(e, host(idx)[:, :, None].astype(np.int64), axis=2)[:, :, 0]
    assert np.all(chosen <= e[:, :, 0])


def test_clipping_lowers_the_layer_error_on_calibration_tokens():
    # the quantized layer's squared error on the calibration tokens drops with
    # the chosen clipping (per-group optima; the cross-group terms are small)
    rng = np.random.default_rng(8)
    T, N, K = 512, 128, 1024
    X = rng.standard_normal((T, K))
    X[:, rng.choice(K, 10, replace=False)] *= 20
    X16 = X.astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    W16[:, ::97] *= 8                                           # a few weight outliers
    s_c, inv_s = O.channel_scales(O.absmean(X16), 0.5)
    idx = awq.clip_search(dev(X16), dev(W16), dev(s_c), dev(inv_s), 20)
    plain = awq.pack(dev(W16), dev(s_c))
    clipped = awq.pack_clipped(dev(W16), dev(s_c), idx, 20)
    y = X16.astype(np.float64) @ W16.astype(np.float64).T
    errs = []
    for qw, sc, zs in (plain, clipped):
        yq, _ = O.linear(X16, host(qw), host(sc), host(zs), inv_s)
        errs.append(((yq - y) ** 2).sum())
    assert errs[1] < errs[0]
