"""GPU parity of the narrow-token tensor-core matmul (M <= 128 tokens, plain
fp16 output, 4- or 8-bit codes in 128- or 64-channel groups).

Its weights enter the MMA as the exact integers q - z and every group's
partial product is scaled by s in fp32, so it rounds differently from the
wide-tile kernel; the bound is the same per-element one against the oracle:
|y_gpu - y_ref| <= 4e-3 sum_k |x~ w^| + 1 fp16 ulp.  Cases cover every token
tile (16, 32, 64, 128 and ragged M), both activation layouts (prescaled and
k-permuted, or the caller's in natural order), ragged N, long K (many
zero-point words per row), split-K against the unsplit launch, several work
items per CTA, and the Llama-2-7B batched-decode shapes on sampled outputs.
For M <= 8 of the default format awq_gemm runs the decode matmul instead
whenever that needs no K split, so those cases check whichever kernel the
library selects (the other formats, and the 7B down shape at M = 8, stay on
the narrow kernel).
"""
import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import dev, host  # noqa: E402

FORMATS = [(4, 128, True), (4, 64, True), (8, 128, True), (8, 64, False), (4, 128, False)]
FIDS = [f"w{b}g{g}{'a' if z else 's'}" for b, g, z in FORMATS]


def _layer(seed, N, K, w_bit=4, group=128, zp=True, with_sc=True):
    rng = np.random.default_rng(seed)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.0, 1.5, size=K)).astype(np.float32) if with_sc else None
    qw, sc, zs = O.awq_pack(W16, s_c, group, w_bit, zp)
    inv_s = (1.0 / s_c.astype(np.float64)).astype(np.float32) if with_sc else None
    return rng, qw, sc, zs, inv_s


def _check(y, X16, qw, sc, zs, inv_s, group=128, w_bit=4):
    y_ref, base = O.linear(X16, qw, sc, zs, inv_s, group, w_bit)
    tol = O.tolerance(y_ref, base)
    yy = y.astype(np.float64)
    assert np.all(np.isfinite(yy)), "non-finite output"
    err = np.abs(yy - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside the bound; worst ratio "
                           f"{float((err / tol).max()):.3f}")


def _gemm(X16, qw, sc, zs, inv_s, w_bit, group, zp, workspace=None):
    args = (dev(X16), dev(qw), dev(sc), dev(zs), dev(inv_s) if inv_s is not None else None)
    return host(awq.gemm(*args, workspace=workspace)) if workspace is not None else \
        host(awq.gemm(*args))


@pytest.mark.parametrize("w_bit,group,zp", FORMATS, ids=FIDS)
@pytest.mark.parametrize("M", [1, 8, 16, 17, 32, 48, 64, 65, 100, 128])
@pytest.mark.parametrize("scaled", [True, False])
def test_narrow_matches_oracle(w_bit, group, zp, M, scaled):
    # N = 3 full 128-row tiles + 8 rows; K = 12 groups of 128 (24 of 64)
    N, K = 392, 1536
    rng, qw, sc, zs, inv_s = _layer(M * 31 + w_bit + group, N, K, w_bit, group, zp, scaled)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = _gemm(X16, qw, sc, zs, inv_s, w_bit, group, zp)
    _check(y, X16, qw, sc, zs, inv_s, group, w_bit)


@pytest.mark.parametrize("w_bit,group", [(4, 128), (4, 64), (8, 128)])
def test_narrow_long_k_and_outliers(w_bit, group):
    # K = 11008 (86 groups of 128: eleven zero-point words per row), activations
    # with 1% of the channels x20
    M, N, K = 24, 256, 11008
    rng, qw, sc, zs, inv_s = _layer(5 + w_bit + group, N, K, w_bit, group)
    X = rng.standard_normal((M, K))
    X[:, rng.choice(K, K // 100, replace=False)] *= 20
    X16 = X.astype(np.float16)
    _check(_gemm(X16, qw, sc, zs, inv_s, w_bit, group, True), X16, qw, sc, zs, inv_s, group,
           w_bit)


@pytest.mark.parametrize("M,N,K", [(16, 256, 4096), (40, 512, 8192), (8, 384, 11008),
                                   (120, 256, 4096)])
def test_narrow_splitk_matches_unsplit(M, N, K):
    # these shapes have few tiles, so the plan splits K when the workspace
    # holds the partial sums; without it the launch runs unsplit
    rng, qw, sc, zs, inv_s = _layer(M + N + K, N, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y1 = _gemm(X16, qw, sc, zs, inv_s, 4, 128, True)
    y2 = _gemm(X16, qw, sc, zs, inv_s, 4, 128, True)
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16)), "not deterministic"
    _check(y1, X16, qw, sc, zs, inv_s)
    ws = torch.empty(((M * K * 2 + 255) // 256) * 256, dtype=torch.uint8, device="cuda")
    y0 = _gemm(X16, qw, sc, zs, inv_s, 4, 128, True, workspace=ws)
    _check(y0, X16, qw, sc, zs, inv_s)


def test_narrow_many_items_per_cta():
    # 320 row tiles x 2 token tiles = 640 work items on 148 CTAs: every CTA
    # walks several items, crossing item boundaries in the code ring, the
    # dequantization teams and the accumulator ring
    M, N, K = 40, 40960, 1024
    rng, qw, sc, zs, inv_s = _layer(77, N, K)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    y = _gemm(X16, qw, sc, zs, inv_s, 4, 128, True)
    rows = np.unique(np.concatenate([np.arange(130), np.linspace(0, N - 1, 300).astype(np.int64),
                                     np.arange(N - 130, N)]))
    _check(y[:, rows], X16, qw[rows], sc[rows], zs[rows], inv_s)


@pytest.mark.parametrize("layer", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("M", [8, 32, 128])
def test_narrow_7b_batched_sampled(layer, M):
    # Llama-2-7B layer shapes at batched decode, on sampled output channels
    K, N, lid = awq_inputs.layer("llama2-7b", layer)
    W16 = awq_inputs.weight(N, K, lid)
    Xc = awq_inputs.calib_tokens(256, K, lid)
    s_c, inv_s = O.channel_scales(O.absmean(Xc), 0.5)
    qw, sc, zs = awq.pack(dev(W16), dev(s_c))
    X = awq_inputs.timed_tokens(M, K, lid)
    y = host(awq.gemm(dev(X), qw, sc, zs, dev(inv_s)))
    rows = np.unique(np.concatenate([np.arange(8), np.linspace(0, N - 1, 120).astype(np.int64)]))
    _check(y[:, rows], X, host(qw)[rows], host(sc)[rows], host(zs)[rows], inv_s)
