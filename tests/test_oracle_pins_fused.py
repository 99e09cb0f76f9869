"""Pins of the oracle's fused-projection and scale-fold functions.

As for the other pins, each test checks the oracle against a closed form, a
special input that reduces it to a textbook operation, or a mathematical
identity, so that a slip (gate and up swapped, silu applied to the wrong
half, the fold applied along the wrong axis, a bound that does not hold)
fails at least one of them.
"""
import numpy as np

import oracle as O


def _rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------- silu
def test_silu_closed_forms():
    # sigma(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3; silu(0) = 0
    assert abs(O.silu(np.log(3.0)) - 0.75 * np.log(3.0)) <= 4e-16
    assert O.silu(0.0) == 0.0
    # sigma(x) + sigma(-x) = 1  =>  silu(x) - silu(-x) = x
    x = _rng().normal(scale=4.0, size=1000)
    assert np.max(np.abs(O.silu(x) - O.silu(-x) - x)) <= 1e-13
    # tails: silu(x) -> x for large x, -> 0 for very negative x
    assert abs(O.silu(40.0) - 40.0) <= 1e-14
    assert abs(O.silu(-40.0)) <= 1e-15


def test_silu_lipschitz_constant_is_tight():
    x = np.linspace(-20.0, 20.0, 400001)
    d = np.diff(O.silu(x)) / np.diff(x)
    assert np.max(np.abs(d)) <= O.SILU_LIP
    assert np.max(np.abs(d)) >= O.SILU_LIP - 1e-3


# ---------------------------------------------------------- fused gate / up
def _fused_layer(seed, I, K):
    rng = _rng(seed)
    W = (rng.normal(scale=0.02, size=(2 * I, K))).astype(np.float16)
    return W, O.awq_pack(W)


def test_silu_mul_one_hot_input_selects_gate_then_up():
    # one token equal to e_c: each projection returns column c of w^'
    I, K, c = 4, 256, 37
    W, (qw, sc, zs) = _fused_layer(1, I, K)
    X = np.zeros((1, K), dtype=np.float16)
    X[0, c] = 1.0
    wq = O.dequant(qw, sc, zs).astype(np.float64)
    Y, tol = O.silu_mul_linear(X, qw, sc, zs)
    assert Y.shape == (1, I)
    g, u = wq[:I, c], wq[I:, c]
    # silu of the gate half, times the up half
    assert np.array_equal(Y[0], g / (1.0 + np.exp(-g)) * u)
    # the halves are not interchangeable: the swapped product differs
    assert not np.allclose(Y[0], u / (1.0 + np.exp(-u)) * g)
    assert np.all(tol > 0)


def test_silu_mul_tolerance_covers_worst_case_perturbations():
    # the bound must hold for any g', u' within the projections' own bounds
    rng = _rng(2)
    I, K = 8, 512
    W, (qw, sc, zs) = _fused_layer(3, I, K)
    X = rng.normal(size=(3, K)).astype(np.float16)
    Y, tol = O.silu_mul_linear(X, qw, sc, zs)
    Y2, B2 = O.linear(X, qw, sc, zs)
    g, u = Y2[:, :I], Y2[:, I:]
    eg, eu = O.TOL_REL * B2[:, :I], O.TOL_REL * B2[:, I:]
    slack = tol - O.ulp_fp16(Y) - 1e-6 * np.abs(Y)
    for sg_ in (-1.0, -0.5, 0.0, 0.5, 1.0):
        for su in (-1.0, -0.3, 0.0, 0.7, 1.0):
            dev = np.abs(O.silu(g + sg_ * eg) * (u + su * eu) - Y)
            assert np.all(dev <= slack * (1 + 1e-12) + 1e-300)


def test_silu_mul_matches_two_separate_layers():
    # the fused weight is the stack [gate; up]: quantizing it whole gives the
    # same codes as quantizing the halves (quantization is per row)
    rng = _rng(4)
    I, K = 8, 256
    W, (qw, sc, zs) = _fused_layer(5, I, K)
    X = rng.normal(size=(2, K)).astype(np.float16)
    qg, sg, zg = O.awq_pack(W[:I])
    qu, su, zu = O.awq_pack(W[I:])
    assert np.array_equal(qw[:I], qg) and np.array_equal(qw[I:], qu)
    yg, _ = O.linear(X, qg, sg, zg)
    yu, _ = O.linear(X, qu, su, zu)
    Y, _ = O.silu_mul_linear(X, qw, sc, zs)
    assert np.array_equal(Y, O.silu(yg) * yu)


# -------------------------------------------------------------- scale fold
def test_fold_identity_and_power_of_two_scales_are_exact():
    rng = _rng(6)
    K, C = 64, 24
    W = rng.normal(size=(K, C)).astype(np.float16)
    assert np.array_equal(O.fold_inv_scales(W, np.ones(K, np.float32)), W)
    p2 = np.exp2(rng.integers(-3, 4, size=K)).astype(np.float32)
    out = O.fold_inv_scales(W, p2)
    assert np.array_equal(out.astype(np.float64), W.astype(np.float64) * p2[:, None])
    # a norm's weight vector is the C = 1 case, along the same axis
    g = rng.normal(size=K).astype(np.float16)
    assert np.array_equal(O.fold_inv_scales(g, p2).astype(np.float64),
                          g.astype(np.float64) * p2)


def test_fold_rounds_once_to_nearest_fp16():
    rng = _rng(7)
    K, C = 32, 16
    W = rng.normal(size=(K, C)).astype(np.float16)
    inv_s = (rng.uniform(0.3, 3.0, size=K)).astype(np.float32)
    out = O.fold_inv_scales(W, inv_s).astype(np.float64)
    exact = W.astype(np.float64) * inv_s.astype(np.float64)[:, None]
    # round to nearest: within half an fp16 ulp of the (fp32-rounded) product
    assert np.all(np.abs(out - exact) <= 0.5 * O.ulp_fp16(exact) * (1 + 1e-6) + 1e-30)


def test_fold_into_previous_linear_is_the_equivalent_transformation():
    # y = x W_prev^T feeds the quantized layer; folding inv_s into W_prev's
    # output rows gives y * inv_s, i.e. the activations x~ of the layer
    rng = _rng(8)
    T, C, K = 16, 48, 128
    x = rng.normal(size=(T, C)).astype(np.float16)
    Wp = (rng.normal(scale=0.1, size=(K, C))).astype(np.float16)
    inv_s = rng.uniform(0.5, 2.0, size=K).astype(np.float32)
    y = x.astype(np.float64) @ Wp.astype(np.float64).T
    y_fold = x.astype(np.float64) @ O.fold_inv_scales(Wp, inv_s).astype(np.float64).T
    scaled = y * inv_s.astype(np.float64)[None, :]
    base = np.abs(x.astype(np.float64)) @ np.abs(Wp.astype(np.float64) * inv_s[:, None]).T
    assert np.all(np.abs(y_fold - scaled) <= 2.0 ** -11 * base + 1e-12)


# ------------------------------------------- one search for q, k and v
def test_search_on_stacked_projections_is_the_row_weighted_mean():
    # mse(alpha) of [Wq; Wk; Wv] = sum of row errors / (T N): the row-count
    # weighted mean of the three layers' own mse curves
    rng = _rng(9)
    T, K = 48, 256
    X = rng.normal(size=(T, K))
    X[:, rng.choice(K, 3, replace=False)] *= 20
    X = X.astype(np.float16)
    parts = [(rng.normal(scale=0.02, size=(n, K))).astype(np.float16) for n in (16, 8, 8)]
    W = np.concatenate(parts, axis=0)
    whole = O.search(X, W, n_grid=6)
    each = [O.search(X, p, n_grid=6) for p in parts]
    n = np.array([p.shape[0] for p in parts], dtype=np.float64)
    mix = sum(e["mse"] * ni for e, ni in zip(each, n)) / n.sum()
    assert np.allclose(whole["mse"], mix, rtol=1e-12, atol=0)
    assert whole["best"] == int(np.argmin(mix))
