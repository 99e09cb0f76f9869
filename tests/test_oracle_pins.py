"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an invariant stated by the
pages, a brute-force search on a tiny input or a hand-derived fixture, chosen
so that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, s_c applied on the wrong side) fails at least one of them.
"""
import os

import numpy as np
import pytest

import awq_inputs
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers
def _grid_weights(rng, N, K, s_exp_lo=-8, s_exp_hi=-3):
    """Weights that lie exactly on a quantization grid: per group a power-of-two
    step s, a zero point z, and codes q that hit both 0 and 15."""
    G = K // O.GROUP
    q = rng.integers(0, 16, size=(N, G, O.GROUP))
    q[:, :, 0] = 0
    q[:, :, 1] = 15
    z = rng.integers(0, 16, size=(N, G))
    s = np.exp2(rng.integers(s_exp_lo, s_exp_hi + 1, size=(N, G))).astype(np.float64)
    w = (q - z[:, :, None]) * s[:, :, None]
    return w.reshape(N, K), q.reshape(N, K), z, s


def _load_golden(name):
    d = {"qweight": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key in ("N", "K"):
                d[key] = int(vals[0])
            elif key == "qweight":
                d["qweight"] += [int(v, 16) for v in vals]
            else:
                d[key] = [int(v, 16) for v in vals]
    return d


# ------------------------------------------------------ quantize / dequant
def test_dequant_exact_on_grid_points():
    """Weights on a grid with power-of-two steps come back bit-for-bit, with
    the same codes and zero points (the grid is the quantizer's fixed point)."""
    rng = np.random.default_rng(0)
    w, q, z, s = _grid_weights(rng, 64, 512)
    W16 = w.astype(np.float16)
    assert np.array_equal(W16.astype(np.float64), w)
    qq, zz, ss = O.quantize(W16)
    assert np.array_equal(qq, q)
    assert np.array_equal(zz, z)
    assert np.array_equal(ss.astype(np.float64), s)
    qw, sc, zs = O.awq_pack(W16)
    assert np.array_equal(O.dequant(qw, sc, zs).astype(np.float64), w)


def test_scaled_grid_and_equivalent_transformation_exact():
    """With power-of-two channel scales, W = grid / s_c: the quantizer must
    multiply W by s_c before rounding (grid points again), and the layer with
    1/s_c on the activations must equal the unquantized X W^T exactly."""
    rng = np.random.default_rng(1)
    N, K, M = 32, 256, 5
    w_grid, q, z, s = _grid_weights(rng, N, K, -6, -4)
    s_c = np.exp2(rng.integers(-2, 3, size=K)).astype(np.float32)
    W = w_grid / s_c[None, :].astype(np.float64)
    W16 = W.astype(np.float16)
    assert np.array_equal(W16.astype(np.float64), W)
    qq, zz, ss = O.quantize(W16, s_c)
    assert np.array_equal(qq, q) and np.array_equal(zz, z)
    qw, sc, zs = O.awq_pack(W16, s_c)
    inv_s = (np.float32(1) / s_c).astype(np.float32)
    X16 = rng.integers(-8, 9, size=(M, K)).astype(np.float16)
    Y, _ = O.linear(X16, qw, sc, zs, inv_s)
    assert np.array_equal(Y, X16.astype(np.float64) @ W.T)


def test_rtn_error_bound():
    """Round-to-nearest error is at most half a step ("AWQ量化实战" §2.2).
    Exactly: |w' - w^'| <= s16/2 + 15|s32 - s16| + 2 ulp(w'), because the fp16
    rounding of the step can move the top grid point by 15|s32 - s16|; and
    almost every weight meets the bare s16/2."""
    rng = np.random.default_rng(2)
    N, K = 256, 1024
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1.5, 1.5, size=K)).astype(np.float32)
    qw, sc, zs = O.awq_pack(W16, s_c)
    wp = W16.astype(np.float64) * s_c.astype(np.float64)
    wq = O.dequant(qw, sc, zs).astype(np.float64)
    g = wp.reshape(N, K // 128, 128)
    s32 = (g.max(2) - g.min(2)) / 15.0
    s16 = sc.astype(np.float64)
    bound = s16 / 2 + 15 * np.abs(s32 - s16)
    err = np.abs(wp - wq).reshape(N, K // 128, 128)
    slack = 4 * np.spacing(np.abs(wp).astype(np.float32)).astype(np.float64).reshape(err.shape)
    assert np.all(err <= bound[:, :, None] + slack)
    frac_half = np.mean(err <= s16[:, :, None] / 2 + slack)
    assert frac_half >= 0.999


def test_codes_are_nearest_by_exhaustive_search():
    """Brute force: each stored code minimises |w'/s - (c - z)| over all 16
    codes c (w'/s as the fp32 quotient), with exact midpoints sent to the
    even integer, unless it is clamped at 0 or 15."""
    rng = np.random.default_rng(3)
    N, K = 48, 256
    W16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    q, z, s16 = O.quantize(W16)
    s = np.repeat(s16.astype(np.float32), 128, axis=1)
    zf = np.repeat(z.astype(np.float64), 128, axis=1)
    quot = (W16.astype(np.float32) / s).astype(np.float64)
    codes = np.arange(16, dtype=np.float64)
    dist = np.abs(quot[:, :, None] - (codes[None, None, :] - zf[:, :, None]))
    best = dist.min(axis=2)
    mine = np.take_along_axis(dist, q[:, :, None].astype(np.int64), 2)[:, :, 0]
    assert np.all(mine == best)
    ties = (dist == best[:, :, None]).sum(axis=2) > 1
    r = q.astype(np.int64) - zf.astype(np.int64)
    assert np.all((r[ties] % 2) == 0)


def test_hand_derived_golden_groups():
    g = _load_golden("hand_derived_groups.txt")
    K = g["K"]
    k = np.arange(K)
    w = np.empty(K, dtype=np.float64)
    w[:128] = ((k[:128] % 16) - 3) / 4.0
    i = np.arange(128)
    u = np.where(i == 0, 0.0, np.where(i == 1, 15.0, 0.5 + ((i - 2) % 15)))
    w[128:256] = u / 4.0
    w[256:] = 1.0
    W16 = w.astype(np.float16)[None, :]
    qw, sc, zs = O.awq_pack(W16)
    assert [int(v) for v in sc.view(np.uint16)[0]] == g["scales"]
    assert [int(v) for v in zs[0]] == g["zeros"]
    assert [int(v) for v in qw[0]] == g["qweight"]
    # the same row stored at half size with s_c = 2 packs identically
    qw2, sc2, zs2 = O.awq_pack((w / 2).astype(np.float16)[None, :],
                               np.full(K, 2.0, dtype=np.float32))
    assert np.array_equal(qw2, qw) and np.array_equal(sc2, sc) and np.array_equal(zs2, zs)


def test_tie_rule_closed_form():
    """Group 1 of the golden row: rint(m + 1/2) = m + (m & 1)."""
    m = np.arange(15)
    i = np.arange(128)
    u = np.where(i == 0, 0.0, np.where(i == 1, 15.0, 0.5 + ((i - 2) % 15)))
    W16 = (u / 4.0).astype(np.float16)[None, :]
    q, z, s16 = O.quantize(W16)
    expect = np.where(i == 0, 0, np.where(i == 1, 15, ((i - 2) % 15) + (((i - 2) % 15) & 1)))
    assert np.array_equal(q[0], expect) and z[0, 0] == 0
    assert set(m + (m & 1)) <= set(range(16))


def test_degenerate_groups():
    """Constant groups (zero range) floor the step at 2^-14; a group of zeros
    dequantizes to zeros; huge ranges cap the step at the largest fp16."""
    W16 = np.zeros((3, 128), dtype=np.float16)
    W16[1, :] = -2.0
    W16[2, :64] = -65000.0
    W16[2, 64:] = 65000.0
    s_c = np.ones(128, dtype=np.float32)
    s_c[:] = 8.0
    q, z, s16 = O.quantize(W16, s_c)
    assert s16[0, 0] == np.float16(2.0 ** -14) and z[0, 0] == 0 and np.all(q[0] == 0)
    # w' = -16: z = clamp(rint(16 / 2^-14)) = 15, q = clamp(-262144 + 15) = 0
    assert z[1, 0] == 15 and np.all(q[1] == 0)
    assert s16[2, 0] == np.float16(65504.0)
    qw, sc, zs = O.awq_pack(W16[:1])
    assert np.all(O.dequant(qw, sc, zs) == 0)


# ---------------------------------------------------------------- packing
def test_pack_roundtrip_and_zero_padding():
    rng = np.random.default_rng(4)
    q = rng.integers(0, 16, size=(7, 11008)).astype(np.uint8)
    assert np.array_equal(O.unpack_codes(O.pack_codes(q)), q)
    z = rng.integers(0, 16, size=(7, 86)).astype(np.uint8)
    zp = O.pack_zeros(z)
    assert zp.shape == (7, 11)
    assert np.array_equal(O.unpack_zeros(zp, 86), z)
    assert np.all((zp[:, -1] >> np.uint32(24)) == 0)   # nibbles 6, 7 of word 10 are padding
    one = np.zeros((1, 8), dtype=np.uint8)
    one[0, 5] = 0xA
    assert int(O.pack_codes(one)[0, 0]) == 0xA << 20


# ------------------------------------------------------------- the linear
def _codes_layer(q, z, s16):
    return O.pack_codes(q), np.asarray(s16, dtype=np.float16), O.pack_zeros(z)


def test_linear_row_sums_closed_form():
    """s = 1 and q = z + 1 everywhere give w^ = 1, so Y^ is the row sums of X."""
    rng = np.random.default_rng(5)
    M, N, K = 6, 16, 384
    z = rng.integers(0, 15, size=(N, K // 128)).astype(np.uint8)
    q = (np.repeat(z, 128, axis=1) + 1).astype(np.uint8)
    s16 = np.ones((N, K // 128), dtype=np.float16)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    Y, B = O.linear(X16, *_codes_layer(q, z, s16))
    rows = X16.astype(np.float64).sum(axis=1)
    assert np.allclose(Y, rows[:, None], rtol=0, atol=1e-12)
    assert np.allclose(B, np.abs(X16.astype(np.float64)).sum(axis=1)[:, None], rtol=0, atol=1e-12)


def test_linear_single_code_picks_one_input_channel():
    """q = z everywhere except one code z+1 at (n0, k0): column n0 of Y^ is
    s * inv_s[k0] * X[:, k0] and every other column is zero (catches a
    transposed operand or a wrong channel index for 1/s_c)."""
    rng = np.random.default_rng(6)
    M, N, K = 5, 24, 512
    n0, k0 = 17, 300
    z = rng.integers(0, 15, size=(N, K // 128)).astype(np.uint8)
    q = np.repeat(z, 128, axis=1).astype(np.uint8)
    q[n0, k0] += 1
    s16 = np.full((N, K // 128), 0.5, dtype=np.float16)
    inv_s = np.exp2(rng.integers(-3, 4, size=K)).astype(np.float32)
    X16 = rng.standard_normal((M, K)).astype(np.float16)
    Y, _ = O.linear(X16, *_codes_layer(q, z, s16), inv_s)
    expect = 0.5 * inv_s[k0] * X16[:, k0].astype(np.float64)
    assert np.array_equal(Y[:, n0], expect)
    Y[:, n0] = 0
    assert np.all(Y == 0)


def test_ulp_fp16_closed_forms():
    u = O.ulp_fp16(np.array([1.0, 1.5, 2.0, 65504.0, 1e-6, 0.0, -3.0, 2.0 ** -14]))
    assert list(u) == [2.0 ** -10, 2.0 ** -10, 2.0 ** -9, 32.0, 2.0 ** -24,
                       2.0 ** -24, 2.0 ** -9, 2.0 ** -24]


# ---------------------------------------------------------------- stats
def test_absmean_closed_form():
    """Columns of alternating +-v have mean |x| = v exactly; a column of
    T-1 zeros and one value v has mean v/T."""
    T, K = 64, 16
    v = np.arange(1, K + 1) / 8.0
    sign = np.where(np.arange(T) % 2 == 0, 1.0, -1.0)
    X = (sign[:, None] * v[None, :]).astype(np.float16)
    X[:, 3] = 0
    X[7, 3] = 6.0
    a = O.absmean(X)
    expect = v.copy()
    expect[3] = 6.0 / T
    assert np.array_equal(a, expect.astype(np.float32))


def test_channel_scales_closed_forms():
    a = np.array([4.0, 16.0, 1.0, 0.0, 9.0], dtype=np.float32)
    s, inv = O.channel_scales(a, 0.5)
    assert list(s[:3]) == [2.0, 4.0, 1.0] and s[4] == 3.0
    assert s[3] == np.float32(np.sqrt(np.float64(np.float32(1e-8))))
    assert list(inv[:3]) == [0.5, 0.25, 1.0]
    s0, inv0 = O.channel_scales(a, 0.0)
    assert np.all(s0 == 1) and np.all(inv0 == 1)
    assert list(O.alpha_grid(20)[:3]) == [0.0, 0.05, 0.1] and len(O.alpha_grid()) == 20
    assert O.alpha_grid(20)[-1] == 0.95


# --------------------------------------------------------------- search
def _toy():
    K, N, lid = awq_inputs.layer("toy", "linear")
    return (awq_inputs.calib_tokens(256, K, lid), awq_inputs.weight(N, K, lid))


def test_alpha_zero_is_plain_rtn():
    """alpha = 0 gives s_c = 1: the first candidate is plain group RTN, and its
    MSE equals the plain layer's error against X W^T."""
    X16, W16 = _toy()
    rows = np.arange(0, 512, 7)
    res = O.search(X16, W16, rows=rows)
    qw, sc, zs = O.awq_pack(W16[rows])
    Yq, _ = O.linear(X16, qw, sc, zs)
    Y = X16.astype(np.float64) @ W16[rows].astype(np.float64).T
    mse0 = np.mean((Yq - Y) ** 2)
    assert abs(res["mse"][0] - mse0) <= 1e-12 * mse0
    s_c, inv_s = O.channel_scales(res["a"], 0.0)
    assert np.array_equal(O.awq_pack(W16, s_c)[0], O.awq_pack(W16)[0])


def test_search_direct_matches_gram_identity():
    """Two routes to the per-row error: the direct T-long sum and
    d^T (X^T X) d.  They differ only by the fp32 rounding of x~ (a few 1e-7
    relative of the output, far below 1e-5 of the squared error)."""
    X16, W16 = _toy()
    H = O.gram(X16)
    a = O.absmean(X16)
    rows = np.arange(0, 512, 3)
    for al in (0.0, 0.35, 0.9):
        s_c, inv_s = O.channel_scales(a, al)
        e_d = O.row_errors(X16, W16, s_c, inv_s, rows)
        e_g = O.row_errors_gram(H, W16, s_c, inv_s, rows)
        assert np.allclose(e_d, e_g, rtol=1e-5, atol=0)


def test_search_uniform_activations_tie_to_smallest_alpha():
    """If every channel has the same strength 1, all candidates coincide, all
    MSEs are equal and the tie goes to alpha = 0."""
    X16, W16 = _toy()
    res = O.search(X16, W16, rows=np.arange(0, 512, 16), a=np.ones(512, np.float32))
    assert np.all(res["mse"] == res["mse"][0])
    assert res["best"] == 0 and res["alpha"] == 0.0


def test_search_beats_rtn_on_outlier_channels():
    """The method's claim ("AWQ量化实战" §2.2): with a few large-activation
    channels, activation-aware scaling lowers the output error below plain
    RTN, so the search picks alpha > 0 with a smaller MSE."""
    X16, W16 = _toy()
    res = O.search(X16, W16, rows=np.arange(0, 512, 2))
    assert res["best"] > 0
    assert res["mse"][res["best"]] < 0.9 * res["mse"][0]


def test_salient_channel_scaling_lowers_its_error():
    """Brute force on tiny layers (one group, K = 128, N = 256, 100 seeds):
    scaling one input channel c by s > 1 before quantization lowers that
    channel's mean effective-weight error |w - w^(s)/s| over the rows where c
    is not the group's min or max ("AWQ量化实战" §2.2), and every row's error
    obeys the scaled half-step bound Delta'/(2s)."""
    K, N = 128, 256
    for seed in range(100):
        rng = np.random.default_rng(1000 + seed)
        W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
        Wf = W16.astype(np.float64)
        c = seed % K
        inner = (np.argmax(Wf, axis=1) != c) & (np.argmin(Wf, axis=1) != c)
        base = None
        for s in (1.0, 1.25, 1.5, 2.0):
            s_c = np.ones(K, dtype=np.float32)
            s_c[c] = s
            qw, sc, zs = O.awq_pack(W16, s_c)
            wq = O.dequant(qw, sc, zs).astype(np.float64)
            e = np.abs(Wf[:, c] - wq[:, c] / s)
            step = sc[:, 0].astype(np.float64)
            assert np.all(e <= step / (2 * s) + 15 * step / 2048 / s + 1e-9)
            m = e[inner].mean()
            if base is None:
                base = m
            else:
                assert m < base, (seed, s)
