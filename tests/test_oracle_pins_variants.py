"""Pins of the oracle's quantization variants: symmetric (zero point off),
group sizes 64 and 32, and 8-bit codes.

Each test checks a closed form (weights that lie exactly on a grid come back
exactly), a brute-force nearest-code search on small inputs, the round-to-
nearest bound, or a hand-built packed word, so that a slip (a wrong range, a
group index taken from the wrong width, a byte in the wrong place, an
off-by-one in the symmetric offset) fails at least one of them.
"""
import itertools

import numpy as np
import pytest

import oracle as O

VARIANTS = list(itertools.product((4, 8), (128, 64, 32), (True, False)))


def _grid(rng, N, K, group, w_bit, zero_point):
    """Weights exactly on a quantization grid that the quantizer must find:
    per group a power-of-two step, codes reaching both ends of the range."""
    G = K // group
    s = np.exp2(rng.integers(-9, -4, size=(N, G))).astype(np.float64)
    if zero_point:
        qmax = (1 << w_bit) - 1
        q = rng.integers(0, qmax + 1, size=(N, G, group))
        q[:, :, 0], q[:, :, 1] = 0, qmax
        z = rng.integers(0, qmax + 1, size=(N, G))
        w = (q - z[:, :, None]) * s[:, :, None]
    else:
        h = 1 << (w_bit - 1)
        q = rng.integers(-(h - 1), h, size=(N, G, group))
        q[:, :, 0] = h - 1              # max |w| = (h - 1) s, so s comes back exactly
        w = q * s[:, :, None]
    return w.reshape(N, K).astype(np.float16), s


@pytest.mark.parametrize("w_bit,group,zero_point", VARIANTS)
def test_grid_weights_come_back_exactly(w_bit, group, zero_point):
    rng = np.random.default_rng(w_bit * 1000 + group + zero_point)
    W16, s = _grid(rng, 8, 256, group, w_bit, zero_point)
    qw, sc, zs = O.awq_pack(W16, None, group, w_bit, zero_point)
    assert qw.shape == (8, 256 * w_bit // 32)
    assert sc.shape == (8, 256 // group)
    assert np.array_equal(sc.astype(np.float64), s)
    assert np.array_equal(O.dequant(qw, sc, zs, group, w_bit).astype(np.float64),
                          W16.astype(np.float64))


@pytest.mark.parametrize("w_bit,group,zero_point", VARIANTS)
def test_codes_are_nearest_and_within_half_a_step(w_bit, group, zero_point):
    rng = np.random.default_rng(7 + w_bit + group)
    N, K = 4, 128
    W16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    q, z, s16 = O.quantize(W16, None, group, w_bit, zero_point)
    s = s16.astype(np.float32)
    qmax = (1 << w_bit) - 1
    W = W16.astype(np.float32)
    for n in range(N):
        for k in range(K):
            g = k // group
            # brute force over every code: the stored one is a nearest grid point
            cand = (np.arange(qmax + 1, dtype=np.float64) - z[n, g]) * s[n, g]
            d = np.abs(cand - W[n, k])
            assert d[q[n, k]] == d.min()
            assert d[q[n, k]] <= 0.5 * s[n, g] * (1 + 1e-6)
    if not zero_point:
        h = 1 << (w_bit - 1)
        assert np.all(z == h)
        # max |w| maps to +-(h - 1): the code 0 (value -h) is never needed
        assert q.min() >= 1


def test_symmetric_step_is_max_abs_over_h_minus_1():
    W = np.zeros((1, 128), dtype=np.float16)
    W[0, 5], W[0, 9] = -0.75, 0.5       # max |w| = 0.75
    _, z, s16 = O.quantize(W, None, 128, 4, False)
    assert float(s16[0, 0]) == np.float16(0.75 / 7)
    assert z[0, 0] == 8
    _, z8, s8 = O.quantize(W, None, 128, 8, False)
    assert float(s8[0, 0]) == np.float16(0.75 / 127)
    assert z8[0, 0] == 128


def test_group_index_is_k_over_group():
    # groups of 32 with very different magnitudes are exact at group 32 only
    rng = np.random.default_rng(3)
    K = 128
    mag = np.exp2(np.repeat(np.array([-12, -2, -8, -4]), 32))
    q = rng.integers(0, 16, size=K)
    q[::32], q[1::32] = 0, 15
    W16 = ((q - 3) * mag).astype(np.float16)[None, :]
    for group, exact in ((32, True), (64, False), (128, False)):
        qw, sc, zs = O.awq_pack(W16, None, group, 4, True)
        same = np.array_equal(O.dequant(qw, sc, zs, group, 4), W16.astype(np.float32))
        assert same == exact, group


def test_eight_bit_packing_by_hand():
    q = np.array([[1, 2, 3, 4, 0xFF, 0x80, 0x7F, 0x00]], dtype=np.uint8)
    qw = O.pack_codes(q, 8)
    assert qw.tolist() == [[0x04030201, 0x007F80FF]]
    assert np.array_equal(O.unpack_codes(qw, 8), q)
    # zero points of 5 groups: 4 per word, padding bytes 0
    z = np.array([[9, 8, 7, 6, 5]], dtype=np.uint8)
    assert O.pack_zeros(z, 8).tolist() == [[0x06070809, 0x00000005]]
    assert np.array_equal(O.unpack_zeros(O.pack_zeros(z, 8), 5, 8), z)


@pytest.mark.parametrize("w_bit,group,zero_point", VARIANTS)
def test_linear_single_code_selects_one_input_channel(w_bit, group, zero_point):
    # one token equal to e_c returns column c of the dequantized weight
    rng = np.random.default_rng(11 + w_bit + group)
    W16 = (rng.standard_normal((16, 256)) * 0.02).astype(np.float16)
    qw, sc, zs = O.awq_pack(W16, None, group, w_bit, zero_point)
    X = np.zeros((1, 256), dtype=np.float16)
    X[0, 77] = 1.0
    y, _ = O.linear(X, qw, sc, zs, None, group, w_bit)
    assert np.array_equal(y[0], O.dequant(qw, sc, zs, group, w_bit)[:, 77].astype(np.float64))


@pytest.mark.parametrize("w_bit,group,zero_point", [(4, 64, True), (4, 128, False), (8, 128, True)])
def test_alpha_zero_is_plain_rtn_for_variants(w_bit, group, zero_point):
    rng = np.random.default_rng(5)
    X16 = rng.standard_normal((64, 256)).astype(np.float16)
    W16 = (rng.standard_normal((16, 256)) * 0.02).astype(np.float16)
    cfg = dict(group=group, w_bit=w_bit, zero_point=zero_point)
    res = O.search(X16, W16, n_grid=4, **cfg)
    e0 = O.row_errors(X16, W16, np.ones(256, np.float32), np.ones(256, np.float32), **cfg)
    assert np.array_equal(res["row_err"][0], e0)
    # and the Gram-identity route agrees with the direct one
    H = O.gram(X16)
    s_c, inv_s = O.channel_scales(res["a"], 0.5)
    d = O.row_errors(X16, W16, s_c, inv_s, **cfg)
    g = O.row_errors_gram(H, W16, s_c, inv_s, **cfg)
    assert np.allclose(d, g, rtol=1e-5, atol=0)


def test_eight_bits_are_finer_than_four():
    rng = np.random.default_rng(9)
    W16 = (rng.standard_normal((32, 512)) * 0.02).astype(np.float16)
    err = {}
    for b in (4, 8):
        qw, sc, zs = O.awq_pack(W16, None, 128, b, True)
        err[b] = np.abs(O.dequant(qw, sc, zs, 128, b) - W16.astype(np.float32)).mean()
    # 17x more levels: the mean error shrinks by about that factor
    assert err[8] * 10 < err[4]
