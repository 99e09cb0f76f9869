"""Pins of the oracle's weight-clipping search: no clipping reproduces the
plain quantizer, the Gram form of the group error equals the error summed
over the tokens, the search picks the best grid ratio by a brute force that
never forms the Gram, and clipping is chosen where it must help."""
import itertools

import numpy as np
import pytest

import oracle as O

VARIANTS = list(itertools.product((4, 8), (128, 64, 32), (True, False)))


@pytest.mark.parametrize("w_bit,group,zero_point", VARIANTS)
def test_ratio_one_is_the_plain_quantizer(w_bit, group, zero_point):
    rng = np.random.default_rng(w_bit + group)
    W16 = (rng.standard_normal((8, 256)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1, 1, size=256)).astype(np.float32)
    idx = np.zeros((8, 256 // group), dtype=np.uint8)
    a = O.quantize_clipped(W16, s_c, idx, 20, group, w_bit, zero_point)
    b = O.quantize(W16, s_c, group, w_bit, zero_point)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_clip_ratio_grid():
    r = O.clip_ratios(10)
    assert r[0] == 1.0 and r.dtype == np.float32
    assert np.allclose(np.diff(r), -0.05)
    assert r[-1] == np.float32(0.55)


def test_shrunk_range_clips_through_the_codes():
    # one group: the largest weight lies outside [r mn, r mx] and saturates
    w = np.linspace(-0.5, 1.0, 128).astype(np.float16)[None, :]
    idx = np.array([[10]], dtype=np.uint8)               # r = 0.75 on a 20-step grid
    q, z, s16 = O.quantize_clipped(w, None, idx, 20)
    r = np.float32(0.75)
    mx = np.float32(r * np.float32(w.max()))
    mn = np.float32(r * np.float32(w.min()))
    assert float(s16[0, 0]) == np.float16((mx - mn) / np.float32(15))
    assert q[0, -1] == 15 and q[0, 0] == 0
    deq = (q[0].astype(np.float64) - z[0, 0]) * float(s16[0, 0])
    assert deq.max() < float(w.max())                     # the top weight was clipped


def test_gram_error_equals_token_sum():
    rng = np.random.default_rng(3)
    T, K, N = 96, 256, 4
    X16 = rng.standard_normal((T, K)).astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s_c = np.exp(rng.uniform(-1, 1, size=K)).astype(np.float32)
    inv_s = (np.float32(1) / s_c).astype(np.float32)
    _, err = O.clip_search(X16, W16, s_c, inv_s, 6)
    xt = O.scaled_activations(X16, inv_s).astype(np.float64)
    wp = (W16.astype(np.float32) * s_c).astype(np.float64)
    for i in range(6):
        q, z, s16 = O.quantize_clipped(W16, s_c, np.full((N, 2), i), 6)
        wq = (q.reshape(N, 2, 128) - z[:, :, None].astype(np.float64)) * s16[:, :, None]
        d = wq.reshape(N, K) - wp
        for g in range(2):
            sl = slice(128 * g, 128 * g + 128)
            direct = ((xt[:, sl] @ d[:, sl].T) ** 2).sum(axis=0)   # sum over tokens
            assert np.allclose(err[:, g, i], direct, rtol=1e-10, atol=0)


def test_search_picks_the_best_ratio_by_brute_force():
    rng = np.random.default_rng(4)
    T, K, N = 64, 128, 6
    X16 = rng.standard_normal((T, K)).astype(np.float16)
    W16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    idx, err = O.clip_search(X16, W16, None, None, 12)
    xt = X16.astype(np.float64)
    for n in range(N):
        best, best_e = None, None
        for i in range(12):                    # ratio by ratio, errors from the tokens
            q, z, s16 = O.quantize_clipped(W16[n:n + 1], None, np.array([[i]]), 12)
            d = (q[0] - float(z[0, 0])) * float(s16[0, 0]) - W16[n].astype(np.float64)
            e = ((xt @ d) ** 2).sum()
            if best_e is None or e < best_e * (1 - 1e-12):
                best, best_e = i, e
        assert idx[n, 0] == best
        assert err[n, 0, idx[n, 0]] <= err[n, 0, 0]   # never worse than no clipping


def test_clipping_is_chosen_for_an_outlier_weight_on_a_silent_channel():
    # channel 0 carries a large weight but no activation: shrinking the range
    # costs nothing there and refines the step of every other weight
    rng = np.random.default_rng(5)
    T, K = 64, 128
    X16 = rng.standard_normal((T, K)).astype(np.float16)
    X16[:, 0] = 0
    w = (rng.standard_normal(K) * 0.01).astype(np.float16)
    w[0] = 0.5
    idx, err = O.clip_search(X16, w[None, :], None, None, 20)
    assert idx[0, 0] > 0
    assert err[0, 0, idx[0, 0]] < 0.5 * err[0, 0, 0]


def test_symmetric_shrunk_range_hand_derived():
    """Symmetric codes (zero point off, "AWQ量化实战" §3.3) from a range shrunk
    to r max|w'| (the clipping reading of §5.1), derived by hand.

    4-bit, 32-channel group, n_clip = 4, index 2: r = 1 - 0.5 * 2 / 4 = 0.75.
    max|w| = 1, so s32 = 0.75 / 7 = 0.107142857... = 1.7142857 * 2^-4; the
    fp16 mantissa field is round(0.7142857 * 1024) = round(731.43) = 731, so
    s = (1 + 731/1024) / 16 = 0.10711669921875.  Codes q = clamp(rint(w / s),
    -8, 7) + 8:  w = -1 -> -9.34 -> -8 -> 0;  1 -> 9.34 -> 7 -> 15;  0.5 ->
    4.67 -> 5 -> 13;  -0.5 -> 3;  0.25 -> 2.33 -> 2 -> 10;  -0.25 -> 6;
    0.125 -> 1.17 -> 1 -> 9;  0 -> 8;  0.75 -> 7.0017 -> 7 -> 15;  -0.75 ->
    1;  0.0625 -> 0.58 -> 1 -> 9;  0.03125 -> 0.29 -> 0 -> 8;  -0.875 ->
    -8.17 -> -8 -> 0;  0.875 -> 8.17 -> 7 -> 15 (clipped).  Without the
    shrink (r = 1) the step would be fp16(1/7) = 0.142822265625."""
    vals = [-1.0, 1.0, 0.5, -0.5, 0.25, -0.25, 0.125, 0.0, 0.75, -0.75, 0.0625, 0.03125,
            -0.875, 0.875, 0.0, 0.0]
    codes = [0, 15, 13, 3, 10, 6, 9, 8, 15, 1, 9, 8, 0, 15, 8, 8]
    w = np.array(vals * 2, dtype=np.float16)[None, :]
    q, z, s16 = O.quantize_clipped(w, None, np.array([[2]]), 4, group=32, w_bit=4,
                                   zero_point=False)
    assert float(s16[0, 0]) == 0.10711669921875
    assert z[0, 0] == 8
    assert q[0].tolist() == codes * 2
    q1, _, s1 = O.quantize_clipped(w, None, np.array([[0]]), 4, group=32, w_bit=4,
                                   zero_point=False)
    assert float(s1[0, 0]) == 0.142822265625


def test_symmetric_shrunk_range_hand_derived_8bit():
    """8-bit symmetric, 32-channel group, n_clip = 10, index 4: r = fp32(0.8).
    max|w| = 1 gives s32 = 0.8 / 127 = 0.0062992 = 1.6125984 * 2^-8; mantissa
    field round(0.6125984 * 1024) = round(627.30) = 627, so s = (1 + 627/1024)
    / 256 = 0.006298065185546875.  Codes q = clamp(rint(w / s), -128, 127) +
    128:  1 -> 158.8 -> 127 -> 255 (clipped);  0.5 -> 79.4 -> 79 -> 207;
    -0.25 -> -39.7 -> -40 -> 88;  fp16(0.1) = 0.0999755859375 -> 15.87 -> 16
    -> 144;  -1 -> -158.8 -> -128 -> 0;  0 -> 128."""
    vals = [1.0, 0.5, -0.25, 0.1, -1.0, 0.0, 0.0, 0.0]
    codes = [255, 207, 88, 144, 0, 128, 128, 128]
    w = np.array(vals * 4, dtype=np.float16)[None, :]
    q, z, s16 = O.quantize_clipped(w, None, np.array([[4]]), 10, group=32, w_bit=8,
                                   zero_point=False)
    assert float(s16[0, 0]) == 0.006298065185546875
    assert z[0, 0] == 128
    assert q[0].tolist() == codes * 4
