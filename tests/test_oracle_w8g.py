"""Pins of the oracle's W8 quantiser and linear layer with one scale per group
of G weights (gemma.cpp's I8Stream: int8 groups of 128 with a shared scale;
runq.c's Q8_0: symmetric, +-127, weights only).

Each check ties the oracle to something other than itself: hand-worked groups
whose scales are exactly 1 and 2, the per-tensor quantiser when every group
has the same maximum, integer arithmetic on small integers, and a float64
matrix product of the dequantised weights.
"""
import numpy as np
import pytest

import oracle
import synth


def _hand_row():
    # group 0 (128 weights): absmax 127 -> scale 1; group 1 (128): absmax 254 -> scale 2
    g0 = np.zeros(128, np.float32)
    g0[:8] = [127, 2.5, 3.5, -2.5, 0.5, -0.5, 126.5, -126.5]
    g1 = np.zeros(128, np.float32)
    g1[:5] = [254, 5, 7, 1, -3]
    return np.concatenate([g0, g1])


def test_w8g_hand_groups():
    q, s = oracle.w8g_quantize(_hand_row()[None, :], 128)
    np.testing.assert_array_equal(s, np.array([[1.0, 2.0]], np.float32))
    np.testing.assert_array_equal(q[0, :8], [127, 2, 4, -2, 0, 0, 126, -126])  # ties to even
    np.testing.assert_array_equal(q[0, 128:133], [127, 2, 4, 0, -2])  # 2.5 -> 2, 3.5 -> 4, 0.5 -> 0, -1.5 -> -2
    assert (q[0, 8:128] == 0).all() and (q[0, 133:] == 0).all()


def test_w8g_ragged_last_group_and_zero_group():
    w = np.zeros((2, 130), np.float32)
    w[0, :128] = 3.0
    w[0, 128:] = [0.5, -1.0]  # the short last group has its own absmax 1.0
    q, s = oracle.w8g_quantize(w, 128)
    assert s.shape == (2, 2)
    np.testing.assert_array_equal(q[0, 128:], [64, -127])  # 0.5 / (1/127) = 63.5 -> 64 (even)
    assert s[0, 1] == np.float32(np.float32(1.0) / np.float32(127.0))
    # an all-zero group: the 1e-9 floor, codes zero
    assert s[1, 0] == np.float32(np.float32(1e-9) / np.float32(127.0)) and (q[1] == 0).all()


def test_w8g_equals_per_tensor_when_groups_share_the_maximum():
    rng = np.random.default_rng(5)
    w = rng.uniform(-1, 1, (3, 512)).astype(np.float32)
    w[:, ::128] = 1.0  # every group of every row reaches 1.0
    qg, sg = oracle.w8g_quantize(w, 128)
    q, s = oracle.w8_quantize(w)
    np.testing.assert_array_equal(qg, q)
    assert (sg == s).all()


def test_w8g_single_group_is_the_row_quantiser():
    d = synth.w8_gemv(13, 1, 300, 1)
    qg, sg = oracle.w8g_quantize(d["w"], 1024)
    q, s = oracle.w8_quantize(d["w"])
    np.testing.assert_array_equal(qg, q)
    assert sg[0, 0] == s


def test_w8g_linear_exact_small_integers():
    q, s = oracle.w8g_quantize(_hand_row()[None, :], 128)
    x = np.zeros((2, 256), np.float32)
    x[0, :8] = [1, 2, 3, 4, 5, 6, 7, 8]
    x[0, 128:133] = [1, -1, 2, -2, 3]
    x[1, 0] = 2
    x[1, 128] = -1
    y = oracle.w8g_linear(x, q, s, 128)
    # by hand: group dot products times their scales
    d0 = np.int64(x[0, :8].astype(np.int64) @ q[0, :8].astype(np.int64))
    d1 = np.int64(x[0, 128:133].astype(np.int64) @ q[0, 128:133].astype(np.int64))
    assert y[0, 0] == np.float32(d0 * 1 + d1 * 2)
    assert y[1, 0] == np.float32(2 * 127 * 1 + (-1) * 127 * 2)


@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 50, 128), (3, 300, 17, 128), (2, 1000, 9, 64)])
def test_w8g_linear_matches_float64_product_of_dequantised_weights(M, K, N, G):
    d = synth.w8_gemv(14, M, K, N)
    q, s = oracle.w8g_quantize(d["w"], G)
    y = oracle.w8g_linear(d["x"], q, s, G)
    wdq = q.astype(np.float64) * np.repeat(s.astype(np.float64), G, axis=1)[:, :K]
    ref = d["x"].astype(np.float64) @ wdq.T
    np.testing.assert_allclose(y, ref, rtol=1e-6, atol=1e-7 * np.abs(ref).max())
    # and the group quantiser tracks the weights within half a step per group
    err = np.abs(wdq - d["w"].astype(np.float64))
    assert (err <= 0.5 * np.repeat(s, G, axis=1)[:, :K] * (1 + 1e-6)).all()
