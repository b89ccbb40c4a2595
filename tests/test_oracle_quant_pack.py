"""Pins of the oracle's quantisers (S1, S3), packing (S2) and ternary linear (S4, S6).

Each check ties the oracle to something other than itself: hand-worked vectors
(tests/golden, cited there), a library routine (numpy.base_repr, integer
matmul), brute force over every byte value, or an invariant.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import read_facts, read_golden


# ---------------------------------------------------------------- S1 / S3 quantisation
@pytest.mark.parametrize("row", read_golden("w8_quant_hand.txt"))
def test_w8_quant_hand_vectors(row):
    w = np.array(row[0], np.float32)
    q, s = oracle.w8_quantize(w)
    np.testing.assert_allclose(np.float32(s), np.float32(float(row[1][0])), rtol=1e-6)
    np.testing.assert_array_equal(q, np.array(row[2], np.int8))


@pytest.mark.parametrize("row", read_golden("w8_quant_hand.txt"))
def test_activation_quant_hand_vectors(row):
    # the per-row activation quantiser uses the same rule
    x = np.array(row[0], np.float32)[None, :]
    xq, xs = oracle.quant_i8(x)
    np.testing.assert_allclose(xs[0], np.float32(float(row[1][0])), rtol=1e-6)
    np.testing.assert_array_equal(xq[0], np.array(row[2], np.int8))


def test_quant_error_bound_and_extremes():
    w = synth.normal_f32(0, 99, (4096,), 0.0, 0.02)
    q, s = oracle.w8_quantize(w)
    # reconstruction within half a step, absmax element maps to +-127
    assert np.max(np.abs(q.astype(np.float64) * s - w)) <= s * 0.5 * (1 + 1e-6)
    i = int(np.argmax(np.abs(w)))
    assert abs(int(q[i])) == 127
    assert q.min() >= -127 and q.max() <= 127


def test_activation_quant_rows_independent():
    x = synth.normal_f32(1, 98, (3, 257))
    xq, xs = oracle.quant_i8(x)
    for m in range(3):
        q1, s1 = oracle.quant_i8(x[m:m + 1])
        np.testing.assert_array_equal(q1[0], xq[m])
        assert s1[0] == xs[m]
    # scaling a row by a power of two scales the step and leaves the codes unchanged
    q2, s2 = oracle.quant_i8(x * 4.0)
    np.testing.assert_array_equal(q2, xq)
    np.testing.assert_array_equal(s2, xs * 4.0)


def test_quant_ties_go_to_even():
    # x/scale lands exactly on .5 values: scale 1 when absmax is 127
    x = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5]], np.float32)
    xq, _ = oracle.quant_i8(x)
    np.testing.assert_array_equal(xq[0], [127, 0, 2, 2, 0, -2, -2])


# ---------------------------------------------------------------- S2 packing
@pytest.mark.parametrize("row", read_golden("t158_pack_hand.txt"))
def test_pack_hand_vectors(row):
    t = np.array(row[0], np.int8)[None, :]
    pk = oracle.t158_pack(t)
    assert pk.shape == (1, 1)
    assert int(pk[0, 0]) == int(row[1][0])


def _trits_of_byte_by_base_repr(b):
    """Trits of byte b from numpy.base_repr (library routine), least significant digit first."""
    digits = np.base_repr(b, 3).rjust(5, "0")[::-1]
    return [int(c) - 1 for c in digits]


def test_pack_unpack_all_243_bytes():
    t = np.array([_trits_of_byte_by_base_repr(b) for b in range(243)], np.int8)  # [243][5]
    pk = oracle.t158_pack(t)
    np.testing.assert_array_equal(pk[:, 0], np.arange(243, dtype=np.uint8))
    np.testing.assert_array_equal(oracle.t158_unpack(pk, 5), t)


@pytest.mark.parametrize("b", range(243, 256))
def test_unpack_rejects_invalid_bytes(b):
    with pytest.raises(ValueError):
        oracle.t158_unpack(np.array([[121, b]], np.uint8), 10)


@pytest.mark.parametrize("K", [1, 4, 5, 6, 31, 1152, 1157])
def test_pack_round_trip_ragged(K):
    t = synth.trits(3, K, (7, K))
    pk = oracle.t158_pack(t)
    assert pk.shape == (7, (K + 4) // 5)
    np.testing.assert_array_equal(oracle.t158_unpack(pk, K), t)
    # the digits past K in the last byte are zero trits (digit 1)
    if K % 5:
        last = pk[:, -1].astype(np.int64)
        for i in range(K % 5, 5):
            np.testing.assert_array_equal((last // 3 ** i) % 3, 1)


def test_pack_filler_bytes_and_pitch():
    t = synth.trits(4, 0, (3, 1152))
    pk = oracle.t158_pack(t, pitch=240)
    assert (pk[:, 231:] == 121).all()
    np.testing.assert_array_equal(pk[:, :231], oracle.t158_pack(t))


def test_pack_rejects_non_trits():
    with pytest.raises(ValueError):
        oracle.t158_pack(np.array([[0, 2, 0]], np.int8))


def test_page_figures():
    f = read_facts()
    assert 3 ** f["trits_per_byte"] == f["pow3_5"] <= 256
    assert 8 / f["trits_per_byte"] == pytest.approx(f["bits_per_weight_packed"])
    assert 1 - f["bits_per_weight_packed"] / 2 == pytest.approx(f["smaller_than_2bit"])
    cfg = synth.DecoderConfig(max_pos=16, **synth.GEMMA3_1B)
    n = cfg.n_layers * sum(r * c for _, r, c in cfg.matrices())
    assert n == 697_761_792 and abs(n - f["decoder_weights_approx"]) / f["decoder_weights_approx"] < 0.01
    assert cfg.vocab == f["vocab"] and cfg.dim == f["dim"] and cfg.n_layers == f["n_blocks"]
    # tokens/s ~= bandwidth / bytes per token
    assert f["bandwidth_gbs_laptop"] * 1e9 / f["bytes_per_token_final"] == pytest.approx(f["tok_s_cap_final"], rel=0.01)
    assert f["bandwidth_gbs_laptop"] * 1e9 / f["bytes_per_token_4bit"] == pytest.approx(f["tok_s_cap_4bit"], rel=0.05)


# ---------------------------------------------------------------- S4 / S6 ternary linear
@pytest.mark.parametrize("row", read_golden("t158_dot_hand.txt"))
def test_t158_dot_hand_vectors(row):
    t = np.array(row[0], np.int8)[None, :]
    xq = np.array(row[1], np.int8)[None, :]
    K = t.shape[1]
    acc, y = oracle.t158_linear(xq, np.ones(1, np.float32), oracle.t158_pack(t), 1.0, K)
    assert int(acc[0, 0]) == int(row[2][0])
    assert y[0, 0] == np.float32(int(row[2][0]))


def test_t158_brute_force_every_5_trit_row():
    rows = np.array([_trits_of_byte_by_base_repr(b) for b in range(243)], np.int8)
    pk = oracle.t158_pack(rows)
    acts = [np.full(5, 127), np.full(5, -127), np.zeros(5), np.ones(5), -np.ones(5),
            np.array([10, -3, 7, 127, -127]), synth.int_range(5, 0, 5, -127, 127)]
    xq = np.array(acts, np.int8)
    acc, _ = oracle.t158_linear(xq, np.ones(len(acts), np.float32), pk, 1.0, 5)
    np.testing.assert_array_equal(acc, xq.astype(np.int64) @ rows.astype(np.int64).T)


@pytest.mark.parametrize("K", [1, 4, 5, 6, 31, 1152])
@pytest.mark.parametrize("M", [1, 3])
def test_t158_random_matches_integer_matmul(M, K):
    t = synth.trits(6, K, (37, K))
    xq = synth.int_range(7, K, M * K, -127, 127).astype(np.int8).reshape(M, K)
    xs = synth.uniform_f32(8, K, (M,), 0.001, 0.1)
    ws = np.float32(0.0371)
    acc, y = oracle.t158_linear(xq, xs, oracle.t158_pack(t, pitch=(K + 4) // 5 + 3), ws, K)
    ref = xq.astype(np.int64) @ t.astype(np.int64).T
    np.testing.assert_array_equal(acc, ref)
    # epilogue: ((float)acc * ws) * xs in fp32, left to right
    np.testing.assert_array_equal(y, (ref.astype(np.float32) * ws) * xs[:, None])


def test_t158_invariants_and_extremes():
    K = 6912
    xq = synth.int_range(9, 0, K, -127, 127).astype(np.int8)[None, :]
    rows = np.stack([np.ones(K), np.zeros(K), -np.ones(K)]).astype(np.int8)
    acc, _ = oracle.t158_linear(xq, np.ones(1, np.float32), oracle.t158_pack(rows), 1.0, K)
    s = int(xq.astype(np.int64).sum())
    np.testing.assert_array_equal(acc[0], [s, 0, -s])
    full = np.full((1, K), 127, np.int8)
    acc, y = oracle.t158_linear(full, np.ones(1, np.float32), oracle.t158_pack(rows[:1]), 1.0, K)
    assert int(acc[0, 0]) == 127 * K == 877_824


# ---------------------------------------------------------------- S5 W8 linear
def test_w8_linear_exact_small_integers():
    w = np.array([[127, 2.5, 3.5, -2.5, 0.5, -0.5, 126.5, -126.5]], np.float32)
    q, s = oracle.w8_quantize(w)
    assert s == 1.0
    x = np.array([[1, 2, 3, 4, 5, 6, 7, 8], [-1, 0, 1, 0, -1, 0, 1, 0]], np.float32)
    y = oracle.w8_linear(x, q, s)
    np.testing.assert_array_equal(y, (x.astype(np.int64) @ q.astype(np.int64).T).astype(np.float32))


@pytest.mark.parametrize("M,K,N", [(1, 288, 768), (4, 300, 65), (16, 64, 33)])
def test_w8_linear_matches_float64_matmul(M, K, N):
    d = synth.w8_gemv(11, M, K, N)
    q, s = oracle.w8_quantize(d["w"])
    y = oracle.w8_linear(d["x"], q, s)
    ref = (d["x"].astype(np.float64) @ q.astype(np.float64).T) * float(s)
    np.testing.assert_allclose(y, ref, rtol=1e-6, atol=1e-7 * np.abs(ref).max())


def test_w8_linear_pitch():
    d = synth.w8_gemv(12, 2, 40, 9)
    q, s = oracle.w8_quantize(d["w"])
    qp = np.zeros((9, 48), np.int8)
    qp[:, :40] = q
    qp[:, 40:] = 99  # padding is never read
    np.testing.assert_array_equal(oracle.w8_linear(d["x"], qp, s, K=40), oracle.w8_linear(d["x"], q, s))


# ---------------------------------------------------------------- zero-group skipping layout
def test_group_pack_hand_worked():
    # one row, K = 6: groups (-1, 0, 1, 1) and (1, -1, pad, pad)
    t = np.array([[-1, 0, 1, 1, 1, -1]], np.int8)
    g = oracle.t158_pack_groups(t, gpitch=3)
    # digits (0, 1, 2, 2) -> 0 + 3 + 18 + 54 = 75; (2, 0, 1, 1) -> 2 + 0 + 9 + 27 = 38; rows past N: 40
    np.testing.assert_array_equal(g, np.array([[75, 40, 40], [38, 40, 40]], np.uint8))


def test_group_pack_all_81_patterns_round_trip():
    pats = np.array([[((v // 3 ** i) % 3) - 1 for i in range(4)] for v in range(81)], np.int8)  # [81][4]
    g = oracle.t158_pack_groups(pats)  # one group, 81 rows
    np.testing.assert_array_equal(g[0], np.arange(81, dtype=np.uint8))
    np.testing.assert_array_equal(oracle.t158_unpack_groups(g, 81, 4), pats)


@pytest.mark.parametrize("N,K", [(7, 13), (64, 1152), (5, 4)])
def test_group_pack_round_trip_and_five_trit_agreement(N, K):
    t = synth.trits(40, 0, (N, K))
    g = oracle.t158_pack_groups(t, gpitch=N + 9)
    np.testing.assert_array_equal(oracle.t158_unpack_groups(g, N, K), t)
    np.testing.assert_array_equal(oracle.t158_unpack(oracle.t158_pack(t), K), t)  # the same trits either way
    assert (g[:, N:] == 40).all()


def test_group_unpack_rejects_bytes_above_80():
    g = np.full((1, 2), 81, np.uint8)
    with pytest.raises(ValueError):
        oracle.t158_unpack_groups(g, 2, 4)
