"""Pins of the oracle's sketch head ([citric] "Step 3: the output layer became
the bottleneck": exact scores over the strongest hidden dimensions, a 1-bit
sign sketch of the rest -- one XOR and one bit count per 64-dimension block,
blocks grouped by size, one weight per block -- then exact scores for the best
approximate candidates only).

Each check ties the oracle to something other than itself: a hand-worked
table, the plain exact output layer when every word is a candidate, integer
arithmetic when every dimension is scored exactly, closed forms of the sketch
when every sign agrees or differs, magnitude tiers that fix the blocks, the
fp32 order of every sum, and the page's reported agreement with exact search
on a synthetic table.
"""
import numpy as np
import pytest

import oracle
import synth


def _bits(a):
    """bf16 bit patterns of values that bf16 holds exactly."""
    f = np.ascontiguousarray(a, np.float32)
    assert ((f.view(np.uint32) & 0xFFFF) == 0).all()
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# Hand-worked table.  x = [3, -1, 0.5, -2, 1, 0.25], k = 2, blocks of B = 2,
# cE = 2, sizes s = [0.1, 5, 1, 0.2, 4, 2] -> order d1 d4 d5 d2 d3 d0.
# Exact dims {0, 3} (|x| 3 and 2).  Block 0 = {d1, d4}: weight mean(1, 1) * 2 = 2;
# block 1 = {d5, d2}: weight mean(0.25, 0.5) * 2 = 0.75; block 2 = {d3, d0}: both
# exact, no sketched dims, weight 0.  Signs of x: d1 -, d4 +, d2 +, d5 +.
_X = [3, -1, 0.5, -2, 1, 0.25]
_S = [0.1, 5, 1, 0.2, 4, 2]
_E = [
    [1, 5, 1, 1, 1, 1],  # exact 3 - 2 = 1; b0: d1 differs, d4 agrees -> 0; b1 agrees twice -> 0.75*2; approx 2.5
    [-1, -1, -1, 1, 1, -1],  # exact -3 - 2 = -5; b0 agrees twice -> 2*2; b1 differs twice -> -0.75*2; approx -2.5
    [0, 0, 0, 0, 0, 0],  # +0 has sign +: b0 -> 0, b1 -> 1.5; approx 1.5
    [2, -1, 1, -0.5, -1, -1],  # exact 6 + 1 = 7; b0: agree + differ; b1: agree + differ; approx 7
    [1, 5, 1, 1, 1, 1],  # same as word 0: approx 2.5 (tie, the lower index ranks first)
    [0, -8, -0.125, 0, -0.125, -0.125],  # exact 0; b0 -> 0; b1 differs twice -> -1.5; approx -1.5
]
_APPROX = [2.5, -2.5, 1.5, 7.0, 2.5, -1.5]
_LOGITS = [-2.25, -3.75, 0.0, 7.25, -2.25, 7.78125]  # full dot products, by hand


def _hand(n_cand, E=None):
    perm = oracle.sketch_perm(np.float32(_S))
    return oracle.sketch_head(_bits(_E if E is None else E), np.float32(_X), perm=perm, B=2, k=2, n_cand=n_cand,
                              cE=2.0)


def test_hand_worked_table():
    np.testing.assert_array_equal(oracle.sketch_perm(np.float32(_S)), [1, 4, 5, 2, 3, 0])
    nxt, cand, cl, approx = _hand(2)
    np.testing.assert_array_equal(approx, np.float32(_APPROX))
    np.testing.assert_array_equal(cand, [0, 3])  # 7, then 2.5 at words 0 and 4 -> word 0
    np.testing.assert_array_equal(cl, np.float32([_LOGITS[0], _LOGITS[3]]))
    # word 5 has the largest full score but not a candidate's approximate score:
    # every word outside the candidates scores minus infinity
    assert nxt == 3
    nxt3, cand3, _, _ = _hand(3)
    np.testing.assert_array_equal(cand3, [0, 3, 4])
    assert nxt3 == 3
    nxt6, cand6, cl6, _ = _hand(6)
    np.testing.assert_array_equal(cand6, np.arange(6))
    np.testing.assert_array_equal(cl6, np.float32(_LOGITS))
    assert nxt6 == 5


def test_size_order():
    np.testing.assert_array_equal(oracle.sketch_perm(np.float32([1, -3, 2, 3, -1])), [1, 3, 2, 0, 4])  # ties: lower d
    np.testing.assert_array_equal(oracle.sketch_perm(None, 5), np.arange(5))


def test_every_word_a_candidate_is_the_exact_output_layer():
    d = synth.sketch_head(21, 3000, 200)
    x = synth.sketch_x(21, 0, d["scale"])
    nxt, cand, cl, _ = oracle.sketch_head(d["emb"], x, perm=oracle.sketch_perm(d["scale"]), k=32, n_cand=3000)
    nx_ref, lg_ref = oracle.lm_head_argmax(d["emb"], x)
    np.testing.assert_array_equal(cand, np.arange(3000))
    np.testing.assert_array_equal(cl, lg_ref)
    assert nxt == nx_ref


@pytest.mark.parametrize("n_cand", [1, 17, 300])
def test_all_dims_exact_is_integer_top_n(n_cand):
    """k = D: no sketch; with small integers every fp32 step is exact, so the
    approximate score is the integer dot product and the candidates are its
    top n (ties to the lower index)."""
    V, D = 2000, 96
    E = synth.int_range(22, 1, V * D, -8, 8).reshape(V, D).astype(np.float32)
    x = synth.int_range(22, 2, D, -8, 8).astype(np.float32)
    E[5] = E[9]  # equal scores at words 5 and 9
    _, cand, cl, approx = oracle.sketch_head(_bits(E), x, k=D, n_cand=n_cand, cE=1.0)
    dots = E.astype(np.int64) @ x.astype(np.int64)
    np.testing.assert_array_equal(approx, dots.astype(np.float32))
    order = np.lexsort((np.arange(V), -dots))
    np.testing.assert_array_equal(cand, np.sort(order[:n_cand]))
    np.testing.assert_array_equal(cl, dots[cand].astype(np.float32))


def test_sketch_closed_forms_when_signs_all_agree_or_all_differ():
    """With the exact dims of a word zeroed, its approximate score is the
    sketch alone: cE * sum of |x| over the sketched dims when every sign agrees
    (each block contributes mean * count), its negative when every sign
    differs -- whatever the block order."""
    D, k, cE = 1152, 32, 0.0172
    d = synth.sketch_head(23, 1, D)
    x = synth.sketch_x(23, 0, d["scale"])
    top = np.argsort(-np.abs(x), kind="stable")[:k]
    rest = np.setdiff1d(np.arange(D), top)
    s = np.where(np.signbit(x), -1.0, 1.0).astype(np.float32)
    E = np.zeros((2, D), np.float32)
    E[0, rest] = 0.5 * s[rest]
    E[1, rest] = -0.25 * s[rest]
    total = cE * np.abs(x[rest]).astype(np.float64).sum()
    for perm in (None, oracle.sketch_perm(d["scale"])):
        _, _, _, approx = oracle.sketch_head(_bits(E), x, perm=perm, k=k, n_cand=1, cE=cE)
        np.testing.assert_allclose(approx, [total, -total], rtol=2e-6)


def test_blocks_follow_the_size_order():
    """Four tiers of 16 dimensions with sizes 8, 4, 2, 1 at scattered places:
    ordered by size, blocks of 16 are the tiers (k = 0).  A word agreeing on
    the 8-tier and differing elsewhere scores cE * 16 * (8 - 4 - 2 - 1)."""
    D, cE = 64, 0.5
    place = synth.splitmix64_seq(24, D).argsort(kind="stable")
    mag = np.empty(D, np.float32)
    mag[place] = np.repeat(np.float32([8, 4, 2, 1]), 16)
    sgn = np.where(synth.splitmix64_seq(25, D) & np.uint64(1), -1.0, 1.0).astype(np.float32)
    x = mag * sgn
    perm = oracle.sketch_perm(mag)
    E = np.zeros((3, D), np.float32)
    E[0] = np.where(mag == 8, sgn, -sgn)
    E[1] = np.where(mag == 1, sgn, -sgn)  # agrees on the 1-tier only: 16 * (1 - 8 - 4 - 2)
    E[2] = sgn  # all agree: 16 * 15
    _, _, _, approx = oracle.sketch_head(_bits(E), x, perm=perm, B=16, k=0, n_cand=1, cE=cE)
    np.testing.assert_array_equal(approx, np.float32([cE * 16 * 1, cE * 16 * -13, cE * 16 * 15]))


def test_last_block_is_partial():
    """D = 5 in blocks of 2: {d0, d1} weight 2.5, {d2, d3} weight 1.5, {d4} weight 1
    (its missing position counts +0 in the sum, not in the count).  A word agreeing
    on d1 only: 2.5 * 0 + 1.5 * -2 + 1 * -1 = -4; all agree: 9 = sum |x|."""
    x = np.float32([1, -4, 1, 2, -1])
    s = np.where(np.signbit(x), -1.0, 1.0)
    E = np.float32([np.where(np.arange(5) == 1, s, -s), s])
    _, _, _, approx = oracle.sketch_head(_bits(E), x, B=2, k=0, n_cand=1, cE=1.0)
    np.testing.assert_array_equal(approx, np.float32([-4.0, 9.0]))


def test_fp32_order_of_the_sketch():
    """Blocks are added one by one in block order: w = [1, t, t] (t = 2^-24)
    gives (1 + t) + t = 1 (ties to even), the reverse order 1 + 2^-23.  Inside a
    block |x| is summed as a balanced tree over its positions: [1, t, t, t]
    gives (1 + t) + (t + t) = 1 + 2^-23 (one by one: 1)."""
    t = np.float32(2.0 ** -24)
    _, _, _, a1 = oracle.sketch_head(_bits(np.ones((1, 3), np.float32)), np.float32([1, t, -t]) * [1, 1, -1],
                                     B=1, k=0, n_cand=1, cE=1.0)
    assert a1[0] == np.float32(1.0)
    _, _, _, a2 = oracle.sketch_head(_bits(np.ones((1, 4), np.float32)), np.float32([1, t, t, t]), B=4, k=0,
                                     n_cand=1, cE=1.0)
    assert a2[0] == np.float32(1.0 + 2.0 ** -23)


def test_exact_part_is_a_pairwise_sum_in_dimension_order():
    """The exact products are summed as a balanced tree (zero-padded to a power
    of two) in ascending dimension order.  With t = 2^-24: [1, t, t] gives
    (1 + t) + (t + 0) = 1 (reversed order: 2t + 1 = 1 + 2^-23); [1, t, t, t]
    gives (1 + t) + (t + t) = 1 + 2^-23 (one by one: 1)."""
    t = np.float32(2.0 ** -24)
    for x, want in (([1, t, t], 1.0), ([1, t, t, t], 1.0 + 2.0 ** -23)):
        x = np.float32(x)
        E = np.ones((1, len(x)), np.float32)
        _, _, _, approx = oracle.sketch_head(_bits(E), x, k=len(x), n_cand=1, cE=1.0)
        assert approx[0] == np.float32(want)


def test_signs_are_sign_bits():
    """Signs are compared bit for bit: -0.0 in x (or in the table) counts as
    negative.  One block (weight mean(2, 0, 1) = 1): the first word differs at
    the -0.0, 3 - 2 = 1; the second word's -0.0 entry agrees with it, 3."""
    x = np.float32([2.0, -0.0, 1.0])
    E = np.float32([[1, 1, 1], [1, -0.0, 1]])
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=0, n_cand=1, cE=1.0)
    np.testing.assert_array_equal(approx, np.float32([1.0, 3.0]))


def test_equal_exact_scores_pick_the_lower_index():
    nxt, cand, _, _ = _hand(2, E=np.float32(_E + [_E[3]]))  # word 6 copies word 3: approx 7, logit 7.25
    np.testing.assert_array_equal(cand, [3, 6])
    assert nxt == 3


def test_agrees_with_exact_search_on_a_synthetic_table():
    """The page reports the same word as exact search on every checked
    position with about 1000 candidates and the 32 strongest dimensions exact."""
    V, D = 65536, 1152
    d = synth.sketch_head(27, V, D)
    emb = d["emb"]
    perm = oracle.sketch_perm(d["scale"])
    cE = oracle.sketch_ce(emb)
    for tok in range(6):
        x = synth.sketch_x(27, tok, d["scale"])
        nxt, _, _, approx = oracle.sketch_head(emb, x, perm=perm, k=32, n_cand=1024, cE=cE)
        nx_ref, lg = oracle.lm_head_argmax(emb, x)
        assert nxt == nx_ref
        assert np.corrcoef(approx, lg)[0, 1] > 0.7


def test_ce_is_the_mean_magnitude():
    assert oracle.sketch_ce(_bits(np.float32([[0.5, -0.5], [-0.5, 0.5]]))) == 0.5
    assert oracle.sketch_ce(_bits(np.float32([[1, -2], [0, 3]]))) == 1.5


@pytest.mark.parametrize("k,n_cand,perm", [(7, 1, None), (2, 5, None), (2, 1, [0, 1, 2, 3, 4, 4]),
                                           (2, 1, [0, 1, 2, 3, 4, 6])])
def test_invalid_arguments(k, n_cand, perm):
    E = _bits(np.zeros((4, 6), np.float32))
    x = np.ones(6, np.float32)
    with pytest.raises(ValueError):
        oracle.sketch_head(E, x, perm=perm, k=k, n_cand=n_cand, cE=1.0)
