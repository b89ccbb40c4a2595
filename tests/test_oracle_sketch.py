"""Pins of the oracle's sketch head ([citric] "Step 3: the output layer became
the bottleneck": exact scores over the strongest hidden dimensions, a 1-bit
sign sketch of the rest with one weight per group, then exact scores for the
best approximate candidates only).

Each check ties the oracle to something other than itself: a hand-worked
table, the plain exact output layer when every word is a candidate, integer
arithmetic when every dimension is scored exactly, closed forms of the sketch
when every sign agrees or disagrees, magnitude tiers that fix the groups, and
the page's reported agreement with exact search on a synthetic table.
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


# Hand-worked table.  x = [3, -1, 0.5, -2, 1, 0.25], k = 2, G = 2, cE = 2.
# |x| ranks: d0 (3), d3 (2), d1 (1), d4 (1, tie -> after d1), d2 (0.5), d5 (0.25).
# Exact dims {0, 3}; group 0 = {1, 4}, weight mean(1, 1) * 2 = 2;
# group 1 = {2, 5}, weight mean(0.5, 0.25) * 2 = 0.75.  Signs of x on the
# sketched dims: d1 -, d4 +, d2 +, d5 +.
_X = [3, -1, 0.5, -2, 1, 0.25]
_E = [
    [1, 5, 1, 1, 1, 1],  # exact 3 - 2 = 1; g0: d1 differs, d4 agrees -> 0; g1: both agree -> 0.75*2; approx 2.5
    [-1, -1, -1, 1, 1, -1],  # exact -3 - 2 = -5; g0 agrees twice -> 2*2; g1 differs twice -> -0.75*2; approx -2.5
    [0, 0, 0, 0, 0, 0],  # +0 has sign +: g0 -> 0, g1 -> 1.5; approx 1.5
    [2, -1, 1, -0.5, -1, -1],  # exact 6 + 1 = 7; g0: agree + differ; g1: agree + differ; approx 7
    [1, 5, 1, 1, 1, 1],  # same as word 0: approx 2.5 (tie, the lower index ranks first)
    [0, -8, -0.125, 0, -0.125, -0.125],  # exact 0; g0 -> 0; g1 differs twice -> -1.5; approx -1.5
]
_APPROX = [2.5, -2.5, 1.5, 7.0, 2.5, -1.5]
_LOGITS = [-2.25, -3.75, 0.0, 7.25, -2.25, 7.78125]  # full dot products, by hand


def test_hand_worked_table():
    nxt, cand, cl, approx = oracle.sketch_head(_bits(_E), np.float32(_X), k=2, G=2, n_cand=2, cE=2.0)
    np.testing.assert_array_equal(approx, np.float32(_APPROX))
    np.testing.assert_array_equal(cand, [0, 3])  # 7, then 2.5 at words 0 and 4 -> word 0
    np.testing.assert_array_equal(cl, np.float32([_LOGITS[0], _LOGITS[3]]))
    # word 5 has the largest full score but not a candidate's approximate score:
    # every word outside the candidates scores minus infinity
    assert nxt == 3
    nxt3, cand3, _, _ = oracle.sketch_head(_bits(_E), np.float32(_X), k=2, G=2, n_cand=3, cE=2.0)
    np.testing.assert_array_equal(cand3, [0, 3, 4])
    assert nxt3 == 3
    nxt6, cand6, cl6, _ = oracle.sketch_head(_bits(_E), np.float32(_X), k=2, G=2, n_cand=6, cE=2.0)
    np.testing.assert_array_equal(cand6, np.arange(6))
    np.testing.assert_array_equal(cl6, np.float32(_LOGITS))
    assert nxt6 == 5


def test_every_word_a_candidate_is_the_exact_output_layer():
    d = synth.sketch_head(21, 3000, 200)
    nxt, cand, cl, _ = oracle.sketch_head(d["emb"], d["x"], k=32, G=8, n_cand=3000)
    nx_ref, lg_ref = oracle.lm_head_argmax(d["emb"], d["x"])
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
    _, cand, cl, approx = oracle.sketch_head(_bits(E), x, k=D, G=1, n_cand=n_cand, cE=1.0)
    dots = E.astype(np.int64) @ x.astype(np.int64)
    np.testing.assert_array_equal(approx, dots.astype(np.float32))
    order = np.lexsort((np.arange(V), -dots))
    np.testing.assert_array_equal(cand, np.sort(order[:n_cand]))
    np.testing.assert_array_equal(cl, dots[cand].astype(np.float32))


def test_sketch_closed_forms_when_signs_all_agree_or_all_differ():
    """With the exact dims of a word zeroed, its approximate score is the
    sketch alone: cE * sum of |x| over the sketched dims when every sign agrees
    (each group contributes mean * count), its negative when every sign differs."""
    D, k, G, cE = 1152, 32, 8, 0.0172
    x = synth.sketch_head(23, 1, D)["x"]
    top = np.argsort(-np.abs(x), kind="stable")[:k]
    rest = np.setdiff1d(np.arange(D), top)
    s = np.where(np.signbit(x), -1.0, 1.0).astype(np.float32)
    E = np.zeros((2, D), np.float32)
    E[0, rest] = 0.5 * s[rest]
    E[1, rest] = -0.25 * s[rest]
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=k, G=G, n_cand=1, cE=cE)
    total = cE * np.abs(x[rest]).astype(np.float64).sum()
    np.testing.assert_allclose(approx, [total, -total], rtol=2e-6)


def test_groups_follow_magnitude_tiers():
    """Four tiers of 16 dimensions each at |x| = 8, 4, 2, 1 make the four groups
    (k = 0): a word agreeing on the 8-tier and differing elsewhere scores
    cE * 16 * (8 - 4 - 2 - 1)."""
    D, cE = 64, 0.5
    perm = synth.splitmix64_seq(24, D).argsort(kind="stable")
    mag = np.repeat(np.float32([8, 4, 2, 1]), 16)
    sgn = np.where(synth.splitmix64_seq(25, D) & np.uint64(1), -1.0, 1.0).astype(np.float32)
    x = np.empty(D, np.float32)
    x[perm] = mag * sgn[:D]
    E = np.zeros((3, D), np.float32)
    s = np.where(np.signbit(x), -1.0, 1.0)
    tier8 = np.abs(x) == 8
    E[0] = np.where(tier8, s, -s)
    E[1] = np.where(np.abs(x) == 1, s, -s)  # agrees on the 1-tier only: 16 * (1 - 8 - 4 - 2)
    E[2] = s  # all agree: 16 * 15
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=0, G=4, n_cand=1, cE=cE)
    np.testing.assert_array_equal(approx, np.float32([cE * 16 * 1, cE * 16 * -13, cE * 16 * 15]))


def test_uneven_groups_take_floor_boundaries():
    """R = 5 sketched dims in G = 2 groups: group g holds ranks floor(g R / G)
    up to floor((g + 1) R / G), so the first group is the smaller one: {4, 2}
    with weight 3, then {1, 1, 1} with weight 1 (cE = 1).  A word agreeing on
    the 4-dimension only scores 3 * (2 - 2) + 1 * (3 - 6) = -3."""
    x = np.float32([1, -4, 1, 2, -1])
    s = np.where(np.signbit(x), -1.0, 1.0)
    E = np.float32([np.where(np.abs(x) == 4, s, -s), s])
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=0, G=2, n_cand=1, cE=1.0)
    np.testing.assert_array_equal(approx, np.float32([-3.0, 9.0]))


def test_groups_are_summed_in_order_from_the_largest():
    """Group terms are added one by one from the group of the largest |x|:
    (1 + 2^-24) + 2^-24 rounds to 1 twice (ties to even), while the other
    order would give 1 + 2^-23."""
    t = np.float32(2.0 ** -24)
    x = np.float32([t, 1.0, -t])
    E = np.float32([[1, 1, -1]])
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=0, G=3, n_cand=1, cE=1.0)
    assert approx[0] == np.float32(1.0)


def test_exact_part_is_a_pairwise_sum_in_dimension_order():
    """The exact products are summed as a balanced tree (zero-padded to a power
    of two) in ascending dimension order.  With t = 2^-24: [1, t, t] gives
    (1 + t) + (t + 0) = 1 (reversed order: 2t + 1 = 1 + 2^-23); [1, t, t, t]
    gives (1 + t) + (t + t) = 1 + 2^-23 (one by one: 1)."""
    t = np.float32(2.0 ** -24)
    for x, want in (([1, t, t], 1.0), ([1, t, t, t], 1.0 + 2.0 ** -23)):
        x = np.float32(x)
        E = np.ones((1, len(x)), np.float32)
        _, _, _, approx = oracle.sketch_head(_bits(E), x, k=len(x), G=1, n_cand=1, cE=1.0)
        assert approx[0] == np.float32(want)


def test_signs_are_sign_bits():
    """Signs are compared bit for bit: -0.0 in x (or in the table) counts as
    negative.  One group (weight mean(2, 0, 1) = 1): the first word differs at
    the -0.0, 3 - 2 = 1; the second word's -0.0 entry agrees with it, 3."""
    x = np.float32([2.0, -0.0, 1.0])
    E = np.float32([[1, 1, 1], [1, -0.0, 1]])
    _, _, _, approx = oracle.sketch_head(_bits(E), x, k=0, G=1, n_cand=1, cE=1.0)
    np.testing.assert_array_equal(approx, np.float32([1.0, 3.0]))


def test_equal_exact_scores_pick_the_lower_index():
    E = np.float32(_E + [_E[3]])  # word 6 copies word 3: approx 7 and logit 7.25 at both
    nxt, cand, _, _ = oracle.sketch_head(_bits(E), np.float32(_X), k=2, G=2, n_cand=2, cE=2.0)
    np.testing.assert_array_equal(cand, [3, 6])
    assert nxt == 3


def test_single_group_weight_is_mean_magnitude():
    """G = 1: the sketch is cE * mean|x| over the sketched dims * (agreeing - differing)."""
    D, k = 300, 20
    d = synth.sketch_head(26, 50, D)
    x = d["x"]
    _, _, _, approx = oracle.sketch_head(d["emb"], x, k=k, G=1, n_cand=1, cE=0.25)
    top = np.argsort(-np.abs(x), kind="stable")[:k]
    rest = np.setdiff1d(np.arange(D), top)
    E = synth.bf16_to_f32(d["emb"]).astype(np.float64)
    exact = E[:, top] @ x[top].astype(np.float64)
    agree = (np.signbit(E[:, rest]) == np.signbit(x[rest])).sum(1)
    sk = 0.25 * np.abs(x[rest]).astype(np.float64).mean() * (2 * agree - len(rest))
    np.testing.assert_allclose(approx, exact + sk, rtol=1e-5, atol=1e-5)


def test_agrees_with_exact_search_on_a_synthetic_table():
    """The page reports the same word as exact search on every checked
    position with about 1000 candidates and the 32 strongest dimensions exact."""
    V, D = 65536, 1152
    emb = synth.sketch_head(27, V, D)["emb"]
    cE = oracle.sketch_ce(emb)
    for seed in range(6):
        x = synth.sketch_head(100 + seed, 1, D)["x"]
        nxt, _, _, approx = oracle.sketch_head(emb, x, k=32, G=8, n_cand=1024, cE=cE)
        nx_ref, lg = oracle.lm_head_argmax(emb, x)
        assert nxt == nx_ref
        assert np.corrcoef(approx, lg)[0, 1] > 0.7


def test_ce_is_the_mean_magnitude():
    assert oracle.sketch_ce(_bits(np.float32([[0.5, -0.5], [-0.5, 0.5]]))) == 0.5
    assert oracle.sketch_ce(_bits(np.float32([[1, -2], [0, 3]]))) == 1.5


@pytest.mark.parametrize("k,G,n_cand", [(7, 1, 1), (0, 7, 1), (2, 1, 5), (2, 5, 1)])
def test_invalid_arguments(k, G, n_cand):
    E = _bits(np.zeros((4, 6), np.float32))
    x = np.ones(6, np.float32)
    with pytest.raises(ValueError):
        oracle.sketch_head(E, x, k=k, G=G, n_cand=n_cand, cE=1.0)
