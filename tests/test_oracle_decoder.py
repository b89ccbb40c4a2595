"""Pins of the oracle's decode step (S8-S16) and generation loop.

* A tiny decoder (2 blocks, hidden 64, 4 query heads / 1 KV head of 16, GeGLU
  160, vocab 512, seed 5) must produce the same 64 greedy tokens from a
  16-token prompt as an independent NumPy reference with dequantised float
  weights -- the check of the cpp20gemma README's "Tests" section (64-step
  greedy decoding matches the reference id for id; final logits within 2e-3).
* With all ternary weights zero, every block adds exactly 0 to the residual,
  so the logits have the closed form E . rmsnorm(E[token]).
"""
import numpy as np
import pytest

import oracle
import synth
from numpy_ref import NumpyDecoder, rmsnorm32


def tiny_cfg(max_pos=96):
    return synth.DecoderConfig(max_pos=max_pos, **synth.TINY)


@pytest.fixture(scope="module")
def tiny():
    cfg = tiny_cfg()
    w = synth.decoder_weights(cfg, seed=5)
    return cfg, w, oracle.Decoder(cfg, w), NumpyDecoder(cfg, w)


def test_tiny_decoder_64_greedy_tokens_match_numpy_reference(tiny):
    cfg, w, orc, ref = tiny
    prompt = synth.prompt_ids(5, 16, cfg.vocab)
    n_steps = 16 + 64 - 1
    ids_or = orc.generate(orc.new_cache(), prompt, 0, n_steps)
    ids_np = ref.generate(orc.new_cache(), prompt, 0, n_steps)
    np.testing.assert_array_equal(ids_or, ids_np)
    assert len(set(ids_or.tolist())) > 10  # argmaxes over the prompt positions vary


def test_tiny_decoder_small_embedding_switches_tokens():
    # A random model greedy-decodes into a fixed point; with a 10x smaller embedding
    # spread the blocks dominate the residual and the run changes token mid-way.
    cfg = tiny_cfg()
    w = synth.decoder_weights(cfg, seed=5, emb_std=0.002)
    orc, ref = oracle.Decoder(cfg, w), NumpyDecoder(cfg, w)
    prompt = synth.prompt_ids(5, 16, cfg.vocab)
    ids_or = orc.generate(orc.new_cache(), prompt, 0, 79)
    np.testing.assert_array_equal(ids_or, ref.generate(orc.new_cache(), prompt, 0, 79))
    assert len(set(ids_or[15:].tolist())) >= 3


def test_tiny_decoder_logits_and_cache_match(tiny):
    cfg, w, orc, ref = tiny
    kv_a, kv_b = orc.new_cache(), orc.new_cache()
    token = 7
    for pos in range(40):
        na, la = orc.step(kv_a, token, pos)
        nb, lb = ref.step(kv_b, token, pos)
        assert na == nb
        np.testing.assert_allclose(la, lb, rtol=0, atol=1e-6 * np.abs(lb).max())
        token = na
    np.testing.assert_array_equal(kv_a, kv_b)  # rotated k and v written at every position


def test_zero_weights_closed_form():
    cfg = tiny_cfg(max_pos=8)
    w = synth.decoder_weights(cfg, seed=6)
    for l in range(cfg.n_layers):
        for name in w["layers"][l]:
            w["layers"][l][name][:] = 0
    orc = oracle.Decoder(cfg, w)
    emb = synth.bf16_to_f32(w["emb"])
    for token, pos in [(3, 0), (500, 5)]:
        nx, logits = orc.step(orc.new_cache(), token, pos)
        hn = rmsnorm32(emb[token], w["g_final"], cfg.eps)
        ref = emb.astype(np.float64) @ hn.astype(np.float64)
        np.testing.assert_allclose(logits, ref, rtol=1e-6, atol=1e-9)
        assert nx == int(np.argmax(ref))


def test_generation_force_feeds_prompt(tiny):
    cfg, w, orc, _ = tiny
    prompt = np.array([11, 22, 33, 44], np.int32)
    ids = orc.generate(orc.new_cache(), prompt, 0, 6)
    # step s consumes prompt[s] for s < 4, so the same forwards give the same argmaxes
    kv = orc.new_cache()
    for s in range(4):
        nx, _ = orc.step(kv, int(prompt[s]), s)
        assert nx == ids[s]
    nx, _ = orc.step(kv, int(ids[3]), 4)
    assert nx == ids[4]


def test_argmax_first_maximum_wins():
    cfg = tiny_cfg(max_pos=4)
    w = synth.decoder_weights(cfg, seed=7)
    for l in range(cfg.n_layers):
        for name in w["layers"][l]:
            w["layers"][l][name][:] = 0
    w["emb"][:] = w["emb"][0]  # every row equal: every logit ties
    orc = oracle.Decoder(cfg, w)
    nx, logits = orc.step(orc.new_cache(), 9, 0)
    assert (logits == logits[0]).all() and nx == 0


def test_hidden_state_is_the_step_before_the_classifier(tiny):
    """The step cut before the classifier: the classifier of its hidden state
    gives the full step's token and logits exactly, the caches are the same,
    and the hidden state is the NumPy reference's final normalised residual."""
    cfg, w, orc, ref = tiny
    kv_a, kv_b, kv_c = orc.new_cache(), orc.new_cache(), orc.new_cache()
    token = 11
    for pos in range(24):
        xn = orc.hidden(kv_a, token, pos)
        nb, lb = orc.step(kv_b, token, pos)
        na, la = oracle.lm_head_argmax(w["emb"], xn)
        assert na == nb
        np.testing.assert_array_equal(la, lb)
        np.testing.assert_allclose(xn, ref.hidden(kv_c, token, pos), rtol=0, atol=1e-5 * np.abs(xn).max())
        token = nb
    np.testing.assert_array_equal(kv_a, kv_b)


def _cache(cfg, n_seqs):
    return np.zeros((n_seqs, cfg.n_layers, 2, cfg.max_pos, cfg.kv_dim), np.float32)


def test_lanes_of_separate_sequences_are_separate_steps(tiny):
    """Lanes of different sequences at different positions: each lane's token,
    logits and cache rows are those of the single-token step on its own cache."""
    cfg, w, orc, _ = tiny
    kvs = _cache(cfg, 3)
    rng_tok = synth.prompt_ids(6, 12, cfg.vocab)
    for s in range(3):  # give every sequence some history
        for p in range(4 + 2 * s):
            orc.step(kvs[s], int(rng_tok[p]), p, want_logits=False)
    ref = kvs.copy()
    tokens, positions, seqs = [11, 22, 33], [4, 6, 8], [0, 1, 2]
    nxt, lg = orc.lanes(kvs, tokens, positions, seqs, want_logits=True)
    for i in range(3):
        nx, l1 = orc.step(ref[seqs[i]], tokens[i], positions[i])
        assert nxt[i] == nx
        np.testing.assert_array_equal(lg[i], l1)
    np.testing.assert_array_equal(kvs, ref)


def test_lanes_of_one_sequence_are_a_prompt_chunk(tiny):
    """Consecutive positions of one sequence in one step (a chunk of a prompt):
    the same as feeding the tokens one step at a time, in whichever order the
    lanes are listed -- every lane's k and v are in the cache before any lane
    attends."""
    cfg, w, orc, _ = tiny
    prompt = synth.prompt_ids(7, 9, cfg.vocab)
    ref = _cache(cfg, 1)
    want = [orc.step(ref[0], int(prompt[p]), p)[0] for p in range(9)]
    for order in (np.arange(9), np.array([8, 0, 7, 1, 6, 2, 5, 3, 4])):
        kvs = _cache(cfg, 1)
        nxt, _ = orc.lanes(kvs, prompt[order], order, np.zeros(9, np.int32))
        np.testing.assert_array_equal(nxt, np.array(want)[order])
        np.testing.assert_array_equal(kvs, ref)


def test_lanes_mix_and_bad_lanes(tiny):
    cfg, w, orc, _ = tiny
    kvs = _cache(cfg, 2)
    # one lane alone is the single-token step
    ref = _cache(cfg, 2)
    nxt, _ = orc.lanes(kvs, [5], [0], [1])
    assert nxt[0] == orc.step(ref[1], 5, 0, want_logits=False)[0]
    np.testing.assert_array_equal(kvs, ref)
    for bad in (([5], [cfg.max_pos], [0]), ([5], [0], [2]), ([cfg.vocab], [0], [0]), ([5], [-1], [0])):
        with pytest.raises(ValueError):
            orc.lanes(kvs, *bad)
