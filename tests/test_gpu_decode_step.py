"""GPU parity of the composed decode step (S8-S16) against the oracle.

* tiny decoder: 79 forwards (16-token prompt + 64 greedy tokens), every
  argmax equal, logits within max-abs-rel 2e-3, KV cache bit-exact;
* Gemma-3-1B-shaped decoder (26 blocks, hidden 1152, 4/1 heads of 256, GeGLU
  6912, vocab 262144, seed 4): the same 16 + 64 greedy run from an empty cache,
  and steps on a cache filled to position 1024 (the throughput state);
* the status word reports an out-of-range token;
* the decode step with the sketch head as its output layer: tokens equal to
  the oracle's step cut at the final norm plus the oracle's sketch head, KV
  cache bit-exact (tiny decoder, and four steps of the Gemma-shaped one at
  position 1024).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import device, host, max_abs_rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def _pair(cfg, seed, dev, emb_std=0.02):
    from weight_streaming_gemv_gb300.decoder import T158Decoder

    w = synth.decoder_weights(cfg, seed=seed, emb_std=emb_std)
    return T158Decoder(cfg, w, device=dev), oracle.Decoder(cfg, w)


def _run_and_compare(gpu, orc, kv_o, prompt, start_pos, n_steps, logit_checks=None):
    import torch

    token = int(prompt[0])
    gpu.token.fill_(token)
    ids_g, ids_o = [], []
    for s in range(n_steps):
        pos = start_pos + s
        want = logit_checks is None or s in logit_checks
        nx_o, lg_o = orc.step(kv_o, token, pos, want_logits=True)
        gpu.step(pos, logits=want)
        torch.cuda.synchronize()
        nx_g = int(gpu.token.item())
        if want:
            err = max_abs_rel(gpu.logits.cpu().numpy(), lg_o)
            assert err <= 2e-3, f"step {s} (pos {pos}): logits max-abs-rel {err}"
        if nx_g != nx_o:
            top = np.sort(lg_o)[-2:]
            raise AssertionError(f"step {s} (pos {pos}): token {nx_g} != oracle {nx_o}; oracle top-2 gap {top[1]-top[0]}")
        ids_g.append(nx_g)
        ids_o.append(nx_o)
        token = int(prompt[s + 1]) if s + 1 < len(prompt) else nx_o
        gpu.token.fill_(token)
    gpu.check_status()
    return np.array(ids_g), np.array(ids_o)


def test_tiny_decoder_79_steps(dev):
    cfg = synth.DecoderConfig(max_pos=96, **synth.TINY)
    for emb_std in (0.02, 0.002):
        gpu, orc = _pair(cfg, 5, dev, emb_std)
        kv_o = orc.new_cache()
        prompt = synth.prompt_ids(5, 16, cfg.vocab)
        _run_and_compare(gpu, orc, kv_o, prompt, 0, 79)
        np.testing.assert_array_equal(host(gpu.kv), kv_o)


@pytest.fixture(scope="module")
def gemma(dev):
    cfg = synth.DecoderConfig(max_pos=1152, **synth.GEMMA3_1B)
    return (cfg,) + _pair(cfg, 4, dev)


def test_gemma_shape_greedy_64_from_prompt(gemma):
    cfg, gpu, orc = gemma
    gpu.kv.zero_()
    kv_o = orc.new_cache()
    prompt = synth.prompt_ids(4, 16, cfg.vocab)
    ids, _ = _run_and_compare(gpu, orc, kv_o, prompt, 0, 16 + 64 - 1, logit_checks={0, 15, 40, 78})
    np.testing.assert_array_equal(host(gpu.kv)[:, :, :79], kv_o[:, :, :79])
    print("generated:", ids[15:].tolist())


def test_gemma_shape_steps_at_pos_1024(gemma):
    import torch

    cfg, gpu, orc = gemma
    kv0 = synth.kv_fill(cfg, 4, 1024)
    gpu.kv.copy_(torch.from_numpy(kv0))
    kv_o = kv0.copy()
    prompt = np.array([int(synth.prompt_ids(4, 1, cfg.vocab)[0])], np.int32)
    _run_and_compare(gpu, orc, kv_o, prompt, 1024, 4)
    np.testing.assert_array_equal(host(gpu.kv)[:, :, 1024:1028], kv_o[:, :, 1024:1028])


def _sketch_run(cfg, gpu, orc, kv_o, token, start_pos, n_steps, k, n_cand):
    """Steps of decode_step_t158_sketch against the oracle's step cut at the
    final norm followed by the oracle's sketch head (size order from the final
    norm gain, the GPU's c_E); tokens fed back; returns the tokens and how many
    agree with the exact output layer."""
    import torch

    perm = oracle.sketch_perm(host(gpu.g_final))
    cE = float(host(gpu.sk_ce)[0])
    gpu.token.fill_(token)
    ids, agree = [], 0
    for s in range(n_steps):
        pos = start_pos + s
        xn = orc.hidden(kv_o, token, pos)
        nx_o, cand_o, cl_o, _ = oracle.sketch_head(orc.emb, xn, perm=perm, k=k, n_cand=n_cand, cE=cE)
        gpu.step_sketch(pos)
        torch.cuda.synchronize()
        nx_g = int(gpu.token.item())
        if nx_g != nx_o:  # only a near-tie among the candidates' exact logits may differ
            tol = 1e-5 * float(np.abs(cl_o).max())
            near = set(cand_o[cl_o >= cl_o.max() - 2 * tol].tolist())
            assert nx_g in near, f"step {s} (pos {pos}): token {nx_g} != oracle {nx_o}"
        agree += int(nx_o == oracle.lm_head_argmax(orc.emb, xn)[0])
        ids.append(nx_g)
        token = nx_o
        gpu.token.fill_(token)
    gpu.check_sketch_status()
    return np.array(ids), agree


def test_tiny_decoder_sketch_head_steps(dev):
    cfg = synth.DecoderConfig(max_pos=96, **synth.TINY)
    gpu, orc = _pair(cfg, 5, dev)
    gpu.prepare_sketch(k=16, n_cand=48)
    kv_o = orc.new_cache()
    ids, _ = _sketch_run(cfg, gpu, orc, kv_o, 7, 0, 40, 16, 48)
    np.testing.assert_array_equal(host(gpu.kv)[:, :, :40], kv_o[:, :, :40])


def test_gemma_shape_sketch_head_steps_at_pos_1024(gemma):
    import torch

    cfg, gpu, orc = gemma
    gpu.prepare_sketch(k=32, n_cand=1024)
    kv0 = synth.kv_fill(cfg, 4, 1024)
    gpu.kv.copy_(torch.from_numpy(kv0))
    kv_o = kv0.copy()
    token = int(synth.prompt_ids(4, 1, cfg.vocab)[0])
    ids, agree = _sketch_run(cfg, gpu, orc, kv_o, token, 1024, 4, 32, 1024)
    np.testing.assert_array_equal(host(gpu.kv)[:, :, 1024:1028], kv_o[:, :, 1024:1028])
    print("sketch tokens:", ids.tolist(), "agree with the exact output layer:", agree, "of", len(ids))


def test_out_of_range_token_sets_status(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    cfg = synth.DecoderConfig(max_pos=8, **synth.TINY)
    gpu, _ = _pair(cfg, 5, dev)
    gpu.step(0, token=torch.tensor([cfg.vocab + 5], dtype=torch.int32, device=dev))
    with pytest.raises(qlin.QlinError) as e:
        gpu.check_status()
    assert e.value.status == 1
    gpu.check_status()  # the word was cleared


def test_decode_step_rejects_bad_arguments(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    cfg = synth.DecoderConfig(max_pos=8, **synth.TINY)
    gpu, _ = _pair(cfg, 5, dev)
    with pytest.raises(qlin.QlinError):
        gpu.step(8)  # pos == max_pos
    with pytest.raises(qlin.QlinError):
        qlin.decode_step_t158(gpu.model, gpu.kv, gpu.workspace, gpu.ws_bytes - 1, gpu.token, 0, None, gpu.token)


def test_bounded_wait_runs_out_and_the_next_step_recovers(dev):
    """Every wait of a CTA on another CTA's words is bounded.  With a 1 ms limit
    and the test hook that makes the CTA owning residual row 0 withhold its
    rows in layer 1,
    every other CTA's wait for them runs out: the status word reports
    QLIN_ERR_TIMEOUT and the kernel ends (nothing faults, the context stays
    usable).  With the hook off, the default limit back, a re-zeroed
    workspace and the step's KV rows rewritten by a rerun, the step matches
    the oracle again."""
    import time

    import torch
    from weight_streaming_gemv_gb300 import qlin

    cfg = synth.DecoderConfig(max_pos=16, **synth.TINY)
    gpu, orc = _pair(cfg, 5, dev)
    kv_o = orc.new_cache()
    token = 3
    nx_o, _ = orc.step(kv_o, token, 0)
    qlin.decode_step_t158_set_wait_limit(1_000_000)
    qlin.decode_step_t158_test_withhold(1)
    try:
        gpu.token.fill_(token)
        t0 = time.perf_counter()
        gpu.step(0, logits=False)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 10.0
        with pytest.raises(qlin.QlinError) as e:
            gpu.check_status()
        assert e.value.status == 5  # QLIN_ERR_TIMEOUT
    finally:
        qlin.decode_step_t158_test_withhold(-1)
        qlin.decode_step_t158_set_wait_limit(0)
    gpu.workspace.zero_()
    gpu.token.fill_(token)
    gpu.step(0)
    torch.cuda.synchronize()
    gpu.check_status()
    assert int(gpu.token.item()) == nx_o
    np.testing.assert_array_equal(host(gpu.kv)[:, :, 0], kv_o[:, :, 0])
