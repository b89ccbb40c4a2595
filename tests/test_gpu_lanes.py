"""GPU parity of the decode step over lanes ([citric] "Many users at once")
against the oracle's lane step: next tokens equal (or in a near tie of the
oracle's fp64 logits), logits within max-abs-rel 2e-3, every KV cache bit for
bit.  Lanes of separate sequences, a prompt chunk listed out of order, one
lane (CUDA-core linears) and 2 or more (tensor cores), attention shapes
(head_dim 64 and 128; 1, 2 and 8 query heads per KV head; two KV heads), the
Gemma-3-1B-shaped decoder at context 1024 with 16 users, and bad lanes.
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


def _pair(cfg, seed, dev):
    from weight_streaming_gemv_gb300.decoder import T158Decoder

    w = synth.decoder_weights(cfg, seed=seed)
    return T158Decoder(cfg, w, device=dev), oracle.Decoder(cfg, w)


def _lane_step(gpu, orc, kvs_o, tokens, positions, seqs, logit_check=True):
    import torch

    M = len(tokens)
    gpu.lane_tokens[:M].copy_(torch.as_tensor(np.int32(tokens)))
    gpu.lane_pos[:M].copy_(torch.as_tensor(np.int32(positions)))
    gpu.lane_seq[:M].copy_(torch.as_tensor(np.int32(seqs)))
    lg = torch.empty((M, gpu.cfg.vocab), dtype=torch.float32, device=gpu.emb.device) if logit_check else None
    gpu.step_lanes(M, logits=lg)
    nx_o, lg_o = orc.lanes(kvs_o, tokens, positions, seqs, want_logits=True)
    gpu.check_lanes_status()
    nx_g = host(gpu.lane_next)[:M]
    # The lanes' hidden states are the oracle's bit for bit (the KV checks below);
    # only the output layer's fp32 accumulation differs from the oracle's fp64
    # sums, by about 1e-6 of the largest logit.  A token may differ only in a
    # tie that close: the runner-up within 2e-5 of the largest |logit|, and the
    # GPU's token must be that runner-up.
    for i in range(M):
        if nx_g[i] != nx_o[i]:
            tol = 2e-5 * np.abs(lg_o[i]).max()
            assert lg_o[i][nx_o[i]] - lg_o[i][nx_g[i]] <= tol, f"lane {i}: {nx_g[i]} != {nx_o[i]}"
    if logit_check:
        for i in range(M):
            assert max_abs_rel(host(lg)[i], lg_o[i]) <= 2e-3
    return nx_o


def test_tiny_lanes_batches_and_prompt_chunks(dev):
    cfg = synth.DecoderConfig(max_pos=96, **synth.TINY)
    gpu, orc = _pair(cfg, 5, dev)
    gpu.prepare_lanes(n_seqs=4, max_lanes=12)
    kvs_o = np.zeros((4, cfg.n_layers, 2, cfg.max_pos, cfg.kv_dim), np.float32)
    prompt = synth.prompt_ids(8, 12, cfg.vocab)
    # a prompt chunk of 9 tokens for sequence 2, listed out of order (9 lanes: tensor-core linears)
    order = np.array([8, 0, 7, 1, 6, 2, 5, 3, 4])
    _lane_step(gpu, orc, kvs_o, prompt[order], order, [2] * 9)
    # single tokens for sequences 0, 1 (2 lanes) and 3 (1 lane): CUDA-core linears at two tokens and one
    _lane_step(gpu, orc, kvs_o, [3, 4], [0, 0], [0, 1])
    _lane_step(gpu, orc, kvs_o, [5], [0], [3])
    # a mixed step: sequence 2 continues at 9 and 10, the others at 1, plus a new
    # sequence-3 chunk: 12 lanes
    _lane_step(gpu, orc, kvs_o, [11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22],
               [9, 10, 1, 1, 1, 2, 3, 4, 5, 6, 7, 8], [2, 2, 0, 1, 3, 3, 3, 3, 3, 3, 3, 3])
    # greedy continuation of four users for a few steps, tokens fed back (4 lanes: tensor-core linears)
    toks = [30, 31, 32, 33]
    for s in range(4):
        nx = _lane_step(gpu, orc, kvs_o, toks, [2 + s, 2 + s, 11 + s, 9 + s], [0, 1, 2, 3], logit_check=(s == 3))
        toks = [int(t) for t in nx]
    np.testing.assert_array_equal(host(gpu.kv_lanes), kvs_o)


@pytest.mark.parametrize("shape", [
    # 8 query heads per KV head, head_dim 64
    dict(n_layers=2, dim=128, n_heads=8, n_kv_heads=1, head_dim=64, ffn=192, vocab=512, eps=1e-6, rope_base=10000.0),
    # 2 KV heads (rows of a chunk are not contiguous: one copy per row), 2 query heads each, head_dim 128
    dict(n_layers=2, dim=128, n_heads=4, n_kv_heads=2, head_dim=128, ffn=160, vocab=512, eps=1e-6, rope_base=10000.0),
    # one query head per KV head
    dict(n_layers=1, dim=64, n_heads=2, n_kv_heads=2, head_dim=64, ffn=96, vocab=300, eps=1e-6, rope_base=10000.0),
])
def test_lanes_attention_shapes(dev, shape):
    # the persistent attention kernel's other head widths and groupings, a prompt
    # chunk across two 32-position chunks, lanes of three sequences at mixed positions
    cfg = synth.DecoderConfig(max_pos=100, **shape)
    gpu, orc = _pair(cfg, 6, dev)
    gpu.prepare_lanes(n_seqs=3, max_lanes=40)
    kvs_o = np.zeros((3, cfg.n_layers, 2, cfg.max_pos, cfg.kv_dim), np.float32)
    prompt = synth.prompt_ids(10, 40, cfg.vocab)
    _lane_step(gpu, orc, kvs_o, prompt[:37], np.arange(37), [0] * 37)
    _lane_step(gpu, orc, kvs_o, prompt[37:40], [37, 0, 0], [0, 1, 2])
    toks = [5, 6, 7]
    for s in range(3):
        nx = _lane_step(gpu, orc, kvs_o, toks, [38 + s, 1 + s, 1 + s], [0, 1, 2], logit_check=(s == 2))
        toks = [int(t) for t in nx]
    np.testing.assert_array_equal(host(gpu.kv_lanes), kvs_o)


def test_gemma_shape_16_users_at_1024(dev):
    import torch

    cfg = synth.DecoderConfig(max_pos=1089, **synth.GEMMA3_1B)
    gpu, orc = _pair(cfg, 4, dev)
    U = 16
    gpu.prepare_lanes(n_seqs=U, max_lanes=U)
    kv0 = synth.kv_fill(cfg, 4, 1024)
    for s in range(U):
        gpu.kv_lanes[s].copy_(torch.from_numpy(kv0))
    kvs_o = np.ascontiguousarray(np.broadcast_to(kv0, (U,) + kv0.shape))
    tokens = synth.prompt_ids(9, U, cfg.vocab)
    nx = _lane_step(gpu, orc, kvs_o, tokens, [1024] * U, np.arange(U))
    nx = _lane_step(gpu, orc, kvs_o, nx, [1025] * U, np.arange(U), logit_check=False)
    got = host(gpu.kv_lanes)
    np.testing.assert_array_equal(got[:, :, :, 1024:1026], kvs_o[:, :, :, 1024:1026])


def test_bad_lanes_set_status(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    cfg = synth.DecoderConfig(max_pos=32, **synth.TINY)
    gpu, _ = _pair(cfg, 5, dev)
    gpu.prepare_lanes(n_seqs=2, max_lanes=4)
    for tok, pos, seq in ((cfg.vocab, 1, 1), (1, cfg.max_pos, 1), (1, 1, 2), (1, -1, 1)):
        gpu.lane_tokens[:2].copy_(torch.tensor([1, tok], dtype=torch.int32))
        gpu.lane_pos[:2].copy_(torch.tensor([0, pos], dtype=torch.int32))
        gpu.lane_seq[:2].copy_(torch.tensor([0, seq], dtype=torch.int32))
        before = host(gpu.kv_lanes).copy()
        gpu.step_lanes(2)
        with pytest.raises(qlin.QlinError):
            gpu.check_lanes_status()
        after = host(gpu.kv_lanes)
        after[0, :, :, 0] = before[0, :, :, 0]  # lane 0's own row
        if tok == cfg.vocab:
            after[1, :, :, 1] = before[1, :, :, 1]  # a bad token still has a slot: its row comes from zeros
        np.testing.assert_array_equal(after, before)  # the bad lane wrote nothing anywhere else


@pytest.mark.parametrize("V,D,U", [(1000, 64, 1), (5000, 136, 5), (129, 8, 17), (3000, 1152, 70), (262144, 1152, 64)])
def test_lm_head_lanes_matches_oracle(dev, V, D, U):
    """The output layer for many lanes on the tensor cores: every lane's logits
    within max-abs-rel 1e-5 of the oracle's fp64 dot products, the greedy pick
    the oracle's unless its best two are closer than that."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    emb = synth.normal_bf16(70, V % 97, (V, D), 0.0, 0.02)
    x = synth.normal_f32(71, U, (U, D), 0.0, 1.0)
    lg = torch.empty((U, V), dtype=torch.float32, device=dev)
    nx = torch.full((U,), -1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_lm_head_lanes_workspace_size(V, D)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_lm_head_lanes(to_dev(emb, dev), to_dev(x, dev), V, D, U, lg, nx, ws, wsb)
    qlin.qlin_lm_head_lanes_status(ws)
    lg_h, nx_h = host(lg), host(nx)
    for u in range(U):
        nx_o, lg_o = oracle.lm_head_argmax(emb, x[u])
        assert max_abs_rel(lg_h[u], lg_o) <= 1e-5, u
        if nx_h[u] != nx_o:
            top = np.sort(lg_o)[-2:]
            assert top[1] - top[0] <= 2e-5 * np.abs(lg_o).max(), (u, nx_h[u], nx_o)
