"""GPU parity of the decode-step building blocks (S8, S9, S11, S12, S14, S16).

Everything that feeds an activation quantiser (RMSNorm, RoPE, attention,
GeGLU) must equal the oracle bit for bit, because its fp32 order is part of
the definition.  lm_head logits are fp32 against the oracle's fp64 (max-abs-rel
1e-5) and the greedy token must match exactly.
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


def _t(shape, dtype, dev):
    import torch

    return torch.empty(shape, dtype=dtype, device=dev)


def test_embed_row_and_out_of_range(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    V, D = 1000, 1152
    emb = synth.normal_bf16(50, 0, (V, D), 0.0, 0.02)
    e = to_dev(emb, dev)
    h = _t((D,), torch.float32, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for tok in (0, 517, V - 1):
        qlin.qlin_embed_bf16(e, V, D, torch.tensor([tok], dtype=torch.int32, device=dev), h, st)
        np.testing.assert_array_equal(host(h), synth.bf16_to_f32(emb[tok]))
    assert host(st)[0] == 0
    qlin.qlin_embed_bf16(e, V, D, torch.tensor([V], dtype=torch.int32, device=dev), h, st)
    assert host(st)[0] == 1 and (host(h) == 0).all()


@pytest.mark.parametrize("n", [16, 64, 1000, 1152, 6912])
def test_rmsnorm_bit_exact(dev, n):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    M = 3
    x = synth.normal_f32(51, n, (M, n), 0.0, 3.0)
    g = synth.normal_f32(52, n, (n,), 1.0, 0.1)
    out = _t((M, n), torch.float32, dev)
    qlin.qlin_rmsnorm(to_dev(x, dev), to_dev(g, dev), out, M, n, 1e-6)
    got = host(out)
    for m in range(M):
        np.testing.assert_array_equal(got[m], oracle.rmsnorm(x[m], g, 1e-6))


@pytest.mark.parametrize("max_pos,hd", [(2048, 256), (64, 16)])
def test_rope_table_bit_exact(dev, max_pos, hd):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    c = _t((max_pos, hd // 2), torch.float32, dev)
    s = _t((max_pos, hd // 2), torch.float32, dev)
    qlin.t158_rope_table(c, s, max_pos, hd, 10000.0)
    co, so = oracle.rope_table(max_pos, hd, 10000.0)
    # cos/sin are computed in double on both sides and rounded to fp32 once
    assert int((host(c) != co).sum()) == 0 and int((host(s) != so).sum()) == 0


@pytest.mark.parametrize("pos,nh,nkv,hd", [(0, 4, 1, 256), (7, 4, 1, 256), (1087, 4, 1, 256), (5, 4, 2, 16)])
def test_rope_kv_append(dev, pos, nh, nkv, hd):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    max_pos = 1100
    co, so = oracle.rope_table(max_pos, hd, 10000.0)
    q = synth.normal_f32(53, pos, (nh * hd,))
    k = synth.normal_f32(54, pos, (nkv * hd,))
    v = synth.normal_f32(55, pos, (nkv * hd,))
    kc = torch.zeros((max_pos, nkv * hd), dtype=torch.float32, device=dev)
    vc = torch.zeros_like(kc)
    qd = to_dev(q, dev)
    qlin.qlin_rope_kv_append(qd, to_dev(k, dev), to_dev(v, dev), kc, vc, to_dev(co, dev), to_dev(so, dev), pos, nh,
                             nkv, hd)
    np.testing.assert_array_equal(host(qd), oracle.rope_apply(q, nh, hd, co[pos], so[pos]))
    np.testing.assert_array_equal(host(kc)[pos], oracle.rope_apply(k, nkv, hd, co[pos], so[pos]))
    np.testing.assert_array_equal(host(vc)[pos], v)
    assert (host(kc)[pos + 1:] == 0).all() and (host(kc)[:pos] == 0).all()


@pytest.mark.parametrize("pos", [0, 1, 31, 32, 33, 100, 1023, 1087])
@pytest.mark.parametrize("nh,nkv,hd", [(4, 1, 256), (4, 2, 16), (8, 2, 64)])
def test_attention_bit_exact(dev, pos, nh, nkv, hd):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    T = pos + 1
    q = synth.normal_f32(56, pos, (nh * hd,), 0.0, 0.5)
    kc = synth.normal_f32(57, pos, (T, nkv * hd))
    vc = synth.normal_f32(58, pos, (T, nkv * hd))
    ref = oracle.attention(q, kc, vc, pos, nh, nkv, hd)
    out = _t((nh * hd,), torch.float32, dev)
    wsb = qlin.qlin_attention_workspace_size(T, nh, hd)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_attention_decode(to_dev(q, dev), to_dev(kc, dev), to_dev(vc, dev), pos, nh, nkv, hd, out, ws, wsb)
    np.testing.assert_array_equal(host(out), ref)


def test_geglu_bit_exact(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    n = 6912
    g = np.concatenate([synth.normal_f32(59, 0, (n - 6,), 0.0, 2.0),
                        np.array([0.0, -0.0, 30.0, -30.0, 1e-30, -12.5], np.float32)])
    u = synth.normal_f32(60, 0, (n,), 0.0, 1.0)
    a = _t((n,), torch.float32, dev)
    qlin.qlin_geglu(to_dev(g, dev), to_dev(u, dev), a, n)
    ref = (oracle.gelu_f32(g) * u).astype(np.float32)
    np.testing.assert_array_equal(host(a), ref)


@pytest.mark.parametrize("V,D", [(262144, 1152), (512, 64), (1000, 8)])
def test_lm_head_argmax(dev, V, D):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    emb = synth.normal_bf16(61, V, (V, D), 0.0, 0.02)
    x = synth.normal_f32(62, V, (D,), 0.0, 1.0)
    nx_o, lg_o = oracle.lm_head_argmax(emb, x)
    lg = _t((V,), torch.float32, dev)
    nx = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_lm_head_workspace_size(V)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_lm_head_argmax(to_dev(emb, dev), to_dev(x, dev), V, D, lg, nx, ws, wsb)
    assert max_abs_rel(host(lg), lg_o) <= 1e-5
    assert int(host(nx)[0]) == nx_o


def test_lm_head_ties_pick_lowest_index(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    V, D = 4096, 64
    emb = np.zeros((V, D), np.uint16)
    emb[[100, 2000, 4000]] = synth.normal_bf16(63, 0, (1, D), 0.5, 0.0)  # three identical best rows
    x = np.ones(D, np.float32)
    lg = _t((V,), torch.float32, dev)
    nx = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_lm_head_workspace_size(V)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_lm_head_argmax(to_dev(emb, dev), to_dev(x, dev), V, D, None, nx, ws, wsb)
    assert int(host(nx)[0]) == 100 == oracle.lm_head_argmax(emb, x)[0]
