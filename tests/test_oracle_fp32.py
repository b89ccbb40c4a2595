"""Pins of the oracle's fp32 building blocks of the decode step (S9, S11, S12, S14).

References used: math.fsum and float64 numpy (error bounds), closed forms
(constant-vector RMSNorm, pos-0 attention, RoPE at pos 0), and structural
probes that fail on a plausible mistake (adjacent instead of half-split RoPE
pairs, wrong GQA head mapping, a sequential instead of pairwise sum).
"""
import math

import numpy as np
import pytest

import oracle
import synth

EPS32 = np.finfo(np.float32).eps


# ---------------------------------------------------------------- pairwise sum
def test_psum_tree_shape():
    # pairwise: (1e8 + 1) + (-1e8 + 1) = 1e8 - 1e8 = 0 in fp32; left-to-right gives 1
    a = np.array([1e8, 1, -1e8, 1], np.float32)
    assert oracle.psum(a) == 0.0
    # zero padding to the next power of two: [a, b, c] = (a + b) + (c + 0)
    a = np.array([1e8, -1e8, 3.0], np.float32)
    assert oracle.psum(a) == np.float32(3.0)
    assert oracle.psum(np.array([], np.float32)) == 0.0
    assert oracle.psum(np.array([2.5], np.float32)) == np.float32(2.5)


@pytest.mark.parametrize("n", [2, 7, 64, 1152, 6912])
def test_psum_error_bound(n):
    a = synth.normal_f32(20, n, (n,))
    exact = math.fsum(float(v) for v in a)
    bound = math.ceil(math.log2(n)) * EPS32 * float(np.abs(a).sum())
    assert abs(float(oracle.psum(a)) - exact) <= bound


# ---------------------------------------------------------------- exp / tanh / gelu
def test_exp_accuracy_dense_grid():
    x = np.concatenate([np.linspace(-87.0, 88.5, 200001, dtype=np.float32),
                        np.linspace(-1, 1, 20001, dtype=np.float32)])
    got = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 2.0


def test_exp_special_values():
    assert oracle.exp_f32([0.0])[0] == 1.0
    assert np.isinf(oracle.exp_f32([89.0])[0])
    assert oracle.exp_f32([-104.0])[0] == 0.0
    # subnormal range is rounded once: compare with float64 exp rounded to fp32
    x = np.linspace(-103.5, -87.5, 4001, dtype=np.float32)
    got = oracle.exp_f32(x)
    ref = np.exp(x.astype(np.float64)).astype(np.float32)
    assert np.max(np.abs(got.astype(np.float64) - ref.astype(np.float64))) <= 2 * 2.0 ** -149


def test_tanh_and_gelu_accuracy():
    z = np.linspace(-12, 12, 48001, dtype=np.float32)
    t = oracle.tanh_f32(z).astype(np.float64)
    assert np.max(np.abs(t - np.tanh(z.astype(np.float64)))) <= 3e-7
    x = np.linspace(-10, 10, 40001, dtype=np.float32)
    g = oracle.gelu_f32(x).astype(np.float64)
    xd = x.astype(np.float64)
    ref = 0.5 * xd * (1 + np.tanh(math.sqrt(2 / math.pi) * (xd + 0.044715 * xd ** 3)))
    assert np.max(np.abs(g - ref) / np.maximum(1.0, np.abs(ref))) <= 5e-7
    # closed points: gelu(0) = 0, identity far right, zero far left
    assert oracle.gelu_f32([0.0])[0] == 0.0
    assert oracle.gelu_f32([30.0])[0] == np.float32(30.0)
    assert oracle.gelu_f32([-30.0])[0] == 0.0


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("c", [0.001, 0.37, 3.0, 250.0])
def test_rmsnorm_constant_vector_closed_form(c):
    n, eps = 1152, 1e-6
    x = np.full(n, c, np.float32)
    o = oracle.rmsnorm(x, np.ones(n, np.float32), eps)
    ref = c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(o, ref, rtol=3 * EPS32)


def test_rmsnorm_vs_float64_and_gain():
    n, eps = 1152, 1e-6
    x = synth.normal_f32(21, 0, (n,), 0.0, 3.0)
    g = synth.normal_f32(21, 1, (n,), 1.0, 0.1)
    o = oracle.rmsnorm(x, g, eps)
    xd = x.astype(np.float64)
    ref = g * xd / np.sqrt(np.mean(xd * xd) + eps)
    np.testing.assert_allclose(o, ref, rtol=4 * EPS32, atol=0)
    # doubling x leaves the output (almost) unchanged; the gain multiplies elementwise
    np.testing.assert_allclose(oracle.rmsnorm(2 * x, g, 0.0), oracle.rmsnorm(x, g, 0.0), rtol=2 * EPS32)


# ---------------------------------------------------------------- RoPE
def test_rope_table_pos0_and_values():
    c, s = oracle.rope_table(8, 256, 10000.0)
    assert (c[0] == 1).all() and (s[0] == 0).all()
    i = np.arange(128)
    ang = 5 * 10000.0 ** (-2 * i / 256)
    np.testing.assert_allclose(c[5], np.cos(ang), rtol=0, atol=EPS32)
    np.testing.assert_allclose(s[5], np.sin(ang), rtol=0, atol=EPS32)


def test_rope_pairs_are_half_split_and_norm_preserving():
    hd = 16
    c, s = oracle.rope_table(4, hd, 10000.0)
    x = np.zeros(hd, np.float32)
    x[0] = 1.0
    y = oracle.rope_apply(x, 1, hd, c[3], s[3])
    nz = np.nonzero(y)[0].tolist()
    assert nz == [0, hd // 2]  # (i, i + d/2) pairing, not (i, i+1)
    assert math.isclose(math.atan2(y[hd // 2], y[0]), 3.0, rel_tol=1e-6)  # angle pos * base^0
    v = synth.normal_f32(22, 0, (4 * hd,))
    r = oracle.rope_apply(v, 4, hd, c[2], s[2])
    a = v.reshape(4, 2, hd // 2)
    b = r.reshape(4, 2, hd // 2)
    np.testing.assert_allclose(np.hypot(b[:, 0], b[:, 1]), np.hypot(a[:, 0], a[:, 1]), rtol=4 * EPS32)
    np.testing.assert_array_equal(oracle.rope_apply(v, 4, hd, c[0], s[0]), v)  # pos 0 is the identity


# ---------------------------------------------------------------- attention
def _attention_f64(q, kc, vc, pos, H, nkv, hd):
    out = np.empty((H, hd))
    for h in range(H):
        kvh = h // (H // nkv)
        k = kc[: pos + 1, kvh * hd:(kvh + 1) * hd].astype(np.float64)
        v = vc[: pos + 1, kvh * hd:(kvh + 1) * hd].astype(np.float64)
        sc = k @ q[h * hd:(h + 1) * hd].astype(np.float64) / math.sqrt(hd)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        out[h] = p @ v
    return out.ravel()


def test_attention_pos0_is_v0_exactly():
    H, nkv, hd = 4, 1, 256
    q = synth.normal_f32(23, 0, (H * hd,))
    kc = synth.normal_f32(23, 1, (4, nkv * hd))
    vc = synth.normal_f32(23, 2, (4, nkv * hd))
    out = oracle.attention(q, kc, vc, 0, H, nkv, hd)
    np.testing.assert_array_equal(out.reshape(H, hd), np.tile(vc[0], (H, 1)))


def test_attention_identical_keys_give_mean_of_v():
    H, nkv, hd, pos = 4, 1, 64, 40
    q = synth.normal_f32(24, 0, (H * hd,))
    kc = np.tile(synth.normal_f32(24, 1, (1, hd)), (pos + 1, 1))
    vc = synth.normal_f32(24, 2, (pos + 1, hd))
    out = oracle.attention(q, kc, vc, pos, H, nkv, hd).reshape(H, hd)
    np.testing.assert_allclose(out, np.tile(vc.astype(np.float64).mean(0), (H, 1)), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("pos", [1, 31, 32, 33, 100, 1087])
@pytest.mark.parametrize("H,nkv,hd", [(4, 1, 256), (4, 2, 16)])
def test_attention_vs_float64_softmax(pos, H, nkv, hd):
    q = synth.normal_f32(25, pos, (H * hd,), 0.0, 0.5)
    kc = synth.normal_f32(25, 1000 + pos, (pos + 1, nkv * hd))
    vc = synth.normal_f32(25, 2000 + pos, (pos + 1, nkv * hd))
    out = oracle.attention(q, kc, vc, pos, H, nkv, hd)
    ref = _attention_f64(q, kc, vc, pos, H, nkv, hd)
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-6 * np.abs(ref).max())
