"""NumPy-style float reference of the ternary decode step (test code only).

Written independently of the oracle's C source, in the style of the
cpp20gemma README's "Tests" section: weights are dequantised (trit * scale)
and the linear layers are float64 matrix products, the same as a NumPy
reference would do.  Because trit * scale * int8 terms are exact in float64,
rounding the product once to fp32 gives the same value as the integer path
followed by the fp32 epilogue, so the two can agree token for token.

The fp32 operations that feed an activation quantiser follow the same stated
definitions as the oracle (pairwise sums, the Cody-Waite exponential), here
in vectorised NumPy; fused multiply-adds are evaluated in float64 and rounded
to fp32 (exact for the operand ranges involved).
"""
from __future__ import annotations

import math

import numpy as np

f32 = np.float32


def pairwise_sum(a: np.ndarray, axis: int = -1) -> np.ndarray:
    """Balanced pairwise sum along `axis`, zero-padded to a power of two, in fp32."""
    a = np.moveaxis(np.asarray(a, f32), axis, -1)
    n = a.shape[-1]
    P = 1
    while P < n:
        P *= 2
    if P != n:
        pad = np.zeros(a.shape[:-1] + (P - n,), f32)
        a = np.concatenate([a, pad], axis=-1)
    while a.shape[-1] > 1:
        a = (a[..., 0::2] + a[..., 1::2]).astype(f32)
    return a[..., 0]


def _fma(a, b, c):
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(f32)


def exp32(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, f32)
    n = np.rint((x * f32(1.44269502162933349609375)).astype(f32)).astype(f32)
    r = _fma(-n, f32(0.693145751953125), x)
    r = _fma(-n, f32(1.4286068203094172321e-06), r)
    p = np.full_like(r, f32(1.0) / f32(5040.0))
    for c in (f32(1) / f32(720), f32(1) / f32(120), f32(1) / f32(24), f32(1) / f32(6), f32(0.5), f32(1), f32(1)):
        p = _fma(p, r, c)
    e = np.clip(n, -150, 128).astype(np.int64)
    with np.errstate(over="ignore"):
        # exact scaling by 2^e: float64 holds p * 2^e exactly, one rounding to fp32
        out = (p.astype(np.float64) * np.power(2.0, e.astype(np.float64))).astype(f32)
    out = np.where(x > f32(88.72283935546875), f32(np.inf), out)
    out = np.where(x < f32(-103.972084045410156), f32(0.0), out)
    return out.astype(f32)


def gelu32(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, f32)
    x3 = ((x * x).astype(f32) * x).astype(f32)
    inner = (x + (f32(0.044715) * x3).astype(f32)).astype(f32)
    z = (f32(0.7978845608028654) * inner).astype(f32)
    e = exp32((f32(2.0) * z).astype(f32))
    with np.errstate(over="ignore", invalid="ignore"):
        t = (f32(1.0) - (f32(2.0) / (e + f32(1.0)).astype(f32)).astype(f32)).astype(f32)
    return ((f32(0.5) * x).astype(f32) * (f32(1.0) + t).astype(f32)).astype(f32)


def rmsnorm32(x, g, eps):
    x = np.asarray(x, f32)
    ss = pairwise_sum((x * x).astype(f32))
    ss = (ss / f32(x.size)).astype(f32)
    ss = (ss + f32(eps)).astype(f32)
    r = (f32(1.0) / np.sqrt(ss).astype(f32)).astype(f32)
    return (np.asarray(g, f32) * (r * x).astype(f32)).astype(f32)


def quant32(x):
    x = np.asarray(x, f32)
    s = max(np.abs(x).max(), f32(1e-9))
    s = f32(s / f32(127.0))
    q = np.clip(np.rint((x / s).astype(f32)), -127, 127).astype(np.int8)
    return q, s


class NumpyDecoder:
    """Dequantised-weight float reference of the decode step."""

    def __init__(self, cfg, weights):
        self.cfg = cfg
        self.wdeq = []  # per layer: dict name -> float64 [N][K] = trit * scale
        names = [m[0] for m in cfg.matrices()]
        for l in range(cfg.n_layers):
            d = {}
            for j, name in enumerate(names):
                d[name] = weights["layers"][l][name].astype(np.float64) * float(weights["scales"][l, j])
            self.wdeq.append(d)
        self.g_attn, self.g_ffn, self.g_final = weights["g_attn"], weights["g_ffn"], weights["g_final"]
        self.emb = (weights["emb"].astype(np.uint32) << 16).view(np.float32)
        half = cfg.head_dim // 2
        self.theta = [cfg.rope_base ** (-(2 * i) / cfg.head_dim) for i in range(half)]

    def _lin(self, W, x):
        q, s = quant32(x)
        return ((W @ q.astype(np.float64)).astype(f32) * s).astype(f32)

    def _rope(self, v, n_heads, pos):
        hd = self.cfg.head_dim
        half = hd // 2
        c = np.array([math.cos(pos * t) for t in self.theta], np.float64).astype(f32)
        s = np.array([math.sin(pos * t) for t in self.theta], np.float64).astype(f32)
        v = v.reshape(n_heads, hd).copy()
        a, b = v[:, :half].copy(), v[:, half:].copy()
        v[:, :half] = ((a * c).astype(f32) - (b * s).astype(f32)).astype(f32)
        v[:, half:] = ((a * s).astype(f32) + (b * c).astype(f32)).astype(f32)
        return v.ravel()

    def _attention(self, q, kc, vc, pos):
        cfg = self.cfg
        H, hd, nkv = cfg.n_heads, cfg.head_dim, cfg.n_kv_heads
        C = 32
        T = pos + 1
        nc = (T + C - 1) // C
        out = np.empty((H, hd), f32)
        div = np.sqrt(f32(hd)).astype(f32)
        for h in range(H):
            kvh = h // (H // nkv)
            K = kc[:T, kvh * hd:(kvh + 1) * hd]
            V = vc[:T, kvh * hd:(kvh + 1) * hd]
            s = (pairwise_sum((K * q[h * hd:(h + 1) * hd]).astype(f32), axis=1) / div).astype(f32)
            sp = np.full(nc * C, -np.inf, f32)
            sp[:T] = s
            sp = sp.reshape(nc, C)
            m_c = sp.max(axis=1)
            e = np.zeros((nc, C), f32)
            valid = np.arange(nc * C).reshape(nc, C) < T
            e[valid] = exp32((sp - m_c[:, None])[valid])
            S_c = pairwise_sum(e, axis=1)
            Vp = np.zeros((nc * C, hd), f32)
            Vp[:T] = V
            Vp = Vp.reshape(nc, C, hd)
            U_c = pairwise_sum((e[:, :, None] * Vp).astype(f32), axis=1)  # [nc][hd]
            m = m_c.max()
            w = exp32((m_c - m).astype(f32))
            S = pairwise_sum((S_c * w).astype(f32))
            U = pairwise_sum((U_c * w[:, None]).astype(f32).T, axis=1)
            out[h] = (U / S).astype(f32)
        return out.ravel()

    def step(self, kv, token, pos):
        hn = self.hidden(kv, token, pos)
        logits = (self.emb.astype(np.float64) @ hn.astype(np.float64)).astype(f32)
        return int(np.argmax(logits)), logits

    def hidden(self, kv, token, pos):
        """The step up to the final norm (appends k and v at pos)."""
        cfg = self.cfg
        h = self.emb[token].astype(f32).copy()
        for l in range(cfg.n_layers):
            W = self.wdeq[l]
            xn = rmsnorm32(h, self.g_attn[l], cfg.eps)
            q = self._lin(W["wq"], xn)
            k = self._lin(W["wk"], xn)
            v = self._lin(W["wv"], xn)
            q = self._rope(q, cfg.n_heads, pos)
            k = self._rope(k, cfg.n_kv_heads, pos)
            kv[l, 0, pos] = k
            kv[l, 1, pos] = v
            att = self._attention(q, kv[l, 0], kv[l, 1], pos)
            h = (h + self._lin(W["wo"], att)).astype(f32)
            xn = rmsnorm32(h, self.g_ffn[l], cfg.eps)
            g = self._lin(W["wg"], xn)
            u = self._lin(W["wu"], xn)
            a = (gelu32(g) * u).astype(f32)
            h = (h + self._lin(W["wd"], a)).astype(f32)
        return rmsnorm32(h, self.g_final, cfg.eps)

    def generate(self, kv, prompt, start_pos, n_steps):
        out = []
        token = int(prompt[0])
        for s in range(n_steps):
            nx, _ = self.step(kv, token, start_pos + s)
            out.append(nx)
            token = int(prompt[s + 1]) if s + 1 < len(prompt) else nx
        return np.array(out, np.int32)
