"""An unblocked float64 reading of the ternary decode step (test code only).

The forward pass of llama2.c "The forward pass -- one token, one position"
(Steps 0-6) with the block structure of the cpp20gemma README ("Architecture
& implementation"), every linear layer a ternary matrix on int8-quantised
inputs ("Gemma 3 1B at 114 tokens per second on a laptop CPU", "Step 2"),
written the plainest way: every value is float64, every sum is NumPy's,
softmax is np.exp over all positions at once with the maximum subtracted,
GELU uses np.tanh, RoPE uses math.cos/sin.  No chunks, no pairwise trees, no
fp32 rounding order.  The int8 quantiser is the same rule (step = max|x| /
127 with a 1e-9 floor, round half to even, clip +-127), evaluated in
float64, so a code can differ from the fp32 oracle's where a value sits
within rounding of a half-integer step.  The oracle is checked against this
reading with a tolerance, not bit for bit.
"""
from __future__ import annotations

import math

import numpy as np

f64 = np.float64


def quant64(x):
    s = max(float(np.abs(x).max()), 1e-9) / 127.0
    return np.clip(np.rint(x / s), -127, 127), s


def rmsnorm64(x, g, eps):
    return np.asarray(g, f64) * (x / math.sqrt(float(np.mean(x * x)) + eps))


def gelu64(x):
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


class PlainDecoder:
    def __init__(self, cfg, weights):
        self.cfg = cfg
        self.w = weights
        self.names = [m[0] for m in cfg.matrices()]
        self.emb_bits = np.ascontiguousarray(weights["emb"], np.uint16)

    def emb_rows(self, lo, hi):
        return (self.emb_bits[lo:hi].astype(np.uint32) << 16).view(np.float32).astype(f64)

    def _lin(self, l, name, x):
        j = self.names.index(name)
        q, s = quant64(x)
        t = self.w["layers"][l][name]
        return (t.astype(f64) @ q) * float(self.w["scales"][l, j]) * s

    def _rope(self, v, n_heads, pos):
        hd = self.cfg.head_dim
        half = hd // 2
        th = np.array([self.cfg.rope_base ** (-(2 * i) / hd) for i in range(half)], f64) * pos
        c, s = np.cos(th), np.sin(th)
        v = v.reshape(n_heads, hd).copy()
        a, b = v[:, :half].copy(), v[:, half:].copy()
        v[:, :half] = a * c - b * s
        v[:, half:] = a * s + b * c
        return v.ravel()

    def _attention(self, q, kc, vc, pos):
        cfg = self.cfg
        H, hd, nkv = cfg.n_heads, cfg.head_dim, cfg.n_kv_heads
        out = np.empty((H, hd), f64)
        for h in range(H):
            kvh = h // (H // nkv)
            K = kc[: pos + 1, kvh * hd:(kvh + 1) * hd]
            V = vc[: pos + 1, kvh * hd:(kvh + 1) * hd]
            sc = K @ q[h * hd:(h + 1) * hd] / math.sqrt(hd)
            p = np.exp(sc - sc.max())
            out[h] = (p / p.sum()) @ V
        return out.ravel()

    def new_cache(self):
        c = self.cfg
        return np.zeros((c.n_layers, 2, c.max_pos, c.kv_dim), f64)

    def hidden(self, kv, token, pos):
        """Appends k and v at pos to kv (float64) and returns the final-normed hidden state."""
        cfg, w = self.cfg, self.w
        h = self.emb_rows(token, token + 1)[0]
        for l in range(cfg.n_layers):
            xn = rmsnorm64(h, w["g_attn"][l], cfg.eps)
            q = self._rope(self._lin(l, "wq", xn), cfg.n_heads, pos)
            kv[l, 0, pos] = self._rope(self._lin(l, "wk", xn), cfg.n_kv_heads, pos)
            kv[l, 1, pos] = self._lin(l, "wv", xn)
            h = h + self._lin(l, "wo", self._attention(q, kv[l, 0], kv[l, 1], pos))
            xn = rmsnorm64(h, w["g_ffn"][l], cfg.eps)
            a = gelu64(self._lin(l, "wg", xn)) * self._lin(l, "wu", xn)
            h = h + self._lin(l, "wd", a)
        return rmsnorm64(h, w["g_final"], cfg.eps)

    def logits(self, x, rows=16384):
        V = self.cfg.vocab
        out = np.empty(V, f64)
        for lo in range(0, V, rows):
            hi = min(V, lo + rows)
            out[lo:hi] = self.emb_rows(lo, hi) @ x
        return out

    def step(self, kv, token, pos):
        lg = self.logits(self.hidden(kv, token, pos))
        return int(np.argmax(lg)), lg
