"""ORACLE -- test infrastructure, not the product.

Thin ctypes access to ``oracle.c``, the plain CPU statement of the quantised
linear layers and of the ternary decode step.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
``--impl reference`` arm) may import this package.  It shares no code with
``weight_streaming_gemv_gb300``.

Every function is pinned by ``tests/test_oracle_*.py`` against hand-worked
vectors, closed forms, brute force, library routines or fp64 references.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EBADBYTE = 0, 1, 3
ATT_CHUNK = 32


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` (plain portable C, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-fno-fast-math", "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class OrModel(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int64), ("dim", ctypes.c_int64), ("n_heads", ctypes.c_int64),
        ("n_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64), ("ffn", ctypes.c_int64),
        ("vocab", ctypes.c_int64), ("max_pos", ctypes.c_int64),
        ("eps", ctypes.c_float), ("rope_base", ctypes.c_double),
        ("w", ctypes.c_void_p * 7), ("pitch", ctypes.c_int64 * 7),
        ("scales", ctypes.c_void_p), ("g_attn", ctypes.c_void_p), ("g_ffn", ctypes.c_void_p),
        ("g_final", ctypes.c_void_p), ("emb", ctypes.c_void_p),
    ]


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p, i64, f32, f64, i32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_double, ctypes.c_int32)
            sig = {
                "or_w8_quantize": ([p, i64, p, p], ctypes.c_int),
                "or_quant_i8": ([p, i64, i64, p, p], ctypes.c_int),
                "or_w8_linear": ([p, p, i64, f32, i64, i64, i64, p], ctypes.c_int),
                "or_w8g_quantize": ([p, i64, i64, i64, p, p], ctypes.c_int),
                "or_w8g_linear": ([p, p, i64, p, i64, i64, i64, i64, i64, p], ctypes.c_int),
                "or_t158_pack": ([p, i64, i64, p, i64], ctypes.c_int),
                "or_t158_unpack": ([p, i64, i64, i64, p], ctypes.c_int),
                "or_t158_pack_groups": ([p, i64, i64, p, i64], ctypes.c_int),
                "or_t158_unpack_groups": ([p, i64, i64, i64, p], ctypes.c_int),
                "or_t158_linear": ([p, p, p, i64, f32, i64, i64, i64, p, p], ctypes.c_int),
                "or_psum_f32": ([p, i64], f32),
                "or_exp_f32": ([f32], f32),
                "or_tanh_f32": ([f32], f32),
                "or_gelu_f32": ([f32], f32),
                "or_rmsnorm": ([p, p, i64, f32, p], None),
                "or_rope_table": ([i64, i64, f64, p, p], None),
                "or_rope_apply": ([p, i64, i64, p, p], None),
                "or_attention": ([p, p, p, i64, i64, i64, i64, p], None),
                "or_lm_head_argmax": ([p, p, i64, i64, p, p], None),
                "or_sketch_ce": ([p, i64, i64, p], ctypes.c_int),
                "or_sketch_perm": ([p, i64, p], ctypes.c_int),
                "or_sketch_head": ([p, i64, i64, p, i64, p, i64, i64, f32, p, p, p, p], ctypes.c_int),
                "or_decode_step": ([ctypes.POINTER(OrModel), p, i32, i64, p, p], ctypes.c_int),
                "or_decode_hidden": ([ctypes.POINTER(OrModel), p, i32, i64, p], ctypes.c_int),
                "or_decode_lanes": ([ctypes.POINTER(OrModel), p, i64, i64, p, p, p, p, p], ctypes.c_int),
                "or_decode_generate": ([ctypes.POINTER(OrModel), p, p, i64, i64, i64, p], ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != OK:
        raise ValueError(f"oracle {what} failed with status {rc}")


# ------------------------------------------------------------------ S1 / S3
def w8_quantize(w: np.ndarray):
    w = np.ascontiguousarray(w, np.float32)
    q = np.empty(w.shape, np.int8)
    s = ctypes.c_float()
    _check(_L().or_w8_quantize(_p(w), w.size, _p(q), ctypes.byref(s)), "w8_quantize")
    return q, np.float32(s.value)


def quant_i8(x: np.ndarray):
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    M, K = x.shape
    xq = np.empty((M, K), np.int8)
    xs = np.empty(M, np.float32)
    _check(_L().or_quant_i8(_p(x), M, K, _p(xq), _p(xs)), "quant_i8")
    return xq, xs


# ------------------------------------------------------------------ S5
def w8_linear(x: np.ndarray, q: np.ndarray, s: float, K: int | None = None):
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    q = np.ascontiguousarray(q, np.int8)
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    N, pitch = q.shape
    y = np.empty((M, N), np.float32)
    _check(_L().or_w8_linear(_p(x), _p(q), pitch, np.float32(s), M, N, K, _p(y)), "w8_linear")
    return y


# ------------------------------------------------------------------ W8 with group scales
def w8g_quantize(w: np.ndarray, G: int = 128):
    """int8 codes [N][K] and fp32 scales [N][ceil(K/G)] (one scale per G weights of a row)."""
    w = np.ascontiguousarray(np.atleast_2d(w), np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.int8)
    s = np.empty((N, (K + G - 1) // G), np.float32)
    _check(_L().or_w8g_quantize(_p(w), N, K, G, _p(q), _p(s)), "w8g_quantize")
    return q, s


def w8g_linear(x: np.ndarray, q: np.ndarray, scales: np.ndarray, G: int = 128, K: int | None = None):
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    q = np.ascontiguousarray(q, np.int8)
    scales = np.ascontiguousarray(scales, np.float32)
    M = x.shape[0]
    K = x.shape[1] if K is None else K
    N, pitch = q.shape
    y = np.empty((M, N), np.float32)
    _check(_L().or_w8g_linear(_p(x), _p(q), pitch, _p(scales), scales.shape[1], G, M, N, K, _p(y)), "w8g_linear")
    return y


# ------------------------------------------------------------------ S2
def packed_pitch(K: int) -> int:
    return (K + 4) // 5


def t158_pack(trits: np.ndarray, pitch: int | None = None):
    t = np.ascontiguousarray(trits, np.int8)
    N, K = t.shape
    pitch = packed_pitch(K) if pitch is None else pitch
    out = np.empty((N, pitch), np.uint8)
    _check(_L().or_t158_pack(_p(t), N, K, _p(out), pitch), "t158_pack")
    return out


def t158_pack_groups(trits: np.ndarray, gpitch: int | None = None):
    """Group-major packing for zero-group skipping: [ceil(K/4)][gpitch] bytes."""
    t = np.ascontiguousarray(trits, np.int8)
    N, K = t.shape
    gpitch = N if gpitch is None else gpitch
    out = np.empty(((K + 3) // 4, gpitch), np.uint8)
    _check(_L().or_t158_pack_groups(_p(t), N, K, _p(out), gpitch), "t158_pack_groups")
    return out


def t158_unpack_groups(packed_g: np.ndarray, N: int, K: int):
    pk = np.ascontiguousarray(packed_g, np.uint8)
    t = np.empty((N, K), np.int8)
    rc = _L().or_t158_unpack_groups(_p(pk), N, K, pk.shape[1], _p(t))
    if rc == EBADBYTE:
        raise ValueError("t158_unpack_groups: byte above 80")
    _check(rc, "t158_unpack_groups")
    return t


def t158_unpack(packed: np.ndarray, K: int):
    pk = np.ascontiguousarray(packed, np.uint8)
    N, pitch = pk.shape
    t = np.empty((N, K), np.int8)
    rc = _L().or_t158_unpack(_p(pk), N, K, pitch, _p(t))
    if rc == EBADBYTE:
        raise ValueError("packed byte above 242")
    _check(rc, "t158_unpack")
    return t


# ------------------------------------------------------------------ S4 / S6
def t158_linear(xq: np.ndarray, xs: np.ndarray, packed: np.ndarray, w_scale: float, K: int):
    xq = np.ascontiguousarray(np.atleast_2d(xq), np.int8)
    xs = np.ascontiguousarray(np.atleast_1d(xs), np.float32)
    pk = np.ascontiguousarray(packed, np.uint8)
    M = xq.shape[0]
    assert xq.shape[1] == K
    N, pitch = pk.shape
    acc = np.empty((M, N), np.int32)
    y = np.empty((M, N), np.float32)
    _check(_L().or_t158_linear(_p(xq), _p(xs), _p(pk), pitch, np.float32(w_scale), M, N, K, _p(acc), _p(y)),
           "t158_linear")
    return acc, y


# ------------------------------------------------------------------ fp32 building blocks
def psum(a: np.ndarray) -> np.float32:
    a = np.ascontiguousarray(a, np.float32)
    return np.float32(_L().or_psum_f32(_p(a), a.size))


def exp_f32(x) -> np.ndarray:
    f = _L().or_exp_f32
    return np.array([f(float(v)) for v in np.asarray(x, np.float32).ravel()], np.float32)


def tanh_f32(x) -> np.ndarray:
    f = _L().or_tanh_f32
    return np.array([f(float(v)) for v in np.asarray(x, np.float32).ravel()], np.float32)


def gelu_f32(x) -> np.ndarray:
    f = _L().or_gelu_f32
    return np.array([f(float(v)) for v in np.asarray(x, np.float32).ravel()], np.float32)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float):
    x = np.ascontiguousarray(x, np.float32)
    g = np.ascontiguousarray(g, np.float32)
    o = np.empty_like(x)
    _L().or_rmsnorm(_p(x), _p(g), x.size, np.float32(eps), _p(o))
    return o


def rope_table(n_pos: int, head_dim: int, base: float):
    c = np.empty((n_pos, head_dim // 2), np.float32)
    s = np.empty((n_pos, head_dim // 2), np.float32)
    _L().or_rope_table(n_pos, head_dim, base, _p(c), _p(s))
    return c, s


def rope_apply(x: np.ndarray, n_heads: int, head_dim: int, c: np.ndarray, s: np.ndarray):
    x = np.array(x, np.float32, copy=True, order="C")
    c = np.ascontiguousarray(c, np.float32)
    s = np.ascontiguousarray(s, np.float32)
    _L().or_rope_apply(_p(x), n_heads, head_dim, _p(c), _p(s))
    return x


def attention(q: np.ndarray, kc: np.ndarray, vc: np.ndarray, pos: int, n_heads: int, n_kv: int, head_dim: int):
    """q [n_heads*head_dim] (already rotated); kc/vc [>pos][n_kv*head_dim]."""
    q = np.ascontiguousarray(q, np.float32)
    kc = np.ascontiguousarray(kc, np.float32)
    vc = np.ascontiguousarray(vc, np.float32)
    out = np.empty(n_heads * head_dim, np.float32)
    _L().or_attention(_p(q), _p(kc), _p(vc), pos, n_heads, n_kv, head_dim, _p(out))
    return out


def lm_head_argmax(emb_bits: np.ndarray, x: np.ndarray):
    """fp64 logits of the bf16 table against x, rounded to fp32, and the first argmax."""
    e = np.ascontiguousarray(emb_bits, np.uint16)
    x = np.ascontiguousarray(x, np.float32)
    V, D = e.shape
    logits = np.empty(V, np.float32)
    nxt = ctypes.c_int32()
    _L().or_lm_head_argmax(_p(e), _p(x), V, D, _p(logits), ctypes.byref(nxt))
    return nxt.value, logits


# ------------------------------------------------------------------ sketch head
def sketch_ce(emb_bits: np.ndarray) -> float:
    """Mean |E| of a bf16 table (fp64 sum, rounded to fp32): the sketch's scale."""
    e = np.ascontiguousarray(emb_bits, np.uint16)
    V, D = e.shape
    out = ctypes.c_float()
    _check(_L().or_sketch_ce(_p(e), V, D, ctypes.byref(out)), "sketch_ce")
    return out.value


def sketch_perm(scale, D: int | None = None) -> np.ndarray:
    """Dimensions by size: largest |scale| first, ties to the lower index (identity if scale is None)."""
    if scale is None:
        sc, D = None, int(D)
    else:
        sc = np.ascontiguousarray(scale, np.float32).reshape(-1)
        D = sc.size
    perm = np.empty(D, np.int64)
    _check(_L().or_sketch_perm(None if sc is None else _p(sc), D, _p(perm)), "sketch_perm")
    return perm


def sketch_head(emb_bits: np.ndarray, x: np.ndarray, perm=None, B: int = 64, k: int = 32, n_cand: int = 1024,
                cE: float | None = None):
    """Candidates first, exact scores for them only.

    perm: the dimension order of the sign blocks (``sketch_perm``; identity if
    None); B: dimensions per block.  Returns ``(next, cand, cand_logits,
    approx)``: the chosen word, the n_cand candidate words in ascending order,
    their exact logits (fp64 dot rounded to fp32) and every word's approximate
    score.
    """
    e = np.ascontiguousarray(emb_bits, np.uint16)
    x = np.ascontiguousarray(x, np.float32).reshape(-1)
    V, D = e.shape
    perm = np.arange(D, dtype=np.int64) if perm is None else np.ascontiguousarray(perm, np.int64)
    if cE is None:
        cE = sketch_ce(e)
    approx = np.empty(V, np.float32)
    cand = np.empty(n_cand, np.int32)
    cl = np.empty(n_cand, np.float32)
    nxt = ctypes.c_int32()
    _check(_L().or_sketch_head(_p(e), V, D, _p(perm), B, _p(x), k, n_cand, cE, _p(approx), _p(cand), _p(cl),
                               ctypes.byref(nxt)), "sketch_head")
    return nxt.value, cand, cl, approx


# ------------------------------------------------------------------ decode step
MATRIX_ORDER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


class Decoder:
    """The oracle's copy of a ternary decoder: its own packing of the synthetic trits."""

    def __init__(self, cfg, weights):
        self.cfg = cfg
        L = cfg.n_layers
        dims = {name: (n, k) for name, n, k in cfg.matrices()}
        self.packed = []
        for name in MATRIX_ORDER:
            n, k = dims[name]
            pitch = packed_pitch(k)
            arr = np.empty((L, n, pitch), np.uint8)
            for l in range(L):
                arr[l] = t158_pack(weights["layers"][l][name])
            self.packed.append(arr)
        self.scales = np.ascontiguousarray(weights["scales"], np.float32)
        self.g_attn = np.ascontiguousarray(weights["g_attn"], np.float32)
        self.g_ffn = np.ascontiguousarray(weights["g_ffn"], np.float32)
        self.g_final = np.ascontiguousarray(weights["g_final"], np.float32)
        self.emb = np.ascontiguousarray(weights["emb"], np.uint16)
        m = OrModel()
        m.n_layers, m.dim, m.n_heads, m.n_kv_heads = L, cfg.dim, cfg.n_heads, cfg.n_kv_heads
        m.head_dim, m.ffn, m.vocab, m.max_pos = cfg.head_dim, cfg.ffn, cfg.vocab, cfg.max_pos
        m.eps, m.rope_base = cfg.eps, cfg.rope_base
        for j, arr in enumerate(self.packed):
            m.w[j] = arr.ctypes.data
            m.pitch[j] = arr.shape[2]
        m.scales, m.g_attn, m.g_ffn = self.scales.ctypes.data, self.g_attn.ctypes.data, self.g_ffn.ctypes.data
        m.g_final, m.emb = self.g_final.ctypes.data, self.emb.ctypes.data
        self.model = m

    def new_cache(self):
        c = self.cfg
        return np.zeros((c.n_layers, 2, c.max_pos, c.kv_dim), np.float32)

    def step(self, kv: np.ndarray, token: int, pos: int, want_logits: bool = True):
        assert kv.flags.c_contiguous and kv.dtype == np.float32
        logits = np.empty(self.cfg.vocab, np.float32) if want_logits else None
        nxt = ctypes.c_int32()
        rc = _L().or_decode_step(ctypes.byref(self.model), _p(kv), int(token), int(pos),
                                 _p(logits) if want_logits else None, ctypes.byref(nxt))
        _check(rc, "decode_step")
        return nxt.value, logits

    def hidden(self, kv: np.ndarray, token: int, pos: int):
        """The step up to the final norm: appends k and v at pos, returns the normalised hidden state."""
        assert kv.flags.c_contiguous and kv.dtype == np.float32
        xn = np.empty(self.cfg.dim, np.float32)
        _check(_L().or_decode_hidden(ctypes.byref(self.model), _p(kv), int(token), int(pos), _p(xn)), "decode_hidden")
        return xn

    def lanes(self, kvs: np.ndarray, tokens, positions, seqs, want_logits: bool = False):
        """One step over M lanes; kvs: [n_seqs][L][2][max_pos][kv_dim].  Returns (next [M], logits [M][V] or None)."""
        assert kvs.flags.c_contiguous and kvs.dtype == np.float32
        t = np.ascontiguousarray(tokens, np.int32)
        p = np.ascontiguousarray(positions, np.int32)
        sq = np.ascontiguousarray(seqs, np.int32)
        M = t.size
        nxt = np.empty(M, np.int32)
        lg = np.empty((M, self.cfg.vocab), np.float32) if want_logits else None
        _check(_L().or_decode_lanes(ctypes.byref(self.model), _p(kvs), kvs.shape[0], M, _p(t), _p(p), _p(sq),
                                    _p(lg) if want_logits else None, _p(nxt)), "decode_lanes")
        return nxt, lg

    def generate(self, kv: np.ndarray, prompt: np.ndarray, start_pos: int, n_steps: int):
        prompt = np.ascontiguousarray(prompt, np.int32)
        out = np.empty(n_steps, np.int32)
        rc = _L().or_decode_generate(ctypes.byref(self.model), _p(kv), _p(prompt), prompt.size,
                                     start_pos, n_steps, _p(out))
        _check(rc, "decode_generate")
        return out
