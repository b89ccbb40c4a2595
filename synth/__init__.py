"""Seeded synthetic inputs, shared by the CUDA path's tests/bench and by the oracle.

Only random draws live here (splitmix64 + Box-Muller, see ``synth.c``); no
quantisation, packing or model arithmetic.  Every workload recipe below states
the shapes and distributions it draws; both sides of a parity test receive the
very same arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_synth.so`` (portable C, no ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, d = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            p = ctypes.c_void_p
            lib.synth_splitmix64_seq.argtypes = [u64, i64, p]
            lib.synth_normal_f32.argtypes = [u64, u64, i64, d, d, p]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, d, d, p]
            lib.synth_uniform_f32.argtypes = [u64, u64, i64, d, d, p]
            lib.synth_trits.argtypes = [u64, u64, i64, d, d, p]
            lib.synth_int_range.argtypes = [u64, u64, i64, i64, i64, p]
            for f in (lib.synth_splitmix64_seq, lib.synth_normal_f32, lib.synth_normal_bf16,
                      lib.synth_uniform_f32, lib.synth_trits, lib.synth_int_range):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- primitives
def splitmix64_seq(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _L().synth_splitmix64_seq(seed, n, _ptr(out))
    return out


def normal_f32(seed: int, stream: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _L().synth_normal_f32(seed, stream, out.size, mean, std, _ptr(out))
    return out


def normal_bf16(seed: int, stream: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std) draws, rounded to nearest even."""
    out = np.empty(shape, np.uint16)
    _L().synth_normal_bf16(seed, stream, out.size, mean, std, _ptr(out))
    return out


def uniform_f32(seed: int, stream: int, shape, lo=0.0, hi=1.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _L().synth_uniform_f32(seed, stream, out.size, lo, hi, _ptr(out))
    return out


def trits(seed: int, stream: int, shape, p_neg=0.3, p_zero=0.4) -> np.ndarray:
    out = np.empty(shape, np.int8)
    _L().synth_trits(seed, stream, out.size, p_neg, p_zero, _ptr(out))
    return out


def int_range(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _L().synth_int_range(seed, stream, n, lo, hi, _ptr(out))
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- workloads
# Streams are fixed small integers so that every array of a workload is
# independent of every other and of its size.

def w8_gemv(seed: int, M: int, K: int, N: int):
    """W8 GEMV/GEMM inputs: fp32 weights ~N(0, 0.02) [N][K], fp32 x ~N(0,1) [M][K]."""
    return {"w": normal_f32(seed, 1, (N, K), 0.0, 0.02), "x": normal_f32(seed, 2, (M, K), 0.0, 1.0)}


def t158_gemv(seed: int, M: int, K: int, N: int):
    """T158 inputs: trits iid P(-1)=P(+1)=0.3, P(0)=0.4 [N][K]; matrix scale U(0.01, 0.05);
    fp32 activations ~N(0,1) [M][K] (to be absmax-quantised per row)."""
    return {
        "trits": trits(seed, 1, (N, K), 0.3, 0.4),
        "w_scale": float(uniform_f32(seed, 3, (1,), 0.01, 0.05)[0]),
        "x": normal_f32(seed, 2, (M, K), 0.0, 1.0),
    }


def sketch_head(seed: int, V: int, D: int):
    """Output-layer inputs: bf16 table ~N(0, 0.02) [V][D] and a per-dimension size
    s_d ~ U(0.5, 2) (the fixed scale of each hidden dimension, as a final norm
    gain gives it); hidden states come from ``sketch_x``."""
    return {
        "emb": normal_bf16(seed, 1, (V, D), 0.0, 0.02),
        "scale": uniform_f32(seed, 3, (D,), 0.5, 2.0),
    }


def sketch_x(seed: int, token: int, scale: np.ndarray) -> np.ndarray:
    """A final hidden state: x_d = N(0,1) * s_d, one draw per token."""
    return (normal_f32(seed, 100 + token, (scale.size,), 0.0, 1.0) * scale).astype(np.float32)


class DecoderConfig:
    """Shape of a Gemma-3-1B-like ternary decoder."""

    def __init__(self, n_layers, dim, n_heads, n_kv_heads, head_dim, ffn, vocab, max_pos,
                 eps=1e-6, rope_base=10000.0):
        self.n_layers, self.dim, self.n_heads, self.n_kv_heads = n_layers, dim, n_heads, n_kv_heads
        self.head_dim, self.ffn, self.vocab, self.max_pos = head_dim, ffn, vocab, max_pos
        self.eps, self.rope_base = eps, rope_base

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    def matrices(self):
        """(name, rows N, cols K) of the seven ternary matrices of one block."""
        d, q, kv, f = self.dim, self.q_dim, self.kv_dim, self.ffn
        return [("wq", q, d), ("wk", kv, d), ("wv", kv, d), ("wo", d, q),
                ("wg", f, d), ("wu", f, d), ("wd", d, f)]

    def as_dict(self):
        return dict(n_layers=self.n_layers, dim=self.dim, n_heads=self.n_heads,
                    n_kv_heads=self.n_kv_heads, head_dim=self.head_dim, ffn=self.ffn,
                    vocab=self.vocab, max_pos=self.max_pos, eps=self.eps, rope_base=self.rope_base)


GEMMA3_1B = dict(n_layers=26, dim=1152, n_heads=4, n_kv_heads=1, head_dim=256, ffn=6912,
                 vocab=262144, eps=1e-6, rope_base=10000.0)
TINY = dict(n_layers=2, dim=64, n_heads=4, n_kv_heads=1, head_dim=16, ffn=160, vocab=512,
            eps=1e-6, rope_base=10000.0)


def decoder_weights(cfg: DecoderConfig, seed: int, emb_std: float = 0.02):
    """Random-init ternary decoder.

    * trits of every matrix iid P(-1)=P(+1)=0.3, P(0)=0.4, one scale per matrix U(0.01, 0.05)
    * RMSNorm gains 1 + 0.1 N(0,1)
    * tied bf16 embedding / lm_head table ~N(0, emb_std), [vocab][dim] (0.02 by default)
    Returns a dict with per-layer lists of trit matrices ``layers[l][name]`` (int8 [N][K]),
    ``scales`` float32 [L][7] (matrix order of ``cfg.matrices()``), ``g_attn``/``g_ffn``
    float32 [L][dim], ``g_final`` [dim], ``emb`` uint16 bf16 bits [vocab][dim].
    """
    L = cfg.n_layers
    layers = []
    for l in range(L):
        mats = {}
        for j, (name, n, k) in enumerate(cfg.matrices()):
            mats[name] = trits(seed, 1000 + 16 * l + j, (n, k), 0.3, 0.4)
        layers.append(mats)
    return {
        "layers": layers,
        "scales": uniform_f32(seed, 7, (L, 7), 0.01, 0.05),
        "g_attn": normal_f32(seed, 8, (L, cfg.dim), 1.0, 0.1),
        "g_ffn": normal_f32(seed, 9, (L, cfg.dim), 1.0, 0.1),
        "g_final": normal_f32(seed, 10, (cfg.dim,), 1.0, 0.1),
        "emb": normal_bf16(seed, 11, (cfg.vocab, cfg.dim), 0.0, emb_std),
    }


def kv_fill(cfg: DecoderConfig, seed: int, n_pos: int) -> np.ndarray:
    """fp32 KV cache [L][2][max_pos][kv_dim] whose positions < n_pos hold N(0,1) draws, rest 0."""
    kv = np.zeros((cfg.n_layers, 2, cfg.max_pos, cfg.kv_dim), np.float32)
    if n_pos > 0:
        kv[:, :, :n_pos, :] = normal_f32(seed, 12, (cfg.n_layers, 2, n_pos, cfg.kv_dim), 0.0, 1.0)
    return kv


def prompt_ids(seed: int, n: int, vocab: int) -> np.ndarray:
    """Prompt token ids: the plain splitmix64 sequence started at ``seed``, mod vocab."""
    return (splitmix64_seq(seed, n) % np.uint64(vocab)).astype(np.int32)
