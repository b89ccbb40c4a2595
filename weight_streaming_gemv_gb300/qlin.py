"""ctypes binding of ``libqlin.so`` (the C ABI declared in ``include/qlin.h``).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the CUDA stream, statuses become exceptions.  Every step of
the computation runs in the library's CUDA kernels (or, for t158_pack /
t158_unpack, its host C code).  If the library is not built this module
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .build import LIB

T158_NMAT = 7
_lock = threading.Lock()
_lib = None


class QlinError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{fn} -> {status_name(status)}: {detail}")


class T158ModelC(ctypes.Structure):
    """Mirror of ``t158_model``."""

    _fields_ = [
        ("n_layers", ctypes.c_int32), ("dim", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("max_pos", ctypes.c_int32),
        ("eps", ctypes.c_float), ("reserved0", ctypes.c_float),
        ("w", ctypes.c_void_p * T158_NMAT), ("pitch", ctypes.c_int64 * T158_NMAT),
        ("scales", ctypes.c_void_p), ("g_attn", ctypes.c_void_p), ("g_ffn", ctypes.c_void_p),
        ("g_final", ctypes.c_void_p), ("emb", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p),
    ]


class T158SketchC(ctypes.Structure):
    """Mirror of ``t158_sketch``."""

    _fields_ = [
        ("emb_t", ctypes.c_void_p), ("signs", ctypes.c_void_p), ("perm", ctypes.c_void_p), ("c_e", ctypes.c_void_p),
        ("k", ctypes.c_int32), ("n_cand", ctypes.c_int32),
    ]


_P, _I, _I64, _F, _D, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                             ctypes.c_size_t)
_ST = ctypes.c_int
# name -> (argtypes, restype), in the order of include/qlin.h
SIGNATURES = {
    "qlin_status_str": ([_I], ctypes.c_char_p),
    "qlin_last_error": ([], ctypes.c_char_p),
    "qlin_version": ([], _I),
    "t158_pitch": ([_I64], _I64),
    "t158_pack": ([_P, _I64, _I64, _P, _I64], _ST),
    "t158_unpack": ([_P, _I64, _I64, _I64, _P], _ST),
    "qlin_w8_quantize": ([_P, _I64, _I64, _P, _I64, _P, _P], _ST),
    "qlin_quant_i8": ([_P, _P, _P, _I, _I, _P], _ST),
    "qlin_t158_i8": ([_P, _P, _P, _I64, _F, _P, _P, _I, _I, _I, _P], _ST),
    "qlin_t158_i8_workspace_size": ([_I, _I], _SZ),
    "qlin_t158_i8_ws": ([_P, _P, _P, _I64, _F, _P, _P, _I, _I, _I, _P, _SZ, _P], _ST),
    "qlin_w8_f32": ([_P, _P, _I64, _F, _P, _I, _I, _I, _P], _ST),
    "qlin_w8_f32_workspace_size": ([_I, _I], _SZ),
    "qlin_w8_f32_ws": ([_P, _P, _I64, _F, _P, _I, _I, _I, _P, _SZ, _P], _ST),
    "qlin_w8g_quantize": ([_P, _I64, _I64, _I, _P, _I64, _P, _I64, _P], _ST),
    "qlin_w8g_f32": ([_P, _P, _I64, _P, _I64, _I, _P, _I, _I, _I, _P], _ST),
    "qlin_embed_bf16": ([_P, _I, _I, _P, _P, _P, _P], _ST),
    "qlin_rmsnorm": ([_P, _P, _P, _I, _I, _F, _P], _ST),
    "t158_rope_table": ([_P, _P, _I, _I, _D, _P], _ST),
    "qlin_rope_kv_append": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _ST),
    "qlin_attention_workspace_size": ([_I, _I, _I], _SZ),
    "qlin_attention_decode": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _ST),
    "qlin_attention_decode_noalloc": ([_P, _P, _P, _I, _I, _I, _I, _P, _P], _ST),
    "qlin_geglu": ([_P, _P, _P, _I, _P], _ST),
    "qlin_lm_head_workspace_size": ([_I], _SZ),
    "qlin_lm_head_argmax": ([_P, _P, _I, _I, _P, _P, _P, _SZ, _P], _ST),
    "qlin_sketch_emb_t_pitch": ([_I], ctypes.c_int64),
    "qlin_sketch_signs_bytes": ([_I, _I], _SZ),
    "qlin_sketch_prepare": ([_P, _I, _I, _P, _P, _P, _P, _P, _P], _ST),
    "qlin_sketch_workspace_size": ([_I], _SZ),
    "qlin_sketch_head": ([_P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _SZ, _P], _ST),
    "qlin_sketch_head_status": ([_P, _P], _ST),
    "decode_step_t158_workspace_size": ([ctypes.POINTER(T158ModelC), ctypes.POINTER(_SZ)], _ST),
    "decode_step_t158": ([ctypes.POINTER(T158ModelC), _P, _P, _SZ, _P, ctypes.c_int32, _P, _P, _P], _ST),
    "decode_step_t158_launches": ([ctypes.POINTER(T158ModelC)], _I),
    "decode_step_t158_status": ([_P, _P], _ST),
    "decode_step_t158_set_wait_limit": ([ctypes.c_uint64], None),
    "decode_step_t158_test_withhold": ([ctypes.c_int], None),
    "decode_step_t158_sketch_workspace_size": ([ctypes.POINTER(T158ModelC), ctypes.POINTER(T158SketchC),
                                                ctypes.POINTER(_SZ)], _ST),
    "decode_step_t158_sketch": ([ctypes.POINTER(T158ModelC), ctypes.POINTER(T158SketchC), _P, _P, _SZ, _P,
                                 ctypes.c_int32, _P, _P], _ST),
    "t158_group_pitch": ([_I64], _I64),
    "t158_pack_groups": ([_P, _I64, _I64, _P, _I64], _ST),
    "qlin_t158_skip_workspace_size": ([_I], _SZ),
    "qlin_t158_i8_skip": ([_P, _P, _P, _I64, _F, _P, _P, _I, _I, _P, _SZ, _P], _ST),
    "qlin_lm_head_lanes_workspace_size": ([_I, _I], _SZ),
    "qlin_lm_head_lanes": ([_P, _P, _I, _I, _I, _P, _P, _P, _SZ, _P], _ST),
    "qlin_lm_head_lanes_status": ([_P, _P], _ST),
    "decode_lanes_t158_workspace_size": ([ctypes.POINTER(T158ModelC), _I, ctypes.POINTER(_SZ)], _ST),
    "decode_lanes_t158": ([ctypes.POINTER(T158ModelC), _P, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _I, _P], _ST),
    "decode_lanes_t158_launches": ([ctypes.POINTER(T158ModelC), _I], _I),
    "decode_lanes_t158_status": ([_P, _P], _ST),
    "decode_step_t158_sketch_status": ([ctypes.POINTER(T158ModelC), ctypes.POINTER(T158SketchC), _P, _P], _ST),
}


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"{LIB} is missing: build it with `python -m weight_streaming_gemv_gb300.build` "
                                   "(there is no fallback implementation)")
            L = ctypes.CDLL(LIB)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_name(s: int) -> str:
    return lib().qlin_status_str(int(s)).decode()


def _check(fn: str, s: int):
    if s != 0:
        raise QlinError(fn, s, lib().qlin_last_error().decode())


def _ptr(t):
    """Device/host address of a torch tensor or numpy array; ints pass through; None is NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ host packing
def t158_pitch(K: int) -> int:
    return int(lib().t158_pitch(K))


def t158_pack(trits: np.ndarray, pitch: int | None = None) -> np.ndarray:
    t = np.ascontiguousarray(trits, np.int8)
    N, K = t.shape
    pitch = t158_pitch(K) if pitch is None else pitch
    out = np.empty((N, pitch), np.uint8)
    _check("t158_pack", lib().t158_pack(_ptr(t), N, K, _ptr(out), pitch))
    return out


def t158_unpack(packed: np.ndarray, K: int) -> np.ndarray:
    pk = np.ascontiguousarray(packed, np.uint8)
    N, pitch = pk.shape
    out = np.empty((N, K), np.int8)
    _check("t158_unpack", lib().t158_unpack(_ptr(pk), N, K, pitch, _ptr(out)))
    return out


# ------------------------------------------------------------------ device calls
def qlin_w8_quantize(w, N, K, w8, w_pitch, scale, stream=None):
    _check("qlin_w8_quantize", lib().qlin_w8_quantize(_ptr(w), N, K, _ptr(w8), w_pitch, _ptr(scale), _stream(stream)))


def qlin_quant_i8(x, xq, x_scale, M, K, stream=None):
    _check("qlin_quant_i8", lib().qlin_quant_i8(_ptr(x), _ptr(xq), _ptr(x_scale), M, K, _stream(stream)))


def qlin_t158_i8(xq, x_scale, w_packed, w_pitch, w_scale, y, acc, M, N, K, stream=None):
    _check("qlin_t158_i8", lib().qlin_t158_i8(_ptr(xq), _ptr(x_scale), _ptr(w_packed), w_pitch, float(w_scale),
                                              _ptr(y), _ptr(acc), M, N, K, _stream(stream)))


def qlin_t158_i8_workspace_size(M, K):
    return int(lib().qlin_t158_i8_workspace_size(M, K))


def qlin_t158_i8_ws(xq, x_scale, w_packed, w_pitch, w_scale, y, acc, M, N, K, workspace, workspace_bytes,
                    stream=None):
    _check("qlin_t158_i8_ws", lib().qlin_t158_i8_ws(_ptr(xq), _ptr(x_scale), _ptr(w_packed), w_pitch,
                                                    float(w_scale), _ptr(y), _ptr(acc), M, N, K, _ptr(workspace),
                                                    workspace_bytes, _stream(stream)))


def qlin_w8_f32(x, w8, w_pitch, w_scale, y, M, N, K, stream=None):
    _check("qlin_w8_f32", lib().qlin_w8_f32(_ptr(x), _ptr(w8), w_pitch, float(w_scale), _ptr(y), M, N, K,
                                            _stream(stream)))


def qlin_w8_f32_workspace_size(M, K):
    return int(lib().qlin_w8_f32_workspace_size(M, K))


def qlin_w8_f32_ws(x, w8, w_pitch, w_scale, y, M, N, K, workspace, workspace_bytes, stream=None):
    _check("qlin_w8_f32_ws", lib().qlin_w8_f32_ws(_ptr(x), _ptr(w8), w_pitch, float(w_scale), _ptr(y), M, N, K,
                                                  _ptr(workspace), workspace_bytes, _stream(stream)))


def qlin_w8g_quantize(w, N, K, G, w8, w_pitch, scales, s_pitch, stream=None):
    _check("qlin_w8g_quantize", lib().qlin_w8g_quantize(_ptr(w), N, K, G, _ptr(w8), w_pitch, _ptr(scales), s_pitch,
                                                        _stream(stream)))


def qlin_w8g_f32(x, w8, w_pitch, scales, s_pitch, G, y, M, N, K, stream=None):
    _check("qlin_w8g_f32", lib().qlin_w8g_f32(_ptr(x), _ptr(w8), w_pitch, _ptr(scales), s_pitch, G, _ptr(y), M, N, K,
                                              _stream(stream)))


def qlin_embed_bf16(emb, vocab, dim, token, h, status_word=None, stream=None):
    _check("qlin_embed_bf16", lib().qlin_embed_bf16(_ptr(emb), vocab, dim, _ptr(token), _ptr(h), _ptr(status_word),
                                                    _stream(stream)))


def qlin_rmsnorm(x, gamma, out, M, n, eps, stream=None):
    _check("qlin_rmsnorm", lib().qlin_rmsnorm(_ptr(x), _ptr(gamma), _ptr(out), M, n, float(eps), _stream(stream)))


def t158_rope_table(cos_t, sin_t, max_pos, head_dim, base, stream=None):
    _check("t158_rope_table", lib().t158_rope_table(_ptr(cos_t), _ptr(sin_t), max_pos, head_dim, float(base),
                                                    _stream(stream)))


def qlin_rope_kv_append(q, k, v, k_cache, v_cache, cos_t, sin_t, pos, n_heads, n_kv, head_dim, stream=None):
    _check("qlin_rope_kv_append", lib().qlin_rope_kv_append(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                                            _ptr(cos_t), _ptr(sin_t), pos, n_heads, n_kv, head_dim,
                                                            _stream(stream)))


def qlin_attention_workspace_size(max_pos, n_heads, head_dim) -> int:
    return int(lib().qlin_attention_workspace_size(max_pos, n_heads, head_dim))


def qlin_attention_decode(q, k_cache, v_cache, pos, n_heads, n_kv, head_dim, out, workspace, workspace_bytes,
                          stream=None):
    _check("qlin_attention_decode", lib().qlin_attention_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), pos, n_heads,
                                                                n_kv, head_dim, _ptr(out), _ptr(workspace),
                                                                workspace_bytes, _stream(stream)))


ATTENTION_NOALLOC_SCRATCH_BYTES = 262144


def qlin_attention_decode_noalloc(q, k_cache, v_cache, pos, n_heads, n_kv, head_dim, out, stream=None):
    """Decode attention without a workspace argument, for callers that cannot allocate
    device memory: the partials go to a fixed 256 KiB array inside the library.  Calls
    that overlap on the GPU share that array and race."""
    _check("qlin_attention_decode_noalloc",
           lib().qlin_attention_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), pos, n_heads, n_kv, head_dim,
                                               _ptr(out), _stream(stream)))


def qlin_geglu(g, u, a, n, stream=None):
    _check("qlin_geglu", lib().qlin_geglu(_ptr(g), _ptr(u), _ptr(a), n, _stream(stream)))


def qlin_lm_head_workspace_size(vocab) -> int:
    return int(lib().qlin_lm_head_workspace_size(vocab))


def qlin_lm_head_argmax(emb, x, vocab, dim, logits, next_token, workspace, workspace_bytes, stream=None):
    _check("qlin_lm_head_argmax", lib().qlin_lm_head_argmax(_ptr(emb), _ptr(x), vocab, dim, _ptr(logits),
                                                            _ptr(next_token), _ptr(workspace), workspace_bytes,
                                                            _stream(stream)))


def qlin_sketch_emb_t_pitch(vocab) -> int:
    return int(lib().qlin_sketch_emb_t_pitch(vocab))


def qlin_sketch_signs_bytes(vocab, dim) -> int:
    return int(lib().qlin_sketch_signs_bytes(vocab, dim))


def qlin_sketch_prepare(emb, vocab, dim, dim_scale, emb_t, signs, perm, c_e, stream=None):
    _check("qlin_sketch_prepare", lib().qlin_sketch_prepare(_ptr(emb), vocab, dim, _ptr(dim_scale), _ptr(emb_t),
                                                            _ptr(signs), _ptr(perm), _ptr(c_e), _stream(stream)))


def qlin_sketch_workspace_size(vocab) -> int:
    return int(lib().qlin_sketch_workspace_size(vocab))


def qlin_sketch_head(emb, emb_t, signs, perm, c_e, vocab, dim, x, k, n_cand, approx, cand, cand_logits,
                     next_token, workspace, workspace_bytes, stream=None):
    _check("qlin_sketch_head", lib().qlin_sketch_head(
        _ptr(emb), _ptr(emb_t), _ptr(signs), _ptr(perm), _ptr(c_e), vocab, dim, _ptr(x), k, n_cand, _ptr(approx),
        _ptr(cand), _ptr(cand_logits), _ptr(next_token), _ptr(workspace), workspace_bytes, _stream(stream)))


def qlin_sketch_head_status(workspace, stream=None):
    _check("qlin_sketch_head_status", lib().qlin_sketch_head_status(_ptr(workspace), _stream(stream)))


def decode_step_t158_workspace_size(model: T158ModelC) -> int:
    n = ctypes.c_size_t()
    _check("decode_step_t158_workspace_size", lib().decode_step_t158_workspace_size(ctypes.byref(model), ctypes.byref(n)))
    return n.value


def decode_step_t158(model: T158ModelC, kv_cache, workspace, workspace_bytes, token, pos, logits, next_token,
                     stream=None):
    _check("decode_step_t158", lib().decode_step_t158(ctypes.byref(model), _ptr(kv_cache), _ptr(workspace),
                                                      workspace_bytes, _ptr(token), int(pos), _ptr(logits),
                                                      _ptr(next_token), _stream(stream)))


def decode_step_t158_launches(model: T158ModelC) -> int:
    return int(lib().decode_step_t158_launches(ctypes.byref(model)))


def decode_step_t158_status(workspace, stream=None):
    _check("decode_step_t158_status", lib().decode_step_t158_status(_ptr(workspace), _stream(stream)))


def decode_step_t158_set_wait_limit(ns: int):
    lib().decode_step_t158_set_wait_limit(int(ns))


def decode_step_t158_test_withhold(layer: int):
    lib().decode_step_t158_test_withhold(int(layer))


def decode_step_t158_sketch_workspace_size(model: T158ModelC, sk: T158SketchC) -> int:
    n = ctypes.c_size_t()
    _check("decode_step_t158_sketch_workspace_size",
           lib().decode_step_t158_sketch_workspace_size(ctypes.byref(model), ctypes.byref(sk), ctypes.byref(n)))
    return n.value


def decode_step_t158_sketch(model: T158ModelC, sk: T158SketchC, kv_cache, workspace, workspace_bytes, token, pos,
                            next_token, stream=None):
    _check("decode_step_t158_sketch", lib().decode_step_t158_sketch(
        ctypes.byref(model), ctypes.byref(sk), _ptr(kv_cache), _ptr(workspace), workspace_bytes, _ptr(token), pos,
        _ptr(next_token), _stream(stream)))


def decode_step_t158_sketch_status(model: T158ModelC, sk: T158SketchC, workspace, stream=None):
    _check("decode_step_t158_sketch_status", lib().decode_step_t158_sketch_status(
        ctypes.byref(model), ctypes.byref(sk), _ptr(workspace), _stream(stream)))


def decode_lanes_t158_workspace_size(model: T158ModelC, max_lanes: int) -> int:
    n = ctypes.c_size_t()
    _check("decode_lanes_t158_workspace_size",
           lib().decode_lanes_t158_workspace_size(ctypes.byref(model), max_lanes, ctypes.byref(n)))
    return n.value


def decode_lanes_t158(model: T158ModelC, kv_caches, n_seqs, n_lanes, tokens, positions, seqs, logits, next_tokens,
                      workspace, workspace_bytes, max_lanes, stream=None):
    _check("decode_lanes_t158", lib().decode_lanes_t158(
        ctypes.byref(model), _ptr(kv_caches), n_seqs, n_lanes, _ptr(tokens), _ptr(positions), _ptr(seqs),
        _ptr(logits), _ptr(next_tokens), _ptr(workspace), workspace_bytes, max_lanes, _stream(stream)))


def decode_lanes_t158_launches(model: T158ModelC, n_lanes: int) -> int:
    return int(lib().decode_lanes_t158_launches(ctypes.byref(model), n_lanes))


def decode_lanes_t158_status(workspace, stream=None):
    _check("decode_lanes_t158_status", lib().decode_lanes_t158_status(_ptr(workspace), _stream(stream)))


def qlin_lm_head_lanes_workspace_size(vocab, dim) -> int:
    return int(lib().qlin_lm_head_lanes_workspace_size(vocab, dim))


def qlin_lm_head_lanes(emb, x, vocab, dim, n_lanes, logits, next_tokens, workspace, workspace_bytes, stream=None):
    _check("qlin_lm_head_lanes", lib().qlin_lm_head_lanes(_ptr(emb), _ptr(x), vocab, dim, n_lanes, _ptr(logits),
                                                          _ptr(next_tokens), _ptr(workspace), workspace_bytes,
                                                          _stream(stream)))


def qlin_lm_head_lanes_status(workspace, stream=None):
    _check("qlin_lm_head_lanes_status", lib().qlin_lm_head_lanes_status(_ptr(workspace), _stream(stream)))


def t158_group_pitch(N: int) -> int:
    return int(lib().t158_group_pitch(N))


def t158_pack_groups(trits, gpitch=None):
    """Host packing by input group (for qlin_t158_i8_skip): [ceil(K/4)][gpitch] uint8."""
    t = np.ascontiguousarray(trits, np.int8)
    N, K = t.shape
    gpitch = t158_group_pitch(N) if gpitch is None else gpitch
    out = np.empty(((K + 3) // 4, gpitch), np.uint8)
    _check("t158_pack_groups", lib().t158_pack_groups(t.ctypes.data, N, K, out.ctypes.data, gpitch))
    return out


def qlin_t158_skip_workspace_size(N) -> int:
    return int(lib().qlin_t158_skip_workspace_size(N))


def qlin_t158_i8_skip(xq, x_scale, w_groups, gpitch, w_scale, y, acc, N, K, workspace, workspace_bytes, stream=None):
    _check("qlin_t158_i8_skip", lib().qlin_t158_i8_skip(_ptr(xq), _ptr(x_scale), _ptr(w_groups), gpitch, w_scale,
                                                        _ptr(y), _ptr(acc), N, K, _ptr(workspace), workspace_bytes,
                                                        _stream(stream)))
