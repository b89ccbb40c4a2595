"""CPU-side checks of the C-ABI library: it loads, exports every symbol that
include/qlin.h declares, its host packing matches the oracle's byte for byte,
and argument validation rejects bad calls before anything is launched."""
import os
import re

import numpy as np
import pytest

import oracle
import synth
from conftest import ROOT, read_golden

qlin = pytest.importorskip("weight_streaming_gemv_gb300.qlin")


@pytest.fixture(scope="module", autouse=True)
def built():
    from weight_streaming_gemv_gb300 import build

    build.build()


def header_functions():
    txt = open(os.path.join(ROOT, "include", "qlin.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", txt)
    skip = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in skip and (n.startswith("qlin_") or n.startswith("t158_")
                                                          or n.startswith("decode_step"))})


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 20
    lib = qlin.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding covers every one of them
    assert set(names) <= set(qlin.SIGNATURES), set(names) - set(qlin.SIGNATURES)


def test_status_strings_and_version():
    assert qlin.status_name(0) == "QLIN_OK"
    assert qlin.status_name(5) == "QLIN_ERR_TIMEOUT"
    assert qlin.lib().qlin_version() >= 100


@pytest.mark.parametrize("K,expect", [(1, 16), (80, 16), (81, 32), (1152, 240), (1024, 208), (6912, 1392)])
def test_gpu_pitch(K, expect):
    assert qlin.t158_pitch(K) == expect


@pytest.mark.parametrize("row", read_golden("t158_pack_hand.txt"))
def test_pack_hand_vectors(row):
    t = np.array(row[0], np.int8)[None, :]
    assert int(qlin.t158_pack(t, 16)[0, 0]) == int(row[1][0])


@pytest.mark.parametrize("K", [1, 4, 5, 6, 31, 1152, 1157, 6912])
def test_pack_matches_oracle_bytes(K):
    t = synth.trits(30, K, (9, K))
    pitch = qlin.t158_pitch(K)
    np.testing.assert_array_equal(qlin.t158_pack(t, pitch), oracle.t158_pack(t, pitch))
    np.testing.assert_array_equal(qlin.t158_unpack(qlin.t158_pack(t, pitch), K), t)


@pytest.mark.parametrize("N,K", [(9, 13), (33, 1152), (6, 4)])
def test_group_pack_matches_oracle_bytes(N, K):
    t = synth.trits(31, K, (N, K))
    gp = qlin.t158_group_pitch(N)
    assert gp % 16 == 0 and gp >= N
    np.testing.assert_array_equal(qlin.t158_pack_groups(t, gp), oracle.t158_pack_groups(t, gp))


def test_unpack_rejects_bytes_above_242():
    pk = np.full((2, 16), 121, np.uint8)
    pk[1, 15] = 243  # in the filler
    with pytest.raises(qlin.QlinError) as e:
        qlin.t158_unpack(pk, 10)
    assert e.value.status == 3


def test_pack_rejects_bad_trits_and_pitch():
    with pytest.raises(qlin.QlinError) as e:
        qlin.t158_pack(np.array([[0, 2, 0]], np.int8), 16)
    assert e.value.status == 1
    with pytest.raises(qlin.QlinError):
        qlin.t158_pack(np.zeros((1, 100), np.int8), 19)


def test_device_calls_validate_before_launch():
    # every one of these fails on the host, so no GPU is needed
    L = qlin.lib()
    assert L.qlin_t158_i8(None, None, None, 16, 1.0, None, None, 1, 1, 1, None) == 1
    assert L.qlin_t158_i8(8, 16, 32, 24, 1.0, 64, None, 1, 8, 100, None) == 1  # pitch not a multiple of 16
    assert L.qlin_t158_i8(8, 16, 40, 32, 1.0, 64, None, 1, 8, 100, None) == 1  # w_packed misaligned
    assert L.qlin_t158_i8(8, 16, 32, 32, 1.0, 64, None, 5000, 8, 100, None) == 2  # M too large
    assert L.qlin_w8_f32(16, 32, 8, 1.0, 64, 1, 1, 16, None) == 1  # pitch < K
    assert L.qlin_w8_f32(16, 32, 16, 1.0, 64, 65, 1, 16, None) == 2  # M > 64
    # the workspace variant: sizes and the workspace checks come before any GPU work
    assert L.qlin_w8_f32_workspace_size(1, 4096) == 0
    assert L.qlin_w8_f32_workspace_size(65, 4096) == 0
    assert L.qlin_w8_f32_workspace_size(16, 4096) >= 16 * 4096 * 6
    nb = L.qlin_w8_f32_workspace_size(4, 300)
    assert L.qlin_w8_f32_ws(16, 32, 16, 1.0, 64, 4, 1, 16, None, nb, None) == 1  # no workspace
    assert L.qlin_w8_f32_ws(16, 32, 16, 1.0, 64, 4, 1, 16, 48, 0, None) == 1  # too small
    assert L.qlin_w8_f32_ws(16, 32, 16, 1.0, 64, 65, 1, 16, 48, 1 << 20, None) == 2  # M > 64
    assert L.qlin_quant_i8(None, 16, 16, 1, 1, None) == 1
    assert L.qlin_attention_decode(16, 16, 16, 0, 4, 1, 24, 16, 16, 1 << 20, None) == 2  # head_dim not pow2
    assert "head_dim" in qlin.lib().qlin_last_error().decode()
    # sketch head: emb, emb_t, signs, perm, c_e, vocab, dim, x, k, n_cand, approx, cand, logits, next, ws, bytes
    ok = (16, 32, 48, 64, 80, 1000, 128, 96, 32, 100, None, 112, 128, 144, 160, 1 << 20, None)
    def sk(**kw):
        names = ("emb", "emb_t", "signs", "perm", "c_e", "V", "D", "x", "k", "n", "approx", "cand", "cl", "nx",
                 "ws", "wsb", "st")
        a = dict(zip(names, ok))
        a.update(kw)
        return L.qlin_sketch_head(*[a[n] for n in names])
    assert sk(k=33) == 1 and sk(k=-1) == 1 and sk(n=0) == 1 and sk(n=1001) == 1
    assert sk(D=132) == 1 and sk(D=4096) == 1 and sk(emb=8) == 1 and sk(x=None) == 1 and sk(perm=None) == 1
    assert sk(D=16, k=20) == 1
    assert "k = 20" in qlin.lib().qlin_last_error().decode()
    assert L.qlin_sketch_prepare(16, 1000, 12, None, 32, 48, 64, 80, None) == 1  # dim % 8
    assert L.qlin_sketch_signs_bytes(1000, 1152) == 18 * 1000 * 8
    assert L.qlin_sketch_emb_t_pitch(1001) == 1008
    m = qlin.T158ModelC()
    import ctypes
    n = ctypes.c_size_t()
    assert L.decode_step_t158_workspace_size(ctypes.byref(m), ctypes.byref(n)) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib

    mod = importlib.import_module("weight_streaming_gemv_gb300.qlin")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        mod.lib()
