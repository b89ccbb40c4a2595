"""The allocation-free decode attention entry point.

qlin_attention_decode_noalloc serves callers that cannot call cudaMalloc (a
plugin inside an application that owns all device memory, a real-time loop
that cannot risk an allocation, a process that reserved its memory up front):
it keeps its chunk partials in a fixed 256 KiB array inside the library
instead of a caller workspace.  These checks call it through the C ABI and
compare it, bit for bit (the tolerance of the attention parity tests), with
the oracle's decode attention and with qlin_attention_decode, which takes a
workspace, on two calls in a row: the second call runs on the array the
first one left behind.  The largest call that fits the array is checked the
same way.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import device, host, to_dev

pytestmark = pytest.mark.gpu


def _with_workspace(qlin, q, kc, vc, pos, nh, nkv, hd, dev):
    import torch

    out = torch.empty(nh * hd, dtype=torch.float32, device=dev)
    wsb = qlin.qlin_attention_workspace_size(pos + 1, nh, hd)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_attention_decode(q, kc, vc, pos, nh, nkv, hd, out, ws, wsb)
    return host(out)


def _inputs(i, pos, nh, nkv, hd):
    q = synth.normal_f32(70, i, (nh * hd,), 0.0, 0.5)
    kc = synth.normal_f32(71, i, (pos + 1, nkv * hd))
    vc = synth.normal_f32(72, i, (pos + 1, nkv * hd))
    return q, kc, vc


def _check(qlin, dev, i, pos, nh, nkv, hd):
    import torch

    q, kc, vc = _inputs(i, pos, nh, nkv, hd)
    ref = oracle.attention(q, kc, vc, pos, nh, nkv, hd)
    qd, kd, vd = to_dev(q, dev), to_dev(kc, dev), to_dev(vc, dev)
    out = torch.full((nh * hd,), float("nan"), dtype=torch.float32, device=dev)
    qlin.qlin_attention_decode_noalloc(qd, kd, vd, pos, nh, nkv, hd, out)
    got = host(out)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(got, _with_workspace(qlin, qd, kd, vd, pos, nh, nkv, hd, dev))


def test_noalloc_matches_oracle_two_calls_in_a_row():
    from weight_streaming_gemv_gb300 import qlin

    dev = device()
    # the Gemma-3-1B shape at context 1088, then a small GQA case on what the first call left
    for i, (pos, nh, nkv, hd) in enumerate([(1087, 4, 1, 256), (40, 4, 2, 16)]):
        _check(qlin, dev, i, pos, nh, nkv, hd)


def test_noalloc_rejects_calls_beyond_its_array():
    import torch
    from weight_streaming_gemv_gb300 import qlin

    dev = device()
    nh, nkv, hd = 4, 1, 256
    pos = 2016  # needs 4 * 64 chunks * 258 floats = 264,192 bytes > 262,144
    assert qlin.qlin_attention_workspace_size(pos + 1, nh, hd) > qlin.ATTENTION_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(nh * hd, dtype=torch.float32, device=dev)
    kc = torch.zeros((pos + 1, nkv * hd), dtype=torch.float32, device=dev)
    out = torch.full((nh * hd,), 7.0, dtype=torch.float32, device=dev)
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_attention_decode_noalloc(q, kc, kc, pos, nh, nkv, hd, out)
    assert e.value.status == 2 and "scratch" in str(e.value)
    assert (host(out) == 7.0).all()  # nothing was launched
    # the largest call that fits (nearly the whole array) is still exact
    assert qlin.qlin_attention_workspace_size(pos, nh, hd) <= qlin.ATTENTION_NOALLOC_SCRATCH_BYTES
    _check(qlin, dev, 2, pos - 1, nh, nkv, hd)
