"""GPU parity of the T158 linear that skips groups of four zero inputs
([citric] "What is next"): acc bit for bit and y bit for bit against the
oracle's T158 linear, for activations with 80% zero groups, dense ones, all
zero, a single nonzero group, ragged K and N, and the decoder's shapes.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import device, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def sparse_codes(seed, K, zero_frac):
    """int8 activation codes of one token whose groups of four are zero with probability zero_frac."""
    x = synth.normal_f32(seed, 1, (1, K), 0.0, 1.0)
    G = (K + 3) // 4
    keep = synth.uniform_f32(seed, 2, (G,), 0.0, 1.0) >= zero_frac
    x[0, :] *= np.repeat(keep, 4)[:K]
    xq, xs = oracle.quant_i8(x)
    return xq, xs


def _run(dev, trits, xq, xs, w_scale):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    N, K = trits.shape
    gp = qlin.t158_group_pitch(N)
    wg = qlin.t158_pack_groups(trits, gp)
    acc = torch.empty(N, dtype=torch.int32, device=dev)
    y = torch.empty(N, dtype=torch.float32, device=dev)
    wsb = qlin.qlin_t158_skip_workspace_size(N)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    wg_d = to_dev(wg, dev)
    for _ in range(2):  # a second call on the same workspace
        qlin.qlin_t158_i8_skip(to_dev(xq, dev), to_dev(xs, dev), wg_d, gp, w_scale, y, acc, N, K, ws, wsb)
    return host(acc), host(y)


@pytest.mark.parametrize("N,K,zero", [(6912, 1152, 0.8), (1152, 6912, 0.8), (6912, 1152, 0.0), (1000, 13, 0.5),
                                      (77, 1025, 0.9), (4096, 4096, 0.95)])
def test_skip_matches_t158_linear(dev, N, K, zero):
    d = synth.t158_gemv(50 + N % 13, 1, K, N)
    xq, xs = sparse_codes(51 + K % 17, K, zero)
    acc, y = _run(dev, d["trits"], xq, xs, d["w_scale"])
    packed = oracle.t158_pack(d["trits"])
    acc_o, y_o = oracle.t158_linear(xq, xs, packed, d["w_scale"], K)
    np.testing.assert_array_equal(acc, acc_o[0])
    np.testing.assert_array_equal(y, y_o[0])


def test_skip_all_zero_and_one_group(dev):
    N, K = 3000, 1152
    t = synth.trits(52, 0, (N, K))
    xq = np.zeros((1, K), np.int8)
    xs = np.ones(1, np.float32)
    acc, y = _run(dev, t, xq, xs, 0.5)
    assert (acc == 0).all() and (y == 0).all()
    xq[0, 404:408] = [3, -7, 127, -128 + 1]  # group 101 only
    acc, _ = _run(dev, t, xq, xs, 0.5)
    want = t[:, 404:408].astype(np.int64) @ xq[0, 404:408].astype(np.int64)
    np.testing.assert_array_equal(acc, want)
