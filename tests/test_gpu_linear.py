"""GPU parity of the linear-layer rows (S1, S3, S4+S6, S5, S7) against the oracle.

Integer results (codes, accumulators) and the exact T158 epilogue must match
bit for bit; the W8 outputs within max-abs-rel 1e-5.  Full sizes of the
benchmark workloads plus ragged and edge shapes.
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


def _empty(shape, dtype, dev):
    import torch

    return torch.empty(shape, dtype=dtype, device=dev)


# ---------------------------------------------------------------- S3 activation quantiser
@pytest.mark.parametrize("M,K", [(1, 1), (1, 1152), (3, 1157), (16, 6912), (512, 1152)])
def test_quant_i8_bit_exact(dev, M, K):
    import torch

    x = synth.normal_f32(40, K, (M, K))
    x[0, 0] = 0.0
    xq_o, xs_o = oracle.quant_i8(x)
    xq = _empty((M, K), torch.int8, dev)
    xs = _empty((M,), torch.float32, dev)
    from weight_streaming_gemv_gb300 import qlin

    qlin.qlin_quant_i8(to_dev(x, dev), xq, xs, M, K)
    np.testing.assert_array_equal(host(xq), xq_o)
    np.testing.assert_array_equal(host(xs), xs_o)


def test_quant_i8_zero_row_and_ties(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    x = np.zeros((2, 8), np.float32)
    x[1] = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5]
    xq_o, xs_o = oracle.quant_i8(x)
    xq = _empty((2, 8), torch.int8, dev)
    xs = _empty((2,), torch.float32, dev)
    qlin.qlin_quant_i8(to_dev(x, dev), xq, xs, 2, 8)
    np.testing.assert_array_equal(host(xq), xq_o)
    np.testing.assert_array_equal(host(xs), xs_o)


def test_quant_i8_half_integer_boundaries(dev):
    """Inputs exactly at (k + 1/2) times the step and a few ulps either side,
    for every code k and for steps of several magnitudes: the codes must be
    those of the IEEE quotient (the kernel decides far-from-boundary cases with
    a product by the rounded reciprocal and these by the quotient itself)."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    absmax = [1.0, 3.7, 127.0, 0.1, 1e-3, 12345.678, 2.0**20 - 1, 0.9999999, 1.0000001, 5e-10]
    rows = []
    for a in absmax:
        a = np.float32(a)
        s = np.float32(max(a, np.float32(1e-9)) / np.float32(127.0))
        vals = [a]
        for k in range(-127, 127):
            x0 = np.float32(np.float32(k + 0.5) * s)
            for d in (-2, -1, 0, 1, 2):
                x = x0
                for _ in range(abs(d)):
                    x = np.nextafter(x, np.float32(np.inf if d > 0 else -np.inf), dtype=np.float32)
                vals.append(x if abs(x) <= a else np.float32(0.0))
        rows.append(np.array(vals, np.float32))
    K = len(rows[0])
    x = np.stack(rows)
    M = x.shape[0]
    xq_o, xs_o = oracle.quant_i8(x)
    xq = _empty((M, K), torch.int8, dev)
    xs = _empty((M,), torch.float32, dev)
    qlin.qlin_quant_i8(to_dev(x, dev), xq, xs, M, K)
    np.testing.assert_array_equal(host(xs), xs_o)
    np.testing.assert_array_equal(host(xq), xq_o)


def test_w8_m1_unaligned_x_tiny_values_and_nonfinite(dev):
    """The one-token W8 path: x that is not 16-byte aligned (element loads), x
    of tiny magnitude (scaled by two powers of two), and a non-finite x (every
    row reads NaN)."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    K, N = 4099, 333
    d = synth.w8_gemv(3, 1, K, N)
    q_o, s_o = oracle.w8_quantize(d["w"])
    pitch = (K + 15) // 16 * 16
    w8 = np.zeros((N, pitch), np.int8)
    w8[:, :K] = q_o
    w8d = to_dev(w8, dev)
    y = _empty((1, N), torch.float32, dev)
    # x at an odd float offset inside a larger buffer
    buf = torch.zeros(K + 1, dtype=torch.float32, device=dev)
    buf[1:] = to_dev(d["x"][0], dev)
    qlin.qlin_w8_f32(buf[1:], w8d, pitch, float(s_o), y, 1, N, K)
    assert max_abs_rel(host(y), oracle.w8_linear(d["x"], q_o, s_o)) <= 1e-5
    # tiny magnitudes (below 2^-100)
    xt = (d["x"] * np.float32(2.0**-110)).astype(np.float32)
    qlin.qlin_w8_f32(to_dev(xt, dev), w8d, pitch, float(s_o), y, 1, N, K)
    assert max_abs_rel(host(y), oracle.w8_linear(xt, q_o, s_o)) <= 1e-5
    # a NaN and an infinity
    for bad in (np.nan, np.inf):
        xb = d["x"].copy()
        xb[0, 77] = bad
        qlin.qlin_w8_f32(to_dev(xb, dev), w8d, pitch, float(s_o), y, 1, N, K)
        assert np.isnan(host(y)).all()


def test_w8_m1_outliers_beside_small_values(dev):
    """The one-token W8 path holds each lane's slice of x as fixed point on the
    scale of the slice's largest |x|.  One outlier (1e4, then 1e6) in every
    16-element chunk of N(0,1) values: with the outliers' weights as drawn the
    result stays within 1e-5 of max|y|; with the outliers' weight columns set
    to zero (the outliers add nothing, the small values carry the sum) every
    row stays within the error bound the entry point states:
    w_scale * sum_k 2^(e(k) - 23) |w8[n][k]| + 2^-19 w_scale sum_k |x[k] w8[n][k]|,
    2^e(k) above the largest |x| of k's slice (here every slice holds an
    outlier, so e is the outlier's exponent)."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    K, N = 4096, 1024
    d = synth.w8_gemv(9, 1, K, N)
    q_o, s_o = oracle.w8_quantize(d["w"])
    for big in (1e4, 1e6):
        x = d["x"].copy()
        x[0, 7::16] = np.float32(big)
        for zero_cols in (False, True):
            q = q_o.copy()
            if zero_cols:
                q[:, 7::16] = 0
            w8d = to_dev(np.ascontiguousarray(q), dev)
            y = _empty((1, N), torch.float32, dev)
            qlin.qlin_w8_f32(to_dev(x, dev), w8d, K, float(s_o), y, 1, N, K)
            got = host(y)[0].astype(np.float64)
            ref = oracle.w8_linear(x, q, s_o)[0].astype(np.float64)
            if not zero_cols:
                assert max_abs_rel(got, ref) <= 1e-5
            e = np.floor(np.log2(np.float64(big))) + 1  # big < 2^e
            qa = np.abs(q.astype(np.float64))
            bound = float(s_o) * (2.0 ** (e - 23)) * qa.sum(1) + 2.0 ** -19 * float(s_o) * (qa @ np.abs(x[0].astype(np.float64)))
            assert (np.abs(got - ref) <= bound).all()


# ---------------------------------------------------------------- S1 W8 quantisation
@pytest.mark.parametrize("N,K", [(768, 288), (4096, 4096), (1, 1), (3, 17)])
def test_w8_quantize_bit_exact(dev, N, K):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    w = synth.normal_f32(41, K, (N, K), 0.0, 0.02)
    q_o, s_o = oracle.w8_quantize(w)
    pitch = (K + 15) // 16 * 16
    w8 = _empty((N, pitch), torch.int8, dev)
    s = _empty((1,), torch.float32, dev)
    qlin.qlin_w8_quantize(to_dev(w, dev), N, K, w8, pitch, s)
    w8h = host(w8)
    np.testing.assert_array_equal(w8h[:, :K], q_o)
    assert (w8h[:, K:] == 0).all()
    assert host(s)[0] == s_o


# ---------------------------------------------------------------- S4 + S6 T158 linear
def _t158_case(dev, M, K, N, seed, trits=None, xq=None, both=True):
    # qlin_t158_i8 and (both) qlin_t158_i8_ws against the oracle, bit for bit
    import torch
    from weight_streaming_gemv_gb300 import qlin

    d = synth.t158_gemv(seed, M, K, N)
    t = d["trits"] if trits is None else trits
    if xq is None:
        xq, xs = oracle.quant_i8(d["x"])
    else:
        xs = np.full(M, 0.01, np.float32)
    acc_o, y_o = oracle.t158_linear(xq, xs, oracle.t158_pack(t), d["w_scale"], K)
    pitch = qlin.t158_pitch(K)
    w = to_dev(qlin.t158_pack(t, pitch), dev)
    xq_d, xs_d = to_dev(xq, dev), to_dev(xs, dev)
    y = _empty((M, N), torch.float32, dev)
    acc = _empty((M, N), torch.int32, dev)
    qlin.qlin_t158_i8(xq_d, xs_d, w, pitch, d["w_scale"], y, acc, M, N, K)
    np.testing.assert_array_equal(host(acc), acc_o)
    np.testing.assert_array_equal(host(y), y_o)
    if both:
        nb = qlin.qlin_t158_i8_workspace_size(M, K)
        work = torch.full((max(nb, 16),), 0x7f, dtype=torch.uint8, device=dev)  # stale bytes must not matter
        y = _empty((M, N), torch.float32, dev)
        acc = _empty((M, N), torch.int32, dev)
        qlin.qlin_t158_i8_ws(xq_d, xs_d, w, pitch, d["w_scale"], y, acc, M, N, K, work, nb)
        np.testing.assert_array_equal(host(acc), acc_o)
        np.testing.assert_array_equal(host(y), y_o)


def test_t158_gemv_gate_up_shape_full_size(dev):
    # M=1, K=1152, N=6912: the Gemma-3-1B GeGLU gate/up shape (rows zero-padded to 1155 trits)
    _t158_case(dev, 1, 1152, 6912, seed=1)


def test_t158_gemv_down_shape_full_size(dev):
    _t158_case(dev, 1, 6912, 1152, seed=2)


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (1, 5, 3), (1, 31, 33), (1, 81, 700), (1, 1024, 1152),
                                   (2, 1157, 333), (3, 640, 65), (4, 1152, 1536), (7, 77, 129),
                                   (16, 6912, 1152), (17, 333, 100)])
def test_t158_ragged_shapes(dev, M, K, N):
    _t158_case(dev, M, K, N, seed=M * 1000 + K)


@pytest.mark.parametrize("K,N", [(2051, 16001), (1999, 3001), (1100, 9800), (333, 9800), (77, 20000)])
def test_t158_m1_row_slot_variants(dev, K, N):
    # one token through the CUDA-core kernel at row counts that select 4, 2 and 1 row slots per warp
    # for each chunk width on a 152-SM GPU; 2051 x 16001 also takes a second grid-stride pass
    _t158_case(dev, 1, K, N, seed=K + N)


@pytest.mark.parametrize("M,K,N", [(2, 6912, 1152), (2, 1999, 3001), (2, 2051, 5000), (4, 6912, 1152),
                                   (4, 1999, 3001), (6, 1100, 9800), (3, 333, 9800), (7, 77, 20000)])
def test_t158_few_tokens_row_slot_variants(dev, M, K, N):
    # 2..7 tokens through the CUDA-core kernel at row counts that select 4 (two tokens only), 2 and 1
    # row slots per warp on a 152-SM GPU
    _t158_case(dev, M, K, N, seed=100 * M + K)


@pytest.mark.parametrize("M,N", [(1, 64), (3, 33), (7, 40)])
def test_t158_longest_rows(dev, M, N):
    # K = 131071, the largest the entry points accept: a few tokens' activation planes no longer fit in
    # shared memory, so the tensor-core kernel takes the call (the same acc and y, bit for bit)
    _t158_case(dev, M, 131071, N, seed=M + N)


def test_t158_adversarial_extremes(dev):
    # all +1 trits against all +127 activations: acc = 127 K at K = 6912, the largest in use
    K, N = 6912, 64
    t = np.ones((N, K), np.int8)
    t[1] = -1
    t[2] = 0
    t[3, ::2] = -1
    xq = np.full((2, K), 127, np.int8)
    xq[1, ::3] = -127
    _t158_case(dev, 2, K, N, seed=9, trits=t, xq=xq)


@pytest.mark.parametrize("K,N", [(1152, 6912), (6912, 1152)])
def test_t158_prefill_m512_full_size(dev, K, N):
    # the two prefill layers: 512 tokens through 1152->6912 and 6912->1152
    _t158_case(dev, 512, K, N, seed=2)


@pytest.mark.parametrize("M,K,N", [(64, 80, 128), (128, 80, 128), (100, 100, 200), (300, 1155, 130), (129, 161, 257),
                                   (512, 6912, 100), (8, 1152, 6912), (16, 6912, 1152), (32, 1152, 300), (9, 77, 33)])
def test_t158_tensor_core_tiles(dev, M, K, N):
    # the tensor-core path (M >= 64): ragged token, row and K tiles against the oracle, bit for bit
    _t158_case(dev, M, K, N, seed=11)


@pytest.mark.parametrize("M,K,N", [(257, 333, 200), (4096, 160, 129), (40, 6912, 1152), (200, 1152, 140),
                                   (64, 1152, 6912), (480, 240, 384)])
def test_t158_tensor_core_token_tiles(dev, M, K, N):
    # token tiles of 32..128 (the MMA's N), one or several per call, with and
    # without split K, against the oracle bit for bit
    _t158_case(dev, M, K, N, seed=13)


def test_t158_tensor_core_extreme_operands(dev):
    # all codes -127 / +127 against all-minus / all-plus trits: the largest
    # partial sums the fp32 accumulator must hold exactly (127 K)
    M, K, N = 96, 6912, 256
    xq = np.full((M, K), 127, np.int8)
    xq[1::2] = -127
    t = np.ones((N, K), np.int8)
    t[::3] = -1
    _t158_case(dev, M, K, N, seed=14, trits=t, xq=xq)


def test_t158_ws_one_workspace_for_many_calls(dev):
    """One workspace of the largest size, filled with stale bytes, serves
    calls of several M and K in a row, twice over, bit for bit against the
    oracle."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    shapes = [(512, 1152, 6912), (40, 6912, 1152), (8, 1152, 700), (130, 333, 2000)]
    nb = max(qlin.qlin_t158_i8_workspace_size(M, K) for M, K, _ in shapes)
    work = torch.full((nb,), 0x7f, dtype=torch.uint8, device=dev)
    cases = []
    for i, (M, K, N) in enumerate(shapes):
        d = synth.t158_gemv(50 + i, M, K, N)
        xq_o, xs_o = oracle.quant_i8(d["x"])
        acc_o, y_o = oracle.t158_linear(xq_o, xs_o, oracle.t158_pack(d["trits"]), d["w_scale"], K)
        pitch = qlin.t158_pitch(K)
        w = torch.from_numpy(qlin.t158_pack(d["trits"], pitch)).to(dev)
        cases.append((M, K, N, pitch, w, to_dev(xq_o, dev), to_dev(xs_o, dev), d["w_scale"], acc_o, y_o))
    for _ in range(2):
        for M, K, N, pitch, w, xq, xs, ws, acc_o, y_o in cases:
            y = _empty((M, N), torch.float32, dev)
            acc = _empty((M, N), torch.int32, dev)
            qlin.qlin_t158_i8_ws(xq, xs, w, pitch, ws, y, acc, M, N, K, work, nb)
            np.testing.assert_array_equal(host(acc), acc_o)
            np.testing.assert_array_equal(host(y), y_o)


def test_t158_ws_rejects_small_workspace(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    M, K, N = 64, 1152, 256
    nb = qlin.qlin_t158_i8_workspace_size(M, K)
    # 64 tokens (one 64-token tile) x 15 steps of 80 inputs, 2 bytes each
    assert nb == 64 * 15 * 80 * 2
    assert qlin.qlin_t158_i8_workspace_size(4, K) == 0  # CUDA-core path: no scratch
    assert qlin.qlin_t158_i8_workspace_size(0, K) == 0 and qlin.qlin_t158_i8_workspace_size(M, 131072) == 0
    xq = torch.zeros((M, K), dtype=torch.int8, device=dev)
    xs = torch.ones(M, dtype=torch.float32, device=dev)
    w = torch.zeros((N, qlin.t158_pitch(K)), dtype=torch.uint8, device=dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    work = torch.empty(nb, dtype=torch.uint8, device=dev)
    with pytest.raises(qlin.QlinError):
        qlin.qlin_t158_i8_ws(xq, xs, w, qlin.t158_pitch(K), 1.0, y, None, M, N, K, work, nb - 16)


def test_t158_tensor_core_unaligned_x_acc_only(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    M, K, N = 96, 333, 140
    d = synth.t158_gemv(12, M, K, N)
    xq_o, xs_o = oracle.quant_i8(d["x"])
    acc_o, _ = oracle.t158_linear(xq_o, xs_o, oracle.t158_pack(d["trits"]), d["w_scale"], K)
    pitch = qlin.t158_pitch(K)
    w = to_dev(qlin.t158_pack(d["trits"], pitch), dev)
    buf = torch.zeros(M * K + 1, dtype=torch.int8, device=dev)
    buf[1:] = to_dev(xq_o.reshape(-1), dev)
    acc = _empty((M, N), torch.int32, dev)
    qlin.qlin_t158_i8(buf[1:], to_dev(xs_o, dev), w, pitch, d["w_scale"], None, acc, M, N, K)
    np.testing.assert_array_equal(host(acc), acc_o)
    # the same through the activation-tile conversion (byte loads: neither aligned nor K % 16 == 0)
    nb = qlin.qlin_t158_i8_workspace_size(M, K)
    work = torch.empty(nb, dtype=torch.uint8, device=dev)
    acc = _empty((M, N), torch.int32, dev)
    qlin.qlin_t158_i8_ws(buf[1:], to_dev(xs_o, dev), w, pitch, d["w_scale"], None, acc, M, N, K, work, nb)
    np.testing.assert_array_equal(host(acc), acc_o)


def test_t158_bad_bytes_are_memory_safe(dev):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    K, N = 100, 50
    pitch = qlin.t158_pitch(K)
    w = torch.full((N, pitch), 255, dtype=torch.uint8, device=dev)
    xq = torch.ones((1, K), dtype=torch.int8, device=dev)
    xs = torch.ones(1, dtype=torch.float32, device=dev)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    qlin.qlin_t158_i8(xq, xs, w, pitch, 1.0, y, None, 1, N, K)
    torch.cuda.synchronize()  # unspecified values, but no fault


# ---------------------------------------------------------------- S5 W8 linear
@pytest.mark.parametrize("M,K,N", [(1, 288, 768), (1, 4096, 11008), (1, 11008, 4096), (1, 4096, 4096),
                                   (4, 4096, 11008), (4, 11008, 4096), (16, 4096, 4096), (16, 11008, 4096),
                                   (16, 4096, 11008), (3, 17, 5), (1, 1, 1), (64, 300, 70),
                                   (1, 5000, 2437), (1, 2047, 9), (1, 300, 7)])
def test_w8_linear(dev, M, K, N):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    d = synth.w8_gemv(3 if K >= 4096 else 0, M, K, N)
    q_o, s_o = oracle.w8_quantize(d["w"])
    y_o = oracle.w8_linear(d["x"], q_o, s_o)
    pitch = (K + 15) // 16 * 16
    w8 = np.zeros((N, pitch), np.int8)
    w8[:, :K] = q_o
    y = _empty((M, N), torch.float32, dev)
    qlin.qlin_w8_f32(to_dev(d["x"], dev), to_dev(w8, dev), pitch, float(s_o), y, M, N, K)
    assert max_abs_rel(host(y), y_o) <= 1e-5


@pytest.mark.parametrize("M,K,N,x_offset,w_pitch", [
    (2, 4096, 4096, 0, None),      # token capacity 4 (MMA N = 16)
    (5, 1000, 300, 0, None),       # capacity 8, K and N ragged against the 128 x 128 weight box
    (8, 11008, 4096, 0, None),     # split K over a cluster of 8
    (13, 4096, 11008, 0, None),    # capacity 16, split K over a cluster of 3
    (17, 2048, 640, 0, None),      # two token tiles
    (33, 129, 257, 0, None),       # three token tiles, one element past a stage, one row past a tile
    (6, 301, 77, 1, None),         # x at an odd float offset, K % 4 != 0: element-wise copies
    (4, 512, 200, 3, 1024),        # x unaligned, row pitch far past K
    (3, 20000, 130, 0, None),      # long rows: a cluster of activation-term CTAs per token
])
def test_w8_tensor_core_shapes(dev, M, K, N, x_offset, w_pitch):
    """The tensor-core path (2 <= M <= 64): token tiles of capacity 4, 8 and 16,
    split K, ragged K and N, unaligned activations and a wide row pitch."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    d = synth.w8_gemv(31, M, K, N)
    q_o, s_o = oracle.w8_quantize(d["w"])
    y_o = oracle.w8_linear(d["x"], q_o, s_o)
    pitch = w_pitch or (K + 15) // 16 * 16
    w8 = np.full((N, pitch), 0x55, np.int8)  # bytes past K are not read as weights
    w8[:, :K] = q_o
    buf = torch.zeros(M * K + x_offset, dtype=torch.float32, device=dev)
    buf[x_offset:] = to_dev(d["x"].reshape(-1), dev)
    w8d = to_dev(w8, dev)
    y = _empty((M, N), torch.float32, dev)
    qlin.qlin_w8_f32(buf[x_offset:], w8d, pitch, float(s_o), y, M, N, K)
    assert max_abs_rel(host(y), y_o) <= 1e-5
    # the same call again: split-K sums in rank order, so the result repeats bit for bit
    y2 = _empty((M, N), torch.float32, dev)
    qlin.qlin_w8_f32(buf[x_offset:], w8d, pitch, float(s_o), y2, M, N, K)
    np.testing.assert_array_equal(host(y2), host(y))
    # the workspace path (activation terms once per call, fp16 operands), twice on one workspace
    nb = qlin.qlin_w8_f32_workspace_size(M, K)
    assert nb > 0
    work = _empty((nb,), torch.uint8, dev)
    y3 = _empty((M, N), torch.float32, dev)
    for _ in range(2):
        qlin.qlin_w8_f32_ws(buf[x_offset:], w8d, pitch, float(s_o), y3, M, N, K, work, nb)
    assert max_abs_rel(host(y3), y_o) <= 1e-5


def test_w8_tensor_core_exact_terms(dev):
    """x values of 24 significant bits over a wide exponent range: the three
    bf16 terms carry them exactly, so with small-integer weights every
    product is exact and the result stays at fp32 accumulation error."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    M, K, N = 16, 2048, 256
    rng = np.random.default_rng(5)
    mant = rng.integers(1 << 23, 1 << 24, size=(M, K)).astype(np.float64)
    expo = rng.integers(-30, 10, size=(M, K))
    sign = rng.choice([-1.0, 1.0], size=(M, K))
    x = (sign * mant * np.exp2(expo - 23)).astype(np.float32)
    q = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    xd, qd = to_dev(x, dev), to_dev(q, dev)
    exact = x.astype(np.float64) @ q.astype(np.float64).T
    bound = 2.0 ** -22 * (np.abs(x).astype(np.float64) @ np.abs(q).astype(np.float64).T) + 1e-30
    y = _empty((M, N), torch.float32, dev)
    qlin.qlin_w8_f32(xd, qd, K, 1.0, y, M, N, K)
    assert (np.abs(host(y) - exact) <= bound).all()
    nb = qlin.qlin_w8_f32_workspace_size(M, K)
    work = _empty((nb,), torch.uint8, dev)
    qlin.qlin_w8_f32_ws(xd, qd, K, 1.0, y, M, N, K, work, nb)
    assert (np.abs(host(y) - exact) <= bound).all()


@pytest.mark.parametrize("ws", [False, True])
def test_w8_tensor_core_nonfinite_token(dev, ws):
    """An infinity or a NaN in one token's x makes that token's outputs NaN and
    leaves the other tokens' outputs as they are."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    M, K, N = 5, 700, 300
    d = synth.w8_gemv(33, M, K, N)
    q_o, s_o = oracle.w8_quantize(d["w"])
    pitch = (K + 15) // 16 * 16
    w8 = np.zeros((N, pitch), np.int8)
    w8[:, :K] = q_o
    x = d["x"].copy()
    x[1, 17] = np.inf
    x[3, 650] = np.nan
    y_o = oracle.w8_linear(np.where(np.isfinite(x), x, 0.0).astype(np.float32), q_o, s_o)
    y = _empty((M, N), torch.float32, dev)
    if ws:
        nb = qlin.qlin_w8_f32_workspace_size(M, K)
        qlin.qlin_w8_f32_ws(to_dev(x, dev), to_dev(w8, dev), pitch, float(s_o), y, M, N, K, _empty((nb,), torch.uint8, dev), nb)
    else:
        qlin.qlin_w8_f32(to_dev(x, dev), to_dev(w8, dev), pitch, float(s_o), y, M, N, K)
    yh = host(y)
    assert np.isnan(yh[[1, 3]]).all()
    ok = [0, 2, 4]
    assert max_abs_rel(yh[ok], y_o[ok]) <= 1e-5


# ---------------------------------------------------------------- W8 with group scales
def _w8g_case(dev, M, K, N, G, seed, x_offset=0, w_pitch=None):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    d = synth.w8_gemv(seed, M, K, N)
    q_o, s_o = oracle.w8g_quantize(d["w"], G)
    y_o = oracle.w8g_linear(d["x"], q_o, s_o, G)
    pitch = w_pitch or (K + 15) // 16 * 16
    ng = (K + G - 1) // G
    s_pitch = (ng + 3) // 4 * 4
    w8 = _empty((N, pitch), torch.int8, dev)
    sc = _empty((N, s_pitch), torch.float32, dev)
    qlin.qlin_w8g_quantize(to_dev(d["w"], dev), N, K, G, w8, pitch, sc, s_pitch)
    w8h, sch = host(w8), host(sc)
    np.testing.assert_array_equal(w8h[:, :K], q_o)
    assert (w8h[:, K:] == 0).all()
    np.testing.assert_array_equal(sch[:, :ng], s_o)
    assert (sch[:, ng:] == 0).all()
    buf = torch.zeros(M * K + x_offset, dtype=torch.float32, device=dev)
    buf[x_offset:] = to_dev(d["x"].reshape(-1), dev)
    y = _empty((M, N), torch.float32, dev)
    qlin.qlin_w8g_f32(buf[x_offset:], w8, pitch, sc, s_pitch, G, y, M, N, K)
    assert max_abs_rel(host(y), y_o) <= 1e-5


@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 11008, 128), (1, 11008, 4096, 128), (1, 300, 70, 128), (1, 1000, 33, 64),
                                     (4, 4096, 1000, 128), (16, 1000, 300, 128), (3, 130, 7, 16)])
def test_w8g_quantize_bit_exact_and_linear(dev, M, K, N, G):
    _w8g_case(dev, M, K, N, G, seed=21)


def test_w8g_unaligned_x_and_wide_pitch(dev):
    # x at an odd float offset; row pitch far past K (chunks past K take no scale)
    _w8g_case(dev, 1, 100, 40, 16, seed=22, x_offset=1, w_pitch=512)
