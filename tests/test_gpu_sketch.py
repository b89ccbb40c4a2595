"""Parity of the sketch head ([citric] "Step 3: the output layer became the
bottleneck") on the GPU, through the C ABI, with the oracle.

The approximate scores are fp32 with a fixed order on both sides, so they, and
the candidate sets they select, are compared bit for bit.  The candidates'
exact logits are fp32 (the lm_head's arithmetic) against the oracle's fp64,
max-abs-rel 1e-5; the chosen word must equal the oracle's unless the oracle's
best two candidates are closer than that tolerance.
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


def _prepare(emb, dev, scale=None):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    V, D = emb.shape
    emb_d = to_dev(emb, dev)
    emb_t = torch.empty((D, qlin.qlin_sketch_emb_t_pitch(V)), dtype=torch.int16, device=dev)
    signs = torch.empty(qlin.qlin_sketch_signs_bytes(V, D) // 8, dtype=torch.int64, device=dev)
    perm = torch.empty(D, dtype=torch.int32, device=dev)
    c_e = torch.zeros(1, dtype=torch.float32, device=dev)
    sc = None if scale is None else to_dev(np.float32(scale), dev)
    qlin.qlin_sketch_prepare(emb_d, V, D, sc, emb_t, signs, perm, c_e)
    return emb_d, emb_t, signs, perm, c_e


def _run(prep, x, k, n_cand, dev, ws=None):
    import torch
    from weight_streaming_gemv_gb300 import qlin

    emb_d, emb_t, signs, perm, c_e = prep
    V, D = emb_d.shape
    approx = torch.empty(V, dtype=torch.float32, device=dev)
    cand = torch.empty(n_cand, dtype=torch.int32, device=dev)
    cl = torch.empty(n_cand, dtype=torch.float32, device=dev)
    nx = torch.full((1,), -7, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_sketch_workspace_size(V)
    if ws is None:
        ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_sketch_head(emb_d, emb_t, signs, perm, c_e, V, D, to_dev(np.float32(x), dev), k, n_cand, approx,
                          cand, cl, nx, ws, wsb)
    qlin.qlin_sketch_head_status(ws)
    return int(host(nx)[0]), host(cand), host(cl), host(approx)


def _check(emb, x, k, n_cand, dev, prep=None, scale=None):
    prep = prep or _prepare(emb, dev, scale)
    cE = float(host(prep[4])[0])
    perm = oracle.sketch_perm(None if scale is None else np.float32(scale), emb.shape[1])
    np.testing.assert_array_equal(host(prep[3]), perm)
    got = _run(prep, x, k, n_cand, dev)
    want = oracle.sketch_head(emb, x, perm=perm, B=64, k=k, n_cand=n_cand, cE=cE)
    nx, cand, cl, approx = got
    nx_o, cand_o, cl_o, approx_o = want
    np.testing.assert_array_equal(approx.view(np.uint32), approx_o.view(np.uint32))
    np.testing.assert_array_equal(cand, cand_o)
    assert max_abs_rel(cl, cl_o) <= 1e-5
    top = cl_o.max()
    tol = 1e-5 * float(np.abs(cl_o).max())
    near = set(cand_o[cl_o >= top - 2 * tol].tolist())
    if len(near) == 1:
        assert nx == nx_o
    else:
        assert nx in near
    return got, want


@pytest.mark.parametrize("V,D,k,n_cand,sized", [
    (5003, 136, 32, 100, True),    # ragged words and dims (two full 64-dim blocks + 8)
    (1000, 64, 0, 17, True),       # no exact dims, one block
    (777, 24, 24, 5, False),       # every dim exact: no sketch
    (4096, 1152, 32, 4096, True),  # every word a candidate
    (300, 2048, 32, 1, True),      # widest hidden state (32 blocks)
    (1, 8, 2, 1, False),           # one word
    (40000, 1152, 7, 1000, False),  # odd k, identity order
    (2500, 512, 32, 64, True),     # 8 blocks
    (2500, 1536, 32, 64, True),    # 24 blocks
    (40000, 1152, 32, 5000, True),  # more candidates than one CTA resolves: the CTAs finish the select together
])
def test_sketch_head_matches_oracle(dev, V, D, k, n_cand, sized):
    d = synth.sketch_head(30 + V % 97, V, D)
    x = synth.sketch_x(30, V % 7, d["scale"])
    _check(d["emb"], x, k, n_cand, dev, scale=d["scale"] if sized else None)


def test_sketch_head_full_size_and_lm_head_agreement(dev):
    """262144 x 1152 with the page's settings (32 exact dims, ~1000 candidates);
    the candidates' logits are the lm_head kernel's, bit for bit, and the word
    is the exact search's."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    V, D = 262144, 1152
    d = synth.sketch_head(31, V, D)
    x = synth.sketch_x(31, 0, d["scale"])
    prep = _prepare(d["emb"], dev, d["scale"])
    (nx, cand, cl, _), _ = _check(d["emb"], x, 32, 1024, dev, prep, d["scale"])
    lg = torch.empty(V, dtype=torch.float32, device=dev)
    nxl = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = qlin.qlin_lm_head_workspace_size(V)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    qlin.qlin_lm_head_argmax(prep[0], to_dev(x, dev), V, D, lg, nxl, ws, wsb)
    np.testing.assert_array_equal(cl.view(np.uint32), host(lg)[cand].view(np.uint32))
    assert nx == int(host(nxl)[0])


def test_prepared_copies(dev):
    """The dimension-major copy, the sign table in its documented order and c_E
    against the oracle's mean |E|."""
    V, D = 1003, 200
    d = synth.sketch_head(32, V, D)
    emb = d["emb"].copy()
    emb[5, :] = 0x8000  # -0.0: sign bit set
    emb_d, emb_t, signs, perm, c_e = _prepare(emb, dev, d["scale"])
    p = oracle.sketch_perm(d["scale"])
    np.testing.assert_array_equal(host(perm), p)
    Vt = emb_t.shape[1]
    et = host(emb_t).view(np.uint16)
    np.testing.assert_array_equal(et[:, :V], emb.T)
    assert (et[:, V:] == 0).all() and Vt % 8 == 0 and Vt >= V
    nblk = (D + 63) // 64
    words = host(signs).view(np.uint64).reshape(nblk, Vt)
    bits = ((words[:, :, None] >> np.arange(64, dtype=np.uint64)) & np.uint64(1)).astype(np.uint8)  # [b][v][p]
    bits = bits.transpose(1, 0, 2).reshape(Vt, nblk * 64)  # [v][position]
    want = np.zeros_like(bits)
    want[:V, :D] = (emb[:, p] >> 15).astype(np.uint8)
    np.testing.assert_array_equal(bits, want)
    ce = float(host(c_e)[0])
    ce_o = oracle.sketch_ce(emb)
    assert abs(ce - ce_o) <= abs(ce_o) * 2.0 ** -23


def test_ties_and_degenerate_inputs(dev):
    """x = 0: every approximate score is +0, so the candidates are the first
    n_cand words; equal |x| (ties for the exact dims) and duplicated rows
    (score ties); a tie across the exact/sketch boundary."""
    V, D = 3000, 128
    d = synth.sketch_head(33, V, D)
    emb = d["emb"].copy()
    emb[2000:2100] = emb[100]  # a hundred copies of one row
    prep = _prepare(emb, dev, d["scale"])
    (nx, cand, _, approx), _ = _check(emb, np.zeros(D, np.float32), 32, 50, dev, prep, d["scale"])
    np.testing.assert_array_equal(cand, np.arange(50))
    x = np.where(synth.splitmix64_seq(34, D) & np.uint64(1), -1.0, 1.0).astype(np.float32)  # all |x| equal
    _check(emb, x, 32, 64, dev, prep, d["scale"])
    x2 = synth.sketch_x(33, 1, d["scale"])
    x2[:40] = 3.0
    _check(emb, x2, 32, 130, dev, prep, d["scale"])


def test_massive_ties(dev):
    """Every approximate score equal (x = 0) over 20000 words: the boundary bin
    holds them all, the CTAs finish the selection together, and the candidates
    are the first n_cand words.  Equal |x| over 1152 dims (more than the
    pairwise ranking of the boundary magnitude bin takes)."""
    V, D = 20000, 1152
    d = synth.sketch_head(36, V, D)
    prep = _prepare(d["emb"], dev, d["scale"])
    (_, cand, _, _), _ = _check(d["emb"], np.zeros(D, np.float32), 32, 300, dev, prep, d["scale"])
    np.testing.assert_array_equal(cand, np.arange(300))
    x = np.where(synth.splitmix64_seq(37, D) & np.uint64(1), -1.0, 1.0).astype(np.float32)
    _check(d["emb"], x, 32, 300, dev, prep, d["scale"])


def test_workspace_is_reusable(dev):
    """Calls leave the workspace ready for the next: later calls on the same
    workspace, with other hidden states, again match the oracle."""
    import torch
    from weight_streaming_gemv_gb300 import qlin

    V, D = 20000, 256
    d = synth.sketch_head(35, V, D)
    prep = _prepare(d["emb"], dev, d["scale"])
    perm = oracle.sketch_perm(d["scale"])
    cE = float(host(prep[4])[0])
    ws = torch.zeros(qlin.qlin_sketch_workspace_size(V), dtype=torch.uint8, device=dev)
    for tok in range(3):
        x = synth.sketch_x(35, tok, d["scale"])
        nx, cand, _, _ = _run(prep, x, 32, 200, dev, ws)
        nx_o, cand_o, _, _ = oracle.sketch_head(d["emb"], x, perm=perm, k=32, n_cand=200, cE=cE)
        np.testing.assert_array_equal(cand, cand_o)
        assert nx == nx_o
