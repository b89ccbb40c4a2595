"""Helpers for the GPU parity tests (the CUDA path is called through the C ABI binding)."""
import numpy as np
import pytest


def device():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_gemv_gb300 import build

    build.build()
    return torch.device("cuda:0")


def to_dev(a: np.ndarray, dev):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def host(t) -> np.ndarray:
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def max_abs_rel(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max |ref| -- the error measure of the parity tolerances."""
    scale = float(np.abs(ref).max())
    return float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max() / (scale if scale > 0 else 1.0))
