"""Shared test helpers: tensor conversion for the oracle and the layer tolerance."""
import numpy as np
import torch

# per-element bound for BF16 layer outputs: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 1e-2
RTOL = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    """float64 numpy copy of a (CPU or CUDA) tensor's values."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 BF16 bit patterns of a BF16 tensor (a copy, on the CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def assert_close(got, ref, name="", atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err = np.abs(got - ref)
    tol = atol + rtol * np.abs(ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} elements outside "
                             f"{atol}+{rtol}|ref|; worst at {i}: got {got[i]} ref {ref[i]}")
    assert np.isfinite(got).all(), name
