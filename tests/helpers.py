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


def outside_stats(got, ref, atol=ATOL, rtol=RTOL):
    """(fraction of elements outside atol + rtol*|ref|, worst |got - ref| / (atol + rtol*|ref|),
    rms error) of got against ref."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    ratio = err / (atol + rtol * np.abs(ref))
    return float((ratio > 1).mean()), float(ratio.max()), float(np.sqrt((err ** 2).mean()))


def assert_within(got, ref, name, max_frac=0.0, max_ratio=1.0):
    """The per-element bound on all but `max_frac` of the elements, and no element beyond
    `max_ratio` times the bound.  With the defaults: the bound on every element."""
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), name
    frac, worst, rms = outside_stats(got, ref)
    print(f"{name}: {frac:.2e} outside {ATOL}+{RTOL}|ref| (limit {max_frac:.1e}), worst {worst:.2f}x "
          f"(limit {max_ratio:.2f}x), rms error {rms:.2e}")
    assert frac <= max_frac, f"{name}: {frac:.2e} of elements outside {ATOL}+{RTOL}|ref| (allowed {max_frac:.1e})"
    assert worst <= max_ratio, f"{name}: worst element at {worst:.2f}x the bound (allowed {max_ratio:.2f}x)"
    return frac, worst
