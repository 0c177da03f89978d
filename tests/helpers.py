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


# Full-size workloads: the per-element bound above must hold on all but a small
# fraction of elements, and every element must stay within a hard bound derived
# from the BF16 operand-rounding cascade.  tests/tolerance_model.py models a
# correct float32-accumulating BF16 implementation on the CPU: against the
# float64 oracle it leaves 1.0e-3 of the 7B prefill outputs outside the
# per-element bound (rms error 5.8e-3, worst 0.044, 2.4x the bound), 1.5e-5 of
# the 7B decode outputs and none of the 70B decode outputs.  The tensor cores'
# float32 accumulation adds a little more spread (2.6e-3 measured on GB300).
FULL_MAX_FRAC_OUTSIDE = 5e-3
FULL_HARD_ATOL = 6e-2


def assert_close_fullsize(got, ref, name=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name
    err = np.abs(got - ref)
    frac = float((err > ATOL + RTOL * np.abs(ref)).mean())
    print(f"{name}: {frac:.2e} outside {ATOL}+{RTOL}|ref|, rms error {float(np.sqrt((err ** 2).mean())):.2e}, "
          f"worst {float((err / (FULL_HARD_ATOL + RTOL * np.abs(ref))).max()):.2f} of the hard bound")
    assert frac <= FULL_MAX_FRAC_OUTSIDE, (
        f"{name}: {frac:.2e} of elements outside {ATOL}+{RTOL}|ref| (allowed {FULL_MAX_FRAC_OUTSIDE})")
    assert_close(got, ref, name + " [hard bound]", atol=FULL_HARD_ATOL, rtol=RTOL)
    return frac
