"""Helpers shared by the GPU parity tests: moving the seeded inputs to the
device and comparing the library's results with the oracle's.

Tolerances (bf16 outputs vs the fp64 oracle): an element passes if its
absolute error is at most max(1e-2, one bf16 ulp of the oracle value) --
1e-2 is the stated bar, and for |o| >= 2 the spacing of bf16 itself reaches
or exceeds it, so rounding the exact result to bf16 could not meet 1e-2
there.  LSE (fp32): absolute error at most 1e-3.  Cache writes: bit-exact.
"""

import numpy as np
import torch

OUT_ATOL = 1e-2
LSE_ATOL = 1e-3
BF16_NAN = np.uint16(0x7FC0)


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


def to_dev(a: np.ndarray, dtype, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.exp2(e - 7)


def assert_out_close(got: np.ndarray, ref: np.ndarray, what: str, atol=OUT_ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    allowed = np.maximum(atol, bf16_ulp(ref))
    bad = err > allowed
    if bad.any():
        idx = np.unravel_index(np.argmax(err - allowed), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond tolerance; worst at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r} err {err[idx]:.3e}")
    return float(err.max()) if err.size else 0.0


def assert_lse_close(got: np.ndarray, ref: np.ndarray, what: str, atol=LSE_ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    ninf_r, ninf_g = np.isneginf(ref), np.isneginf(got)
    assert np.array_equal(ninf_r, ninf_g), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    err = np.abs(got[fin] - ref[fin])
    if err.size and err.max() > atol:
        raise AssertionError(f"{what}: LSE error {err.max():.3e} > {atol}")
    return float(err.max()) if err.size else 0.0
