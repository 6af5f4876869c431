"""Shared helpers for the GPU parity tests: tolerances and comparisons.

Tolerances (fixed by the serving spec): bf16 outputs within rtol = atol =
2e-2 elementwise against the fp64 oracle, and - because outputs at these
input distributions are ~4e-3 in magnitude, where atol alone cannot catch a
wrong answer - within 1e-2 relative Frobenius norm; fp32 states within 1e-3
relative Frobenius; indices and untouched memory bit-exact.

bf16 recurrent states: within 5e-3 relative Frobenius.  The bound is the
fp32 state bound plus one bf16 rounding step (2^-8 relative) on every
element: the kernel and the oracle round the same values, but values lying
within the fp32 path's error of a bf16 rounding boundary may go either way.
"""
from __future__ import annotations

import numpy as np
import torch

OUT_RTOL = 2e-2
OUT_ATOL = 2e-2
OUT_REL_FRO = 1e-2
STATE_REL_FRO = 1e-3
STATE_BF16_REL_FRO = 1e-3 + 2.0 ** -8


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check_out(gpu_out: torch.Tensor, ref: np.ndarray, what: str = "out"):
    got = np64(gpu_out).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    np.testing.assert_allclose(got, ref, rtol=OUT_RTOL, atol=OUT_ATOL, err_msg=what)
    r = rel_fro(got, ref)
    assert r <= OUT_REL_FRO, f"{what}: relative Frobenius error {r:.3e} > {OUT_REL_FRO}"
    return r


def check_state(gpu_state: torch.Tensor, ref: np.ndarray, what: str = "state"):
    got = np64(gpu_state).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_fro(got, ref)
    assert r <= STATE_REL_FRO, f"{what}: relative Frobenius error {r:.3e} > {STATE_REL_FRO}"
    return r


def check_state_bf16(gpu_state: torch.Tensor, ref: np.ndarray, what: str = "bf16 state"):
    """A bf16 state against the oracle's (itself rounded to bf16)."""
    assert gpu_state.dtype == torch.bfloat16, f"{what}: expected a bf16 tensor"
    got = np64(gpu_state).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_fro(got, ref)
    assert r <= STATE_BF16_REL_FRO, f"{what}: relative Frobenius error {r:.3e} > {STATE_BF16_REL_FRO:.3e}"
    return r
