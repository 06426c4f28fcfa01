"""Comparison helpers for the GPU parity tests.

Tolerances (stated by the attention build's target): max |O - O_ref| <= 1e-2 for
fp32 O and max |LSE - LSE_ref| <= 1e-3, where *_ref is the CPU FP64 oracle on
the same bf16 inputs widened exactly.  For bf16 O the output rounding alone
can reach 2^-8 |O| (round to nearest even on an 8-bit significand), so the bf16
check adds that term element by element: |O - O_ref| <= 1e-2 + 2^-8 |O_ref|.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_O = 1e-2
TOL_LSE = 1e-3
BF16_REL = 2.0 ** -8


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def lse_error(lse, lse_ref):
    a, b = to_np(lse), np.asarray(lse_ref, dtype=np.float64)
    ia, ib = np.isneginf(a), np.isneginf(b)
    assert np.array_equal(ia, ib), "rows with no visible key disagree (-inf LSE)"
    assert not np.any(np.isnan(a)), "NaN in LSE"
    if np.all(ia):
        return 0.0
    return float(np.abs(a[~ia] - b[~ib]).max())


def o_error(o, o_ref):
    a, b = to_np(o), np.asarray(o_ref, dtype=np.float64)
    assert not np.any(np.isnan(a)), "NaN in O"
    return float(np.abs(a - b).max()) if a.size else 0.0


def assert_close(o, lse, o_ref, lse_ref, bf16_out=False, what=""):
    a, b = to_np(o), np.asarray(o_ref, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert not np.any(np.isnan(a)), f"{what}: NaN in O"
    if bf16_out:
        bound = TOL_O + BF16_REL * np.abs(b)
        excess = float((np.abs(a - b) - bound).max()) if a.size else -1.0
        assert excess <= 0, f"{what}: bf16 O error exceeds 1e-2 + 2^-8|O| by {excess:.3e}"
    else:
        err = o_error(a, b)
        assert err <= TOL_O, f"{what}: max|dO| = {err:.3e}"
    if lse is not None:
        el = lse_error(lse, lse_ref)
        assert el <= TOL_LSE, f"{what}: max|dLSE| = {el:.3e}"
