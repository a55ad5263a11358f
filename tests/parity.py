"""Helpers for comparing the CUDA path with the fp64 oracle.

Error metric (per output tensor): err = max_i |g_i - o_i| / max(|o_i|, rms(o)),
rms over the whole reference tensor.  Near zeros of the gate or cancelling
sums a plain relative error is meaningless; normalising by the tensor's rms
keeps the bar relative to the output's scale.  Bars: 2e-3 for bf16 inputs
(fp32 accumulation), 1e-5 for fp32 inputs.
"""
from __future__ import annotations

import numpy as np

TOL = {"bf16": 2e-3, "f32": 1e-5}


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    denom = np.maximum(np.abs(ref), rms)
    denom = np.where(denom == 0, 1.0, denom)
    return float(np.max(np.abs(got - ref) / denom))


def assert_close(got, ref, tol, what=""):
    e = rel_err(got, ref)
    assert e <= tol, "%s: max normalised error %.3e > %.1e" % (what, e, tol)
    return e


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (for the bf16-output check)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_bf16_output(got_bf16, ref, tol, what=""):
    """bf16 output: within one bf16 spacing of the reference plus the fp32 bar."""
    got = np.asarray(got_bf16, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = bf16_ulp(ref) + tol * np.maximum(np.abs(ref), rms)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), "%s: %d bf16 outputs off by more than one spacing" % (what, int(bad.sum()))
