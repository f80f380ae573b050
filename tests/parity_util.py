"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerance (per output tensor, per call), from the arithmetic of the two
dtype paths:
  float32 q/k/v:  max|gpu - ref| <= 1e-3 * max|ref| + 1e-5
  bf16 q/k/v:     max|gpu - ref| <= 2e-2 * max|ref|
The oracle runs in float64 on the exact stored input values (bf16 and f32
convert to f64 exactly), so the bound measures kernel error only.
"""
import numpy as np
import torch

from channelwise_gated_delta_gb300.inputs import to_f64


def tolerance(dtype, ref):
    m = float(np.abs(ref).max()) if ref.size else 0.0
    if dtype == torch.float32:
        return 1e-3 * m + 1e-5
    return 2e-2 * m


def assert_close(name, got, ref, dtype):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.isfinite(got).all(), "%s: non-finite values" % name
    err = float(np.abs(got - ref).max())
    tol = tolerance(dtype, ref)
    assert err <= tol, "%s: max|err| = %.3e > tol %.3e (max|ref| = %.3e)" % (
        name, err, tol, float(np.abs(ref).max()))
    return err


def to_cuda(d, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in d.items()}
