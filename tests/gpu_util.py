"""Helpers for the GPU parity tests: host/device conversion and the error measures.

Error measures (the oracle is float64 on the same rounded inputs):
* ``slice_rel``: max over (batch, head) slices of max|Y - Y_ref| / max|Y_ref|.
  Y is a weighted mean of V and sits near zero, so an elementwise relative
  error is ill-posed; the slice maximum is the scale.
* ``rel``: elementwise |a - b| / |b| (for the positive denominators).
"""

import numpy as np
import torch

# Parity bars: fp32 mode 1e-4, bf16 mode 2e-2 on Y; the denominator 1e-3
# relative in bf16 mode (its values reach 1e4, where fp32 itself cannot hold
# an absolute 1e-3) and 1e-4 in fp32 mode.
TOL_Y = {"f32": 1e-4, "bf16": 2e-2}
TOL_DEN = {"f32": 1e-4, "bf16": 1e-3}


def to_device(arr, device="cuda"):
    """numpy float32 array or uint16 bf16 bit array -> contiguous CUDA tensor."""
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(arr).to(device)


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def torch_dtype(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


def slice_rel(y, ref, lead=2):
    y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
    n = int(np.prod(ref.shape[:lead]))
    err = np.abs(y - ref).reshape(n, -1).max(axis=1)
    scale = np.abs(ref).reshape(n, -1).max(axis=1)
    return float((err / np.maximum(scale, 1e-30)).max())


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float((np.abs(a - b) / np.abs(b)).max())


def assert_close_y(y, ref, dtype, lead=2, what="Y"):
    e = slice_rel(y, ref, lead)
    assert np.all(np.isfinite(y)), f"{what}: non-finite values"
    assert e <= TOL_Y[dtype], f"{what}: slice-relative error {e:.3e} > {TOL_Y[dtype]}"
    return e


def assert_close_den(den, ref, dtype, what="den"):
    e = rel(den, ref)
    assert e <= TOL_DEN[dtype], f"{what}: relative error {e:.3e} > {TOL_DEN[dtype]}"
    return e
