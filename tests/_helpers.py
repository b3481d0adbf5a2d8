"""Test helpers: bit-exact views of device/host tensors as fp64 for the oracle."""

import numpy as np
import torch

from oracle import codecs


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 value of every element of a bf16 / e4m3 / f32 tensor."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return codecs.bf16_to_f64(t.view(torch.int16).numpy())
    if t.dtype == torch.float8_e4m3fn:
        return codecs.e4m3_to_f64(t.view(torch.uint8).numpy())
    if t.dtype in (torch.float32, torch.float64):
        return t.numpy().astype(np.float64)
    raise TypeError(t.dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int32).numpy()


def max_abs(a, b, mask=None):
    d = np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))
    if mask is not None:
        d = d[mask]
    return float(d.max()) if d.size else 0.0


def gemm_tolerance(ref, abs_sum):
    """Bound for a bf16-output GEMM with fp32 accumulation: half a bf16 ulp of
    the result (2^-9 relative, 2^-8 used for margin) plus K-term fp32
    accumulation error (<= 2^-20 of the sum of |products| for K <= 512)."""
    return np.abs(ref) * 2.0 ** -8 + abs_sum * 2.0 ** -20 + 1e-30


def lse_close(gpu, ref, tol):
    g, r = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    both_inf = np.isneginf(g) & np.isneginf(r)
    d = np.where(both_inf, 0.0, np.abs(g - r))
    return float(np.nanmax(d)) if d.size else 0.0, bool(np.all(~np.isnan(d)))
