"""Elementwise and row-wise steps between the verify projections.

The pages give no layer internals for the targets [reading: a Qwen3-style
dense block, with RMSNorm (weight 1.0 unless given), residual adds and a
SwiGLU MLP].  Each function takes and returns bf16 bit patterns; arithmetic
is fp64 with a single rounding to bf16 at the end.
"""

import numpy as np

from .quant import bf16_bits_to_f32, f32_to_bf16_bits

RMS_EPS = 1e-6   # [reading] the usual epsilon of the target family


def _f64(x_bf16):
    return bf16_bits_to_f32(x_bf16).astype(np.float64)


def _to_bf16(y64):
    return f32_to_bf16_bits(np.asarray(y64, dtype=np.float64).astype(np.float32))


def rmsnorm(x_bf16, weight_bf16=None, eps=RMS_EPS):
    """y[m, k] = x[m, k] / sqrt(mean_k x[m, k]^2 + eps) * weight[k]."""
    x = _f64(x_bf16)
    r = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)
    w = 1.0 if weight_bf16 is None else _f64(np.asarray(weight_bf16)[None, :])
    return _to_bf16(x * r * w)


def residual_add(h_bf16, t_bf16):
    """h + t."""
    return _to_bf16(_f64(h_bf16) + _f64(t_bf16))


def silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu(g_bf16, u_bf16):
    """silu(g) * u."""
    g = _f64(g_bf16)
    return _to_bf16(silu(g) * _f64(u_bf16))
