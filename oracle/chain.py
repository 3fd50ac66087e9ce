"""One verify round through a stack of quantized dense layers.

mlx-dspark wiki page, "Architecture": one target forward over the M = 1 + m
rows [anchor] + drafts, then the accept step.  PyPI page, "The Apple-Silicon
speedup ceiling": verify cost is the quantized matmul over every linear layer.
The layer body is a [reading] (the pages give none): RMSNorm, the q/k/v
projections, the o projection fed by q (no attention: the synthetic workload
has no KV state), residual add, RMSNorm, gate/up projections, SwiGLU, down
projection, residual add; after the last layer a final RMSNorm and the vocab
head.

A projection is a dict ``{"wq", "scales", "biases", "K", "bits"}``; a layer is
a dict with projections ``q, k, v, o, gate, up, down``.

[reading] Each RMSNorm (weight 1.0) is folded into the projections that
consume it: (x / rms(x)) W^T = (x W^T) / rms(x), evaluated in fp64 with one
rounding of the projection's output, so the normalised row itself is never
stored.  That is the round's own contract; a standalone RMSNorm that stores
its output in bf16 is ``glue.rmsnorm``.
"""

import numpy as np

from .accept import spec_accept
from .glue import RMS_EPS, residual_add, swiglu
from .qmm import qmm_verify, row_stats
from .quant import bf16_bits_to_f32, dequantize, f32_to_bf16_bits


def project(p, x_bf16):
    return qmm_verify(p["wq"], p["scales"], p["biases"], p["K"], p["bits"], x_bf16)


def normed_f64(p, h_bf16, eps=RMS_EPS):
    """fp64 (h W^T) / sqrt(mean(h^2) + eps) for bf16 rows h (the RMSNorm of h
    feeding projection p)."""
    x = bf16_bits_to_f32(h_bf16).astype(np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)
    w_hat = dequantize(p["wq"], p["scales"], p["biases"], p["K"], p["bits"]).astype(np.float64)
    return (x @ w_hat.T) * r


def project_normed(p, h_bf16):
    """bf16 output of projection p applied to RMSNorm(h)."""
    return f32_to_bf16_bits(normed_f64(p, h_bf16).astype(np.float32))


def layer_forward(h_bf16, layer):
    """Hidden state bf16 [M, H] after one layer; k and v are computed and unused."""
    q = project_normed(layer["q"], h_bf16)
    project_normed(layer["k"], h_bf16)
    project_normed(layer["v"], h_bf16)
    h = residual_add(h_bf16, project(layer["o"], q))
    s = swiglu(project_normed(layer["gate"], h), project_normed(layer["up"], h))
    return residual_add(h, project(layer["down"], s))


def round_logits(h0_bf16, layers, head, temperature):
    """Returns (hidden states after each layer, logits, max, argmax, sumexp)."""
    h, hs = h0_bf16, []
    for layer in layers:
        h = layer_forward(h, layer)
        hs.append(h)
    logits = normed_f64(head, h).astype(np.float32)      # fp32 logits of the final RMSNorm
    zmax, argmax, sumexp = row_stats(logits, temperature)
    return hs, logits, zmax, argmax, sumexp


def verify_round(h0_bf16, layers, head, temperature, draft, q=None, u=None):
    """(out_len, tokens, logits) of one full verify round."""
    _, logits, _, _, _ = round_logits(h0_bf16, layers, head, temperature)
    out_len, tokens = spec_accept(logits, q, draft, temperature, u)
    return out_len, tokens, logits
