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
"""

from .accept import spec_accept
from .glue import residual_add, rmsnorm, swiglu
from .qmm import lm_head_verify, qmm_verify


def project(p, x_bf16):
    return qmm_verify(p["wq"], p["scales"], p["biases"], p["K"], p["bits"], x_bf16)


def layer_forward(h_bf16, layer):
    """Hidden state bf16 [M, H] after one layer; k and v are computed and unused."""
    a = rmsnorm(h_bf16)
    q = project(layer["q"], a)
    project(layer["k"], a)
    project(layer["v"], a)
    h = residual_add(h_bf16, project(layer["o"], q))
    a2 = rmsnorm(h)
    s = swiglu(project(layer["gate"], a2), project(layer["up"], a2))
    return residual_add(h, project(layer["down"], s))


def round_logits(h0_bf16, layers, head, temperature):
    """Returns (hidden states after each layer, logits, max, argmax, sumexp)."""
    h, hs = h0_bf16, []
    for layer in layers:
        h = layer_forward(h, layer)
        hs.append(h)
    a = rmsnorm(h)
    logits, zmax, argmax, sumexp = lm_head_verify(
        head["wq"], head["scales"], head["biases"], head["K"], head["bits"], a, temperature)
    return hs, logits, zmax, argmax, sumexp


def verify_round(h0_bf16, layers, head, temperature, draft, q=None, u=None):
    """(out_len, tokens, logits) of one full verify round."""
    _, logits, _, _, _ = round_logits(h0_bf16, layers, head, temperature)
    out_len, tokens = spec_accept(logits, q, draft, temperature, u)
    return out_len, tokens, logits
