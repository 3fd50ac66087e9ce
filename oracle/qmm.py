"""The verify matmul and the vocab head, as plain definitions.

mlx-dspark wiki page, "Architecture": each round the target runs the anchor
token plus m draft tokens through one forward, so every linear layer sees an
activation block of M = 1 + m rows, and the draft is compared against the
target's own logits.  "Key techniques" on the same page describes the verify
kernel as a few-row quantized matmul.  Here that matmul is its definition:

    Y[m, n] = sum_k X[m, k] * w_hat[n, k]

with w_hat from ``quant.dequantize`` (fp32), the products and the sum taken in
fp64, the fp64 result rounded once to fp32 and then (for hidden projections)
once more to bf16.  The vocab head keeps the fp32 logits [reading: the accept
step consumes fp32 logits] and adds, per row, the max, the lowest index that
attains it, and sum_k exp((z_k - max) / T) in fp64.
"""

import numpy as np

from .quant import bf16_bits_to_f32, dequantize, f32_to_bf16_bits, GROUP


def _check_x(x_bf16, K):
    x = np.asarray(x_bf16, dtype=np.uint16)
    if x.ndim != 2 or x.shape[1] != K:
        raise ValueError("x must be bf16 bits [M, K]")
    return bf16_bits_to_f32(x)


def qmm_f32(wq, scales, biases, K, bits, x_bf16, group=GROUP):
    """fp32 [M, N]: fp64 sum of fp32 products X * w_hat, rounded once to fp32."""
    w_hat = dequantize(wq, scales, biases, K, bits, group)
    x = _check_x(x_bf16, K)
    y64 = x.astype(np.float64) @ w_hat.astype(np.float64).T
    return y64.astype(np.float32)


def qmm_verify(wq, scales, biases, K, bits, x_bf16, group=GROUP):
    """bf16 bits [M, N] of one verify projection (rounded to nearest even)."""
    return f32_to_bf16_bits(qmm_f32(wq, scales, biases, K, bits, x_bf16, group))


def row_stats(logits, temperature):
    """Per row of fp32 logits: (max fp32, argmax int64, sumexp fp64).

    argmax is the lowest index attaining the row maximum [reading: ties go to
    the lowest index].  sumexp = sum_k exp((z_k - max) / T) in fp64; for
    T == 0 (greedy) it is not defined and returned as NaN.
    """
    z = np.asarray(logits, dtype=np.float32)
    zmax = z.max(axis=1)
    argmax = np.argmax(z, axis=1)      # numpy returns the first maximal index
    if temperature > 0:
        d = (z.astype(np.float64) - zmax.astype(np.float64)[:, None]) / float(temperature)
        sumexp = np.exp(d).sum(axis=1)
    else:
        sumexp = np.full(z.shape[0], np.nan)
    return zmax, argmax.astype(np.int64), sumexp


def lm_head_verify(wq, scales, biases, K, bits, x_bf16, temperature, group=GROUP):
    """Vocab head of the round: fp32 logits [M, V] plus their per-row stats."""
    logits = qmm_f32(wq, scales, biases, K, bits, x_bf16, group)
    zmax, argmax, sumexp = row_stats(logits, temperature)
    return logits, zmax, argmax, sumexp


def target_probs(logits_row, temperature):
    """p = softmax(z / T) of one fp32 logits row, in fp64."""
    z = np.asarray(logits_row, dtype=np.float64)
    e = np.exp((z - z.max()) / float(temperature))
    return e / e.sum()


def gather_qmm(experts, x_bf16, pair_rows, pair_experts):
    """bf16 [P, N]: row p = X[pair_rows[p]] times expert pair_experts[p]'s weight.

    mlx-dspark PyPI page, "Results at a glance" (MoE rows): each verify row
    selects its own experts.  ``experts`` is a list of E weight dicts
    ``{"wq", "scales", "biases", "K", "bits"}`` of the same shape; every pair is
    the plain verify matmul of one activation row with one expert."""
    x = np.asarray(x_bf16, dtype=np.uint16)
    out = []
    for r, e in zip(pair_rows, pair_experts):
        w = experts[int(e)]
        out.append(qmm_verify(w["wq"], w["scales"], w["biases"], w["K"], w["bits"], x[int(r):int(r) + 1])[0])
    return np.stack(out)
