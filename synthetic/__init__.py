"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This module only draws random numbers and converts them to storage formats; it
holds none of the verify round's arithmetic.  Both the CUDA path and the CPU
oracle consume what it returns, byte for byte.

Distributions (the workload descriptions this library is measured on):

* packed codes: uniform random uint32 words, so every 4- or 8-bit code field is
  uniform over its range;
* scales ~ U[lo, hi] and biases ~ N(0, sigma), stored fp16;
* activations ~ N(0, 1), stored bf16;
* target logits ~ N(0, 2) fp32 and draft probabilities
  q = softmax(logits + N(0, 1)) (the draft sees a noisy copy of the target);
* drafts: sampled from q, or equal to the target argmax with a fixed
  probability and otherwise a uniformly drawn other token.

Everything comes from numpy's PCG64 with an explicit seed (host side) or from a
seeded ``torch.Generator`` on the device for the multi-GB weight sets.
"""

import numpy as np

GROUP = 64

# Per-workload weight statistics: (scale_lo, scale_hi, bias_sigma[, centre]).
# With a centre c the bias is -c * scale + N(0, bias_sigma): the affine form
# of a quantiser whose group minimum sits c scales below zero, so codes are
# centred on zero.  The 2-bit tiny workload uses it: with free N(0, 0.05)
# biases a 2-bit row would be dominated by the biases' group sums.
TINY_4BIT = (0.005, 0.02, 0.05)
TINY_2BIT = (0.005, 0.02, 0.002, 1.5)
LARGE_8BIT = (1e-4, 4e-4, 0.02)


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _bf16_bits(x):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def quant_weight(r, N, K, bits, stats):
    """Host arrays {'wq', 'scales', 'biases', 'K', 'bits'} for an N x K weight."""
    lo, hi, sigma = stats[:3]
    centre = stats[3] if len(stats) > 3 else 0.0
    wq = r.integers(0, 2 ** 32, size=(N, K * bits // 32), dtype=np.uint32)
    s16 = r.uniform(lo, hi, size=(N, K // GROUP)).astype(np.float16)
    scales = s16.view(np.uint16)
    biases = (r.standard_normal((N, K // GROUP)) * sigma - centre * s16.astype(np.float64)).astype(
        np.float16).view(np.uint16)
    return {"wq": wq, "scales": scales, "biases": biases, "K": K, "bits": bits}


def activations(r, M, K, sigma=1.0):
    """bf16 bits [M, K], N(0, sigma^2)."""
    return _bf16_bits(r.standard_normal((M, K)) * sigma)


def logits_and_draft_probs(r, m, V, logit_sigma=2.0, noise_sigma=1.0):
    """Target logits fp32 [m + 1, V] and draft probabilities fp32 [m, V]."""
    import torch
    z = (r.standard_normal((m + 1, V)) * logit_sigma).astype(np.float32)
    noisy = torch.from_numpy(z[:m].astype(np.float64) + r.standard_normal((m, V)) * noise_sigma)
    q = torch.softmax(noisy, dim=1).to(torch.float32).numpy()
    return z, q


def sample_drafts(r, q):
    """One token per row of q (fp32 probabilities), by numpy's categorical draw."""
    out = []
    for row in np.asarray(q, dtype=np.float64):
        out.append(int(r.choice(row.shape[0], p=row / row.sum())))
    return np.asarray(out, dtype=np.int32)


def agreeing_drafts(r, target_tokens, V, agree_prob=0.7):
    """draft[i] = target_tokens[i] with probability agree_prob, else another token."""
    out = []
    for t in target_tokens:
        if r.random() < agree_prob:
            out.append(int(t))
        else:
            o = int(r.integers(0, V - 1))
            out.append(o if o < int(t) else o + 1)
    return np.asarray(out, dtype=np.int32)


def accept_uniforms(r, n):
    """fp32 uniforms in [0, 1) for tests that feed u directly."""
    return r.random(n).astype(np.float32)


# ---------------------------------------------------------------- device side

def device_quant_weight(gen, N, K, bits, stats, device="cuda"):
    """Same distributions as ``quant_weight`` drawn on the device (torch tensors).

    Codes: int32 words reinterpreted as uint32 (uniform bit patterns).  Scales
    and biases are drawn in fp32 and stored as fp16.
    """
    import torch
    lo, hi, sigma = stats[:3]
    centre = stats[3] if len(stats) > 3 else 0.0
    wq = torch.randint(-2 ** 31, 2 ** 31, (N, K * bits // 32), generator=gen,
                       dtype=torch.int32, device=device)
    scales = (torch.rand((N, K // GROUP), generator=gen, device=device) * (hi - lo) + lo).to(torch.float16)
    biases = (torch.randn((N, K // GROUP), generator=gen, device=device) * sigma
              - centre * scales.float()).to(torch.float16)
    return {"wq": wq, "scales": scales, "biases": biases, "K": K, "bits": bits}


def device_activations(gen, M, K, device="cuda"):
    import torch
    return torch.randn((M, K), generator=gen, device=device).to(torch.bfloat16)
