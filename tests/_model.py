"""Synthetic dense quantized models for the round tests and the benchmark.

A model is described once per projection (q, k, v, o, gate, up, down, plus the
vocab head); the device copy stacks q|k|v and gate|up along N exactly as the
library's round layout expects.  Random draws only: no verify arithmetic.
"""

import numpy as np
import torch

import synthetic


def host_model(seed, n_layers, hidden, q_dim, kv_dim, inter, vocab, bits, stats):
    r = synthetic.rng(seed)
    layers = []
    for _ in range(n_layers):
        layers.append({
            "q": synthetic.quant_weight(r, q_dim, hidden, bits, stats),
            "k": synthetic.quant_weight(r, kv_dim, hidden, bits, stats),
            "v": synthetic.quant_weight(r, kv_dim, hidden, bits, stats),
            "o": synthetic.quant_weight(r, hidden, q_dim, bits, stats),
            "gate": synthetic.quant_weight(r, inter, hidden, bits, stats),
            "up": synthetic.quant_weight(r, inter, hidden, bits, stats),
            "down": synthetic.quant_weight(r, hidden, inter, bits, stats),
        })
    head = synthetic.quant_weight(r, vocab, hidden, bits, stats)
    return layers, head


def _stack(ws):
    return {"wq": np.concatenate([w["wq"] for w in ws]), "scales": np.concatenate([w["scales"] for w in ws]),
            "biases": np.concatenate([w["biases"] for w in ws]), "K": ws[0]["K"], "bits": ws[0]["bits"]}


def to_device(w):
    return {"wq": torch.from_numpy(np.ascontiguousarray(w["wq"]).view(np.int32)).cuda(),
            "scales": torch.from_numpy(np.ascontiguousarray(w["scales"]).view(np.float16)).cuda(),
            "biases": torch.from_numpy(np.ascontiguousarray(w["biases"]).view(np.float16)).cuda(),
            "K": w["K"], "bits": w["bits"]}


def device_layers(layers):
    return [{"qkv": to_device(_stack([l["q"], l["k"], l["v"]])), "o": to_device(l["o"]),
             "gate_up": to_device(_stack([l["gate"], l["up"]])), "down": to_device(l["down"])} for l in layers]


def device_random_model(seed, n_layers, hidden, q_dim, kv_dim, inter, vocab, bits, stats):
    """The same distributions drawn directly on the device (for multi-GB models)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    layers = []
    for _ in range(n_layers):
        layers.append({
            "qkv": synthetic.device_quant_weight(gen, q_dim + 2 * kv_dim, hidden, bits, stats),
            "o": synthetic.device_quant_weight(gen, hidden, q_dim, bits, stats),
            "gate_up": synthetic.device_quant_weight(gen, 2 * inter, hidden, bits, stats),
            "down": synthetic.device_quant_weight(gen, hidden, inter, bits, stats),
        })
    head = synthetic.device_quant_weight(gen, vocab, hidden, bits, stats)
    return layers, head


def host_copy(w, rows=None):
    """Device weight dict -> host numpy dict (optionally a row range)."""
    sl = slice(None) if rows is None else slice(*rows)
    return {"wq": w["wq"][sl].cpu().numpy().view(np.uint32), "scales": w["scales"][sl].cpu().numpy().view(np.uint16),
            "biases": w["biases"][sl].cpu().numpy().view(np.uint16), "K": w["K"], "bits": w["bits"]}


def split_device_layer(dl, q_dim, kv_dim, inter):
    """Host per-projection dicts of one stacked device layer."""
    return {"q": host_copy(dl["qkv"], (0, q_dim)), "k": host_copy(dl["qkv"], (q_dim, q_dim + kv_dim)),
            "v": host_copy(dl["qkv"], (q_dim + kv_dim, q_dim + 2 * kv_dim)), "o": host_copy(dl["o"]),
            "gate": host_copy(dl["gate_up"], (0, inter)), "up": host_copy(dl["gate_up"], (inter, 2 * inter)),
            "down": host_copy(dl["down"])}
