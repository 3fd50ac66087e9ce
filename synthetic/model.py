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


def interleave_gate_up(gate, up, block=64):
    """gate | up rows interleaved in blocks of 64 (the round's gate_up layout)."""
    I = gate["wq"].shape[0]

    def inter(a, b):
        a = np.asarray(a).reshape(I // block, block, -1)
        b = np.asarray(b).reshape(I // block, block, -1)
        return np.ascontiguousarray(np.stack([a, b], axis=1).reshape(2 * I, -1))
    return {"wq": inter(gate["wq"], up["wq"]), "scales": inter(gate["scales"], up["scales"]),
            "biases": inter(gate["biases"], up["biases"]), "K": gate["K"], "bits": gate["bits"]}


def device_layers(layers):
    return [{"qkv": to_device(_stack([l["q"], l["k"], l["v"]])), "o": to_device(l["o"]),
             "gate_up": to_device(interleave_gate_up(l["gate"], l["up"])), "down": to_device(l["down"])}
            for l in layers]


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


def split_device_layer(dl, q_dim, kv_dim, inter, block=64):
    """Host per-projection dicts of one stacked device layer (gate/up de-interleaved)."""
    gu = host_copy(dl["gate_up"])
    blk = (np.arange(2 * inter) // block) % 2
    pick = lambda sel: {k: (v[blk == sel] if k in ("wq", "scales", "biases") else v) for k, v in gu.items()}
    return {"q": host_copy(dl["qkv"], (0, q_dim)), "k": host_copy(dl["qkv"], (q_dim, q_dim + kv_dim)),
            "v": host_copy(dl["qkv"], (q_dim + kv_dim, q_dim + 2 * kv_dim)), "o": host_copy(dl["o"]),
            "gate": pick(0), "up": pick(1), "down": host_copy(dl["down"])}
