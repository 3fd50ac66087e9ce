"""Pins for the verify-round chain: the greedy losslessness invariant on a toy
language model, and closed forms of the layer body."""

import numpy as np
import pytest

from oracle import accept, chain, glue, qmm, quant
import synthetic


class ToyLM:
    """Embedding -> causal running mean -> one quantized layer -> vocab head."""

    def __init__(self, seed, V, H=128, bits=4):
        r = synthetic.rng(seed)
        self.V, self.H = V, H
        self.emb = (r.standard_normal((V, H)) * 1.0).astype(np.float64)
        self.layer = synthetic.quant_weight(r, H, H, bits, synthetic.TINY_4BIT)
        self.head = synthetic.quant_weight(r, V, H, bits, synthetic.TINY_4BIT)

    def rows(self, tokens, positions):
        """Logits rows for the given positions of a token sequence (causal)."""
        h = np.stack([self.emb[tokens[:p + 1]].mean(axis=0) for p in positions])
        h = quant.f32_to_bf16_bits(h.astype(np.float32))
        h = glue.residual_add(h, chain.project(self.layer, glue.rmsnorm(h)))
        a = glue.rmsnorm(h)
        return qmm.qmm_f32(self.head["wq"], self.head["scales"], self.head["biases"],
                           self.H, self.head["bits"], a)

    def greedy(self, prompt, n):
        toks = list(prompt)
        for _ in range(n):
            toks.append(int(np.argmax(self.rows(toks, [len(toks) - 1])[0])))
        return toks[len(prompt):]

    def speculative(self, prompt, n, drafter):
        toks = list(prompt)
        rounds = 0
        while len(toks) - len(prompt) < n:
            draft = drafter(toks)
            ctx = toks + draft
            logits = self.rows(ctx, list(range(len(toks) - 1, len(ctx))))
            _, committed = accept.greedy_accept(logits, draft)
            toks += committed
            rounds += 1
        return toks[len(prompt):len(prompt) + n], rounds


@pytest.mark.parametrize("V", [16, 1000])
def test_speculative_greedy_equals_sequential_greedy(V):
    lm = ToyLM(70 + V, V)
    r = synthetic.rng(71)
    prompt = [int(t) for t in r.integers(0, V, 5)]
    n = 24
    want = lm.greedy(prompt, n)

    def random_drafter(toks):
        return [int(t) for t in r.integers(0, V, int(r.integers(0, 8)))]

    def oracle_drafter(toks):         # perfect drafts, with one planted error half the time
        out = lm.greedy(toks, 6)
        if r.random() < 0.5:
            j = int(r.integers(0, 6))
            out[j] = (out[j] + 1) % V
        return out

    def empty_drafter(toks):
        return []

    for drafter in (random_drafter, oracle_drafter, empty_drafter):
        got, rounds = lm.speculative(prompt, n, drafter)
        assert got == want
    got, rounds = lm.speculative(prompt, n, lambda toks: lm.greedy(toks, 7))
    assert got == want and rounds <= -(-n // 8)   # perfect drafts: 8 tokens per round


def _zero_layer(H, I, Dq, bits):
    def z(N, K):
        return {"wq": np.zeros((N, K * bits // 32), np.uint32),
                "scales": np.zeros((N, K // 64), np.uint16),
                "biases": np.zeros((N, K // 64), np.uint16), "K": K, "bits": bits}
    return {"q": z(Dq, H), "k": z(64, H), "v": z(64, H), "o": z(H, Dq),
            "gate": z(I, H), "up": z(I, H), "down": z(H, I)}


def test_zero_weights_leave_hidden_state_unchanged():
    r = synthetic.rng(80)
    h = synthetic.activations(r, 4, 128)
    out = chain.layer_forward(h, _zero_layer(128, 256, 192, 8))
    assert np.array_equal(out, h)


def test_layer_with_only_o_bias_adds_bias_row_sum_of_q():
    # q = 0 (zero q weights), o has zero codes and bias beta: o(q) = beta * sum(q) = 0,
    # down has bias beta on every group and the MLP input s = silu(0) * 0 = 0 -> h unchanged;
    # now give 'up' bias 1 and 'gate' bias 1: s = silu(sum a2) * sum a2 per column.
    r = synthetic.rng(81)
    H, I = 128, 128
    layer = _zero_layer(H, I, 128, 8)
    one = np.ones((I, H // 64), np.float16).view(np.uint16)
    layer["gate"]["biases"] = one
    layer["up"]["biases"] = one
    h = synthetic.activations(r, 2, H)
    out = chain.layer_forward(h, layer)
    assert np.array_equal(out, h)                  # down is still zero
    a2 = glue.rmsnorm(h)
    rs = quant.bf16_bits_to_f32(a2).astype(np.float64).sum(axis=1)
    g = quant.bf16_bits_to_f32(chain.project(layer["gate"], a2)).astype(np.float64)
    assert np.allclose(g, np.repeat(rs[:, None], I, axis=1), rtol=2 ** -8, atol=1e-6)
