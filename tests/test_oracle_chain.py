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


# ---------------------------------------------------------------------------
# Wiring of the layer body and of the round, pinned by closed forms computed
# here from the layer description (RMSNorm -> q -> o -> residual -> RMSNorm ->
# gate / up -> SwiGLU -> down -> residual; final RMSNorm -> head), not by
# calling the oracle's own layer code.  Weights are built so every projection
# has a closed form: a scaled identity (codes one-hot, scale c, bias 0) gives
# c * x exactly; a bias-only weight (codes 0, scale 0, bias beta) gives
# beta * sum_k x[k] in every output column.

EPS = 1e-6


def _bf16(v64):
    """fp64 -> fp32 -> bf16 bits: one rounding to fp32, then one to bf16."""
    return quant.f32_to_bf16_bits(np.asarray(v64, np.float64).astype(np.float32))


def _f(b):
    return quant.bf16_bits_to_f32(b).astype(np.float64)


def _fp16_bits(v, shape):
    return np.full(shape, v, np.float16).view(np.uint16)


def _identity(N, K, c, bits=8):
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), np.arange(N) % K] = 1
    return {"wq": quant.pack_codes(codes, bits), "scales": _fp16_bits(c, (N, K // 64)),
            "biases": _fp16_bits(0.0, (N, K // 64)), "K": K, "bits": bits}


def _bias_only(N, K, beta, bits=8):
    return {"wq": np.zeros((N, K * bits // 32), np.uint32), "scales": _fp16_bits(0.0, (N, K // 64)),
            "biases": _fp16_bits(beta, (N, K // 64)), "K": K, "bits": bits}


def _rms(x64):
    return _bf16(x64 / np.sqrt((x64 * x64).mean(axis=1, keepdims=True) + EPS))


def _r(x64):
    """RMSNorm row factor 1 / sqrt(mean(x^2) + eps) (fp64): the layer folds it
    into the consuming projection's output, one rounding per output."""
    return 1.0 / np.sqrt((x64 * x64).mean(axis=1, keepdims=True) + EPS)


C_Q, C_K, C_V, C_O = 2.0, 4.0, 8.0, 0.25
B_G, B_U, B_D = 0.25, -0.5, 0.125


def _wired_layer(H):
    # q, k, v all H x H so that o could (wrongly) take any of them or the
    # normalized input itself: each choice gives a different multiple of a
    return {"q": _identity(H, H, C_Q), "k": _identity(H, H, C_K), "v": _identity(H, H, C_V),
            "o": _identity(H, H, C_O), "gate": _bias_only(H, H, B_G), "up": _bias_only(H, H, B_U),
            "down": _bias_only(H, H, B_D)}


def _wired_layer_by_hand(h_bits):
    """The layer body written out for the weights of ``_wired_layer``."""
    x = _f(h_bits)
    q = _bf16(C_Q * x * _r(x))                         # q = c_q * RMSNorm(h)
    o = _bf16(C_O * _f(q))                             # o is fed by q
    hm = _bf16(x + _f(o))                              # first residual
    x2 = _f(hm)                                        # second RMSNorm, of the updated h
    sigma = x2.sum(axis=1, keepdims=True)              # exact in fp64 for these bf16 rows
    H = x.shape[1]
    g = _bf16(np.repeat(B_G * sigma * _r(x2), H, axis=1))   # gate = beta_g * sum(RMSNorm(hm))
    u = _bf16(np.repeat(B_U * sigma * _r(x2), H, axis=1))   # up = beta_u * sum(RMSNorm(hm))
    gf, uf = _f(g), _f(u)
    s = _bf16(gf / (1.0 + np.exp(-gf)) * uf)          # SwiGLU: silu(gate) * up
    d = _bf16(np.repeat(B_D * _f(s).sum(axis=1, keepdims=True), H, axis=1))
    return _bf16(_f(hm) + _f(d))                       # second residual


def test_layer_wiring_closed_form():
    r = synthetic.rng(90)
    H = 128
    h = synthetic.activations(r, 5, H, sigma=3.0)
    want = _wired_layer_by_hand(h)
    got = chain.layer_forward(h, _wired_layer(H))
    assert np.array_equal(got, want)


def test_layer_wiring_closed_form_catches_planted_mistakes():
    """Each plausible wiring mistake, applied to the hand formula, changes the
    result for these weights: the closed form above tells them apart."""
    r = synthetic.rng(91)
    H = 128
    h = synthetic.activations(r, 4, H, sigma=3.0)
    ref = _wired_layer_by_hand(h)
    x = _f(h)
    a = _rms(x)

    def tail(hm, mlp_in, swap=False, keep_residual=True):
        x2 = _f(mlp_in)
        sigma = x2.sum(axis=1, keepdims=True)
        g = _f(_bf16(np.repeat(B_G * sigma * _r(x2), H, axis=1)))
        u = _f(_bf16(np.repeat(B_U * sigma * _r(x2), H, axis=1)))
        if swap:
            g, u = u, g
        s = _bf16(g / (1.0 + np.exp(-g)) * u)
        d = _bf16(np.repeat(B_D * _f(s).sum(axis=1, keepdims=True), H, axis=1))
        return _bf16((_f(hm) if keep_residual else 0.0) + _f(d))

    def hm_with(o_input_scale):
        return _bf16(x + _f(_bf16(C_O * _f(_bf16(o_input_scale * _f(a))))))

    hm = hm_with(C_Q)
    assert np.array_equal(tail(hm, hm), ref)          # the helper reproduces the closed form
    mistakes = {
        "o fed by the normalized input": tail(hm_with(1.0), hm_with(1.0)),
        "o fed by k": tail(hm_with(C_K), hm_with(C_K)),
        "o fed by v": tail(hm_with(C_V), hm_with(C_V)),
        "gate/up fed by the layer input": tail(hm, h),
        "gate/up fed by the stored first RMSNorm": tail(hm, a),
        "SwiGLU as silu(up) * gate": tail(hm, hm, swap=True),
        "second residual dropped": tail(hm, hm, keep_residual=False),
        "first residual dropped": tail(_bf16(_f(_bf16(C_O * C_Q * _f(a)))), _bf16(_f(_bf16(C_O * C_Q * _f(a))))),
    }
    for name, wrong in mistakes.items():
        assert not np.array_equal(wrong, ref), name


def _selector_head(V, H, c):
    """Head row v picks hidden column v % H, scaled by c (a one-hot selector)."""
    codes = np.zeros((V, H), np.uint8)
    codes[np.arange(V), np.arange(V) % H] = 1
    return {"wq": quant.pack_codes(codes, 8), "scales": _fp16_bits(c, (V, H // 64)),
            "biases": _fp16_bits(0.0, (V, H // 64)), "K": H, "bits": 8}


def test_round_logits_chain_and_final_norm_closed_form():
    r = synthetic.rng(92)
    H, V, c = 128, 192, 2.0
    h0 = synthetic.activations(r, 3, H, sigma=3.0)
    layers = [_wired_layer(H), _wired_layer(H)]
    h1 = _wired_layer_by_hand(h0)
    h2 = _wired_layer_by_hand(h1)                     # layers applied in order, each feeding the next
    x = _f(h2)
    want = (c * x[:, np.arange(V) % H] * _r(x)).astype(np.float32)   # final RMSNorm before the head
    hs, logits, zmax, argmax, sumexp = chain.round_logits(h0, layers, _selector_head(V, H, c), 0.7)
    assert len(hs) == 2 and np.array_equal(hs[0], h1) and np.array_equal(hs[1], h2)
    assert logits.dtype == np.float32 and np.array_equal(logits, want)
    assert np.array_equal(zmax, want.max(axis=1))
    assert np.array_equal(argmax, np.argmax(want, axis=1))   # ties: lowest index
    d = (want.astype(np.float64) - want.max(axis=1, keepdims=True)) / 0.7
    assert np.allclose(sumexp, np.exp(d).sum(axis=1), rtol=1e-12)
    # without the final RMSNorm the logits would be c * h2: a different result
    assert not np.array_equal((c * x[:, np.arange(V) % H]).astype(np.float32), want)


def test_verify_round_greedy_closed_form():
    r = synthetic.rng(93)
    H, V, c = 128, 128, 2.0
    h0 = synthetic.activations(r, 4, H, sigma=3.0)
    layers = [_wired_layer(H)]
    x = _f(_wired_layer_by_hand(h0))
    a = c * x * _r(x)
    target = np.argmax(a.astype(np.float32), axis=1)
    draft = target[:3].astype(np.int32).copy()
    draft[2] = (draft[2] + 1) % V                     # first mismatch at position 2
    out_len, tokens, logits = chain.verify_round(h0, layers, _selector_head(V, H, c), 0.0, draft)
    assert out_len == 3 and list(tokens) == [int(draft[0]), int(draft[1]), int(target[2])]
    assert np.array_equal(logits, a.astype(np.float32))
