"""Pins for the weight format, the 16-bit conversions and the verify matmul oracle."""

import numpy as np
import pytest
import torch

from oracle import quant, qmm
import synthetic


def test_unpack_hand_words_8bit():
    # LSB-first: the low byte of a word is element k = 0.
    wq = np.array([[0x44332211, 0x000000FF]], dtype=np.uint32)
    assert quant.unpack_codes(wq, 8, 8).tolist() == [[0x11, 0x22, 0x33, 0x44, 0xFF, 0, 0, 0]]


def test_unpack_hand_words_4bit():
    wq = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert quant.unpack_codes(wq, 16, 4).tolist() == [list(range(16))]


def test_unpack_hand_words_2bit():
    # 0xE4 = 11 10 01 00: fields 0..3 of a byte, least significant first
    wq = np.array([[0xE4E4E4E4, 0x0000001B]], dtype=np.uint32)
    assert quant.unpack_codes(wq, 32, 2).tolist() == [[0, 1, 2, 3] * 4 + [3, 2, 1, 0] + [0] * 12]


def test_pack_is_inverse_of_unpack():
    r = synthetic.rng(1)
    for bits in (2, 4, 8):
        codes = r.integers(0, 1 << bits, size=(5, 128)).astype(np.uint8)
        assert np.array_equal(quant.unpack_codes(quant.pack_codes(codes, bits), 128, bits), codes)


def test_bf16_rounding_matches_torch():
    r = synthetic.rng(2)
    x = np.concatenate([
        r.standard_normal(20000).astype(np.float32) * 100,
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -3e-39, 3.4e38, 1.0 + 2 ** -8,
                  1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, 65504.0], dtype=np.float32),
        # exact ties between two bf16 neighbours
        (np.arange(1, 200, dtype=np.float32) * 2 ** -8 + 1).astype(np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(quant.f32_to_bf16_bits(x), ref)
    back = quant.bf16_bits_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_dequant_group_index_and_affine_form():
    # codes 1 everywhere, scale of group g = g + 1, bias 0  ->  w_hat[n, k] = k // 64 + 1
    K = 256
    codes = np.ones((3, K), dtype=np.uint8)
    s = np.tile(np.arange(1, K // 64 + 1, dtype=np.float16), (3, 1)).view(np.uint16)
    b = np.zeros((3, K // 64), dtype=np.float16).view(np.uint16)
    for bits in (4, 8):
        w = quant.dequantize(quant.pack_codes(codes, bits), s, b, K, bits)
        assert np.array_equal(w, np.tile(np.arange(K) // 64 + 1, (3, 1)).astype(np.float32))
    # scale 0  ->  w_hat = bias of the group, whatever the codes
    r = synthetic.rng(3)
    codes = r.integers(0, 256, size=(3, K)).astype(np.uint8)
    b = (r.standard_normal((3, K // 64))).astype(np.float16)
    w = quant.dequantize(quant.pack_codes(codes, 8), np.zeros_like(b).view(np.uint16), b.view(np.uint16), K, 8)
    assert np.array_equal(w, np.repeat(b.astype(np.float32), 64, axis=1))


def test_qmm_hand_example():
    # X = ones(1, 64); codes[n, k] = k % 16; s = 1; b = 0 -> Y = sum_k (k % 16) = 4 * 120 = 480;
    # with b = 0.5 the 64 biases add 32 -> 512.  Both are exact in bf16.
    codes = np.tile(np.arange(64) % 16, (2, 1)).astype(np.uint8)
    x = quant.f32_to_bf16_bits(np.ones((1, 64), dtype=np.float32))
    one = np.ones((2, 1), dtype=np.float16).view(np.uint16)
    for bits in (4, 8):
        wq = quant.pack_codes(codes, bits)
        y = qmm.qmm_verify(wq, one, np.zeros((2, 1), np.float16).view(np.uint16), 64, bits, x)
        assert quant.bf16_bits_to_f32(y).tolist() == [[480.0, 480.0]]
        y = qmm.qmm_verify(wq, one, np.full((2, 1), 0.5, np.float16).view(np.uint16), 64, bits, x)
        assert quant.bf16_bits_to_f32(y).tolist() == [[512.0, 512.0]]


def test_qmm_codes_zero_closed_form():
    # all codes 0 -> Y[m, n] = sum_g bias[n, g] * sum_{k in g} x[m, k]
    r = synthetic.rng(4)
    N, K, M = 7, 320, 3
    b = (r.standard_normal((N, K // 64)) * 0.1).astype(np.float16)
    s = r.uniform(0.1, 0.2, (N, K // 64)).astype(np.float16)
    x = synthetic.activations(r, M, K)
    wq = np.zeros((N, K // 4), dtype=np.uint32)
    y = qmm.qmm_f32(wq, s.view(np.uint16), b.view(np.uint16), K, 8, x)
    xs = quant.bf16_bits_to_f32(x).astype(np.float64).reshape(M, K // 64, 64).sum(axis=2)
    expect = xs @ b.astype(np.float64).T
    assert np.allclose(y, expect, rtol=1e-6, atol=1e-6)


def test_qmm_one_hot_rows_select_weight_columns():
    # X row m = e_{k_m}  ->  Y[m, :] = w_hat[:, k_m]; N != K catches a transposed operand.
    r = synthetic.rng(5)
    N, K = 5, 192
    for bits in (4, 8):
        w = synthetic.quant_weight(r, N, K, bits, synthetic.TINY_4BIT)
        ks = [0, 63, 64, 130, 191]
        x = np.zeros((len(ks), K), dtype=np.float32)
        for m, k in enumerate(ks):
            x[m, k] = 1.0
        y = qmm.qmm_f32(w["wq"], w["scales"], w["biases"], K, bits, quant.f32_to_bf16_bits(x))
        per_word = 32 // bits
        for m, k in enumerate(ks):
            for n in range(N):
                word = int(w["wq"][n, k // per_word])
                code = (word >> ((k % per_word) * bits)) & ((1 << bits) - 1)
                s = np.float32(np.uint16(w["scales"][n, k // 64]).view(np.float16))
                b = np.float32(np.uint16(w["biases"][n, k // 64]).view(np.float16))
                assert y[m, n] == np.float32(np.float32(s * np.float32(code)) + b)


def test_qmm_4bit_and_8bit_packings_agree():
    r = synthetic.rng(6)
    N, K, M = 9, 256, 4
    codes = r.integers(0, 16, size=(N, K)).astype(np.uint8)
    s = r.uniform(0.005, 0.02, (N, K // 64)).astype(np.float16).view(np.uint16)
    b = (r.standard_normal((N, K // 64)) * 0.05).astype(np.float16).view(np.uint16)
    x = synthetic.activations(r, M, K)
    y4 = qmm.qmm_verify(quant.pack_codes(codes, 4), s, b, K, 4, x)
    y8 = qmm.qmm_verify(quant.pack_codes(codes, 8), s, b, K, 8, x)
    assert np.array_equal(y4, y8)
    c2 = codes & 3                                 # codes that fit 2 bits: all three packings agree
    y2 = qmm.qmm_verify(quant.pack_codes(c2, 2), s, b, K, 2, x)
    assert np.array_equal(y2, qmm.qmm_verify(quant.pack_codes(c2, 8), s, b, K, 8, x))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qmm_brute_force_tiny(bits):
    r = synthetic.rng(7 + bits)
    N, K, M = 3, 128, 2
    w = synthetic.quant_weight(r, N, K, bits, synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, K)
    y = qmm.qmm_f32(w["wq"], w["scales"], w["biases"], K, bits, x)
    codes = quant.unpack_codes(w["wq"], K, bits)
    xf = quant.bf16_bits_to_f32(x)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                s = float(np.uint16(w["scales"][n, k // 64]).view(np.float16))
                b = float(np.uint16(w["biases"][n, k // 64]).view(np.float16))
                wk = np.float32(np.float32(np.float32(s) * np.float32(codes[n, k])) + np.float32(b))
                acc += float(xf[m, k]) * float(wk)
            assert y[m, n] == np.float32(acc)


def test_qmm_rows_are_independent_and_linear():
    r = synthetic.rng(11)
    N, K = 40, 512
    w = synthetic.quant_weight(r, N, K, 8, synthetic.LARGE_8BIT)
    x = synthetic.activations(r, 6, K)
    y = qmm.qmm_f32(w["wq"], w["scales"], w["biases"], K, 8, x)
    for m in range(6):
        ym = qmm.qmm_f32(w["wq"], w["scales"], w["biases"], K, 8, x[m:m + 1])
        assert np.allclose(ym[0], y[m], rtol=1e-6, atol=1e-7)
    # Y(-X) = -Y(X): negating a bf16 flips its sign bit exactly
    yn = qmm.qmm_f32(w["wq"], w["scales"], w["biases"], K, 8, x ^ np.uint16(0x8000))
    assert np.array_equal(yn, -y)


def test_gather_qmm_pairs_are_independent_verify_matmuls():
    r = synthetic.rng(12)
    E, N, K, M = 5, 24, 128, 4
    experts = [synthetic.quant_weight(r, N, K, 4, synthetic.TINY_4BIT) for _ in range(E)]
    x = synthetic.activations(r, M, K)
    rows = np.array([0, 0, 1, 3, 2, 3, 0])
    exps = np.array([4, 1, 1, 0, 4, 4, 2])
    y = qmm.gather_qmm(experts, x, rows, exps)
    assert y.shape == (len(rows), N)
    # one expert and the identity routing is the plain verify matmul
    w = experts[1]
    assert np.array_equal(qmm.gather_qmm(experts, x, np.arange(M), np.full(M, 1)),
                          qmm.qmm_verify(w["wq"], w["scales"], w["biases"], K, 4, x))
    # a pair's result depends only on its own (row, expert): permuting the pairs permutes the rows
    perm = r.permutation(len(rows))
    assert np.array_equal(qmm.gather_qmm(experts, x, rows[perm], exps[perm]), y[perm])
    # brute force on one pair from the dequantized expert
    wh = quant.dequantize(experts[4]["wq"], experts[4]["scales"], experts[4]["biases"], K, 4).astype(np.float64)
    want = quant.f32_to_bf16_bits((quant.bf16_bits_to_f32(x[2]).astype(np.float64) @ wh.T).astype(np.float32))
    assert np.array_equal(y[4], want)
