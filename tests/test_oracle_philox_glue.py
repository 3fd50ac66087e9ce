"""Pins for the Philox oracle (published known answers) and the glue oracle."""

import os

import numpy as np
import scipy.stats
import torch

from oracle import glue, philox, quant
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for row in rows:
        v = [int(t, 16) for t in row]
        assert philox.philox4x32_10(v[0:4], v[4:6]) == tuple(v[6:10])


def test_uniform_stream_offsets_and_range():
    a = philox.uniforms(7, 3, 0, 64)
    for i in (0, 1, 5, 33, 63):
        assert philox.uniforms(7, 3, i, 1)[0] == a[i]
    assert not np.array_equal(a, philox.uniforms(7, 4, 0, 64))     # subsequences differ
    assert not np.array_equal(a, philox.uniforms(8, 3, 0, 64))     # seeds differ
    assert a.dtype == np.float32 and (a >= 0).all() and (a < 1).all()
    # the word-to-float map: u * 2^24 is the integer x >> 8
    assert np.array_equal(a * 2 ** 24, np.floor(a * 2 ** 24))


def test_uniforms_chi_square():
    u = philox.uniforms(1234, 0, 0, 40000)
    counts = np.histogram(u, bins=40, range=(0, 1))[0]
    assert scipy.stats.chisquare(counts).pvalue > 1e-3


def test_rmsnorm_matches_torch_and_closed_form():
    r = synthetic.rng(60)
    x = synthetic.activations(r, 5, 300)
    got = quant.bf16_bits_to_f32(glue.rmsnorm(x)).astype(np.float64)
    xt = torch.from_numpy(quant.bf16_bits_to_f32(x).astype(np.float64))
    ref = torch.nn.functional.rms_norm(xt, (300,), eps=glue.RMS_EPS).numpy()
    assert np.allclose(got, ref, rtol=2 ** -8, atol=0)
    # constant row c: every output is sign(c) / sqrt(1 + eps / c^2)
    c = quant.f32_to_bf16_bits(np.full((1, 64), -3.0, np.float32))
    y = quant.bf16_bits_to_f32(glue.rmsnorm(c))
    assert np.all(y == quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(np.float32(-1 / np.sqrt(1 + 1e-6 / 9)))))
    w = quant.f32_to_bf16_bits(np.linspace(0.5, 2, 64).astype(np.float32))
    yw = quant.bf16_bits_to_f32(glue.rmsnorm(c, w)).astype(np.float64)
    assert np.allclose(yw, -quant.bf16_bits_to_f32(w), rtol=2 ** -8)


def test_swiglu_and_residual():
    r = synthetic.rng(61)
    g = synthetic.activations(r, 3, 128, 3.0)
    u = synthetic.activations(r, 3, 128, 3.0)
    got = quant.bf16_bits_to_f32(glue.swiglu(g, u)).astype(np.float64)
    gt = torch.from_numpy(quant.bf16_bits_to_f32(g).astype(np.float64))
    ref = (torch.nn.functional.silu(gt) * torch.from_numpy(quant.bf16_bits_to_f32(u).astype(np.float64))).numpy()
    assert np.allclose(got, ref, rtol=2 ** -8, atol=1e-30)
    h = glue.residual_add(g, u)
    assert np.array_equal(h, quant.f32_to_bf16_bits(quant.bf16_bits_to_f32(g) + quant.bf16_bits_to_f32(u)))
