"""Philox bit-exactness and glue-kernel parity against the oracle."""

import numpy as np
import pytest
import torch

from oracle import glue, philox
import synthetic
from tests._util import dev_bf16, host_bf16_bits
from oracle import quant

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,sub,off,n", [(0, 0, 0, 16), (1234, 3, 5, 1000), (2 ** 40 + 7, 2 ** 33, 2 ** 35 + 3, 777)])
def test_philox_bit_exact(lib, seed, sub, off, n):
    got = lib.philox_uniforms(seed, sub, off, n).cpu().numpy()
    assert np.array_equal(got, philox.uniforms(seed, sub, off, n))


def _bf16_match(got_bits, want_bits):
    g = quant.bf16_bits_to_f32(got_bits).astype(np.float64)
    w = quant.bf16_bits_to_f32(want_bits).astype(np.float64)
    assert np.all(np.abs(g - w) <= np.abs(w) * 2 ** -7 + 1e-30)
    assert np.mean(got_bits == want_bits) > 0.98


@pytest.mark.parametrize("M,H", [(1, 4096), (8, 4096), (17, 2560), (32, 5120)])
def test_rmsnorm(lib, M, H):
    r = synthetic.rng(1000 + M)
    x = synthetic.activations(r, M, H, 7.0)
    y = lib.rmsnorm(dev_bf16(x))
    torch.cuda.synchronize()
    _bf16_match(host_bf16_bits(y), glue.rmsnorm(x))
    wt = synthetic.activations(r, 1, H)[0]
    y = lib.rmsnorm(dev_bf16(x), weight=dev_bf16(wt))
    torch.cuda.synchronize()
    _bf16_match(host_bf16_bits(y), glue.rmsnorm(x, wt))


@pytest.mark.parametrize("M,I", [(1, 12288), (16, 9728), (32, 17408)])
def test_swiglu_and_residual(lib, M, I):
    r = synthetic.rng(1100 + M)
    g = synthetic.activations(r, M, I, 3.0)
    u = synthetic.activations(r, M, I, 3.0)
    s = lib.swiglu(dev_bf16(g), dev_bf16(u))
    torch.cuda.synchronize()
    _bf16_match(host_bf16_bits(s), glue.swiglu(g, u))
    h = dev_bf16(g).clone()
    lib.residual_add(h, dev_bf16(u))
    torch.cuda.synchronize()
    _bf16_match(host_bf16_bits(h), glue.residual_add(g, u))
    assert lib.device_error() == 0
