"""Verify-matmul parity: the CUDA path through the C ABI against the CPU oracle."""

import numpy as np
import pytest
import torch

from oracle import qmm as oq
import synthetic
from tests._util import assert_close_bf16, assert_close_rms, dev_bf16, dev_weight, host_f32_of_bf16, host_bf16_bits, sub_weight
from oracle import quant

pytestmark = pytest.mark.gpu


def _run(lib, w, x_bits, residual=None, **kw):
    dw = dev_weight(w)
    x = dev_bf16(x_bits)
    res = dev_bf16(residual) if residual is not None else None
    y = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], w["K"], w["bits"], x, residual=res, **kw)
    torch.cuda.synchronize()
    return y


def _oracle_f32(w, x_bits):
    return quant.bf16_bits_to_f32(oq.qmm_verify(w["wq"], w["scales"], w["biases"], w["K"], w["bits"], x_bits))


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_tiny_4bit_layer(lib, M):
    r = synthetic.rng(100)
    w = synthetic.quant_weight(r, 1024, 1024, 4, synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, 1024)
    y = _run(lib, w, x)
    assert_close_bf16(host_f32_of_bf16(y), _oracle_f32(w, x), what="tiny M=%d" % M)
    assert lib.device_error() == 0


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K", [(1000, 1536), (37, 512), (130, 2048), (64, 4096)])
@pytest.mark.parametrize("M", [1, 3, 9, 17, 24, 32])
def test_ragged_shapes(lib, bits, N, K, M):
    r = synthetic.rng(1000 * bits + N + K + M)
    w = synthetic.quant_weight(r, N, K, bits, {2: synthetic.TINY_2BIT, 4: synthetic.TINY_4BIT, 8: synthetic.LARGE_8BIT}[bits])
    x = synthetic.activations(r, M, K)
    y = _run(lib, w, x)
    assert_close_bf16(host_f32_of_bf16(y), _oracle_f32(w, x), what="N=%d K=%d M=%d" % (N, K, M))


SHAPES_8B = {"q": (4096, 4096), "k": (1024, 4096), "o": (4096, 4096), "gate": (12288, 4096), "down": (4096, 12288)}


@pytest.mark.parametrize("name", list(SHAPES_8B))
def test_qwen3_8b_projection_shapes(lib, name):
    """One-layer 8-bit shapes at every verify width of the sweep (rows are independent)."""
    N, K = SHAPES_8B[name]
    r = synthetic.rng(200 + list(SHAPES_8B).index(name))
    w = synthetic.quant_weight(r, N, K, 8, synthetic.LARGE_8BIT)
    x17 = synthetic.activations(r, 17, K)
    want = _oracle_f32(w, x17)
    for M in (1, 2, 4, 6, 8, 12, 16, 17):
        y = _run(lib, w, x17[:M])
        assert_close_bf16(host_f32_of_bf16(y), want[:M], what="%s M=%d" % (name, M))


def test_residual_in_place_and_strides(lib):
    r = synthetic.rng(7)
    N, K, M = 4096, 4096, 8
    w = synthetic.quant_weight(r, N, K, 8, synthetic.LARGE_8BIT)
    x = synthetic.activations(r, M, K)
    h = synthetic.activations(r, M, N, 4.0)
    dw = dev_weight(w)
    # strided activation (ldx > K) and in-place residual (y aliases h)
    xbig = torch.zeros((M, K + 256), dtype=torch.bfloat16, device="cuda")
    xbig[:, :K] = dev_bf16(x)
    hd = dev_bf16(h).clone()
    lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, 8, xbig[:, :K], y=hd, residual=hd)
    torch.cuda.synchronize()
    t = oq.qmm_verify(w["wq"], w["scales"], w["biases"], K, 8, x)
    from oracle import glue
    want = quant.bf16_bits_to_f32(glue.residual_add(h, t))
    assert_close_bf16(host_f32_of_bf16(hd), want, what="residual")


def test_bitwise_reproducible(lib):
    r = synthetic.rng(8)
    w = synthetic.quant_weight(r, 12288, 4096, 8, synthetic.LARGE_8BIT)
    x = synthetic.activations(r, 16, 4096)
    a = host_bf16_bits(_run(lib, w, x))
    b = host_bf16_bits(_run(lib, w, x))
    assert np.array_equal(a, b)


def test_large_activation_range(lib):
    """Rows with very different magnitudes (the per-row power-of-two scaling)."""
    r = synthetic.rng(9)
    N, K = 256, 2048
    w = synthetic.quant_weight(r, N, K, 8, synthetic.LARGE_8BIT)
    x = r.standard_normal((5, K)).astype(np.float32)
    x *= np.array([1e-12, 1e-3, 1.0, 3e4, 1e20], dtype=np.float32)[:, None]
    xb = quant.f32_to_bf16_bits(x)
    y = host_f32_of_bf16(_run(lib, w, xb))
    want = _oracle_f32(w, xb)
    for m in range(5):
        assert_close_bf16(y[m:m + 1], want[m:m + 1], what="row %d" % m)


def test_host_rejections(lib):
    from speculative_decoding_verify_qmm_gb300.binding import SVError
    r = synthetic.rng(10)
    w = synthetic.quant_weight(r, 128, 1024, 8, synthetic.LARGE_8BIT)
    dw = dev_weight(w)
    x = dev_bf16(synthetic.activations(r, 513, 1024))
    with pytest.raises(SVError) as e:
        lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], 1024, 8, x, workspace=lib.workspace(1 << 20))
    assert e.value.status == 2
    small = lib.workspace(256)
    with pytest.raises(SVError) as e:
        lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], 1024, 8, x[:4], workspace=small)
    assert e.value.status == 1
    assert lib.device_error() == 0
