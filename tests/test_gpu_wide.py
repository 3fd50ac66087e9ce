"""Wide blocks (33..512 rows) through sv_qmm_verify: the tensor-memory kernel
against the CPU oracle.  Weight rows are independent, so the large shapes are
checked on a sampled subset of output columns (each computed by the oracle in
full); the small ones everywhere."""

import numpy as np
import pytest
import torch

from oracle import qmm as oq, quant
import synthetic
from tests._util import assert_close_bf16, dev_bf16, dev_weight, host_f32_of_bf16, sub_weight

pytestmark = pytest.mark.gpu

STATS = {2: synthetic.TINY_2BIT, 4: synthetic.TINY_4BIT, 8: synthetic.LARGE_8BIT}


def _check(lib, w, x, cols=None, residual=None, what=""):
    dw = dev_weight(w)
    res = dev_bf16(residual) if residual is not None else None
    y = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], w["K"], w["bits"], dev_bf16(x), residual=res)
    torch.cuda.synchronize()
    got = host_f32_of_bf16(y)
    ws = w if cols is None else sub_weight(w, cols)
    want = oq.qmm_f32(ws["wq"], ws["scales"], ws["biases"], w["K"], w["bits"], x)
    if residual is not None:
        r = quant.bf16_bits_to_f32(residual if cols is None else residual[:, cols])
        want = quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(
            r + quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(want))))
    else:
        want = quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(want))
    assert_close_bf16(got if cols is None else got[:, cols], want, what=what)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("M", [33, 48, 64, 100, 128, 256, 257, 300, 512])
def test_wide_small_shape_everywhere(lib, bits, M):
    r = synthetic.rng(1800 + bits + M)
    N, K = 200, 1536                                  # ragged last tile, k split across CTAs
    w = synthetic.quant_weight(r, N, K, bits, STATS[bits])
    x = synthetic.activations(r, M, K)
    _check(lib, w, x, what="wide N=%d K=%d M=%d bits=%d" % (N, K, M, bits))
    assert lib.device_error() == 0


@pytest.mark.parametrize("M", [40, 300])
def test_wide_unaligned_output_rows(lib, M):
    """N = 203: output rows that are not 16-byte aligned take the epilogue's
    element-by-element stores (bf16 output and, with k split across CTAs,
    the fp32 partials).  The product is checked against the oracle; the
    residual form must equal bf16(residual + product) with the GPU's own
    (deterministic) product, element for element."""
    r = synthetic.rng(1970 + M)
    N, K, bits = 203, 2048, 4
    w = synthetic.quant_weight(r, N, K, bits, STATS[bits])
    x = synthetic.activations(r, M, K)
    res = synthetic.activations(r, M, N)
    _check(lib, w, x, what="wide N=203 M=%d" % M)
    dw = dev_weight(w)
    prod = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x))
    y = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), residual=dev_bf16(res))
    torch.cuda.synchronize()
    want = quant.f32_to_bf16_bits(quant.bf16_bits_to_f32(res) + host_f32_of_bf16(prod))
    assert np.array_equal(host_f32_of_bf16(y), quant.bf16_bits_to_f32(want))
    assert lib.device_error() == 0


SHAPES = {  # Qwen3-8B-shaped (8-bit) and 4B-shaped (4-bit) projections
    "8b_q": (4096, 4096, 8), "8b_gate": (12288, 4096, 8), "8b_down": (4096, 12288, 8),
    "4b_q": (4096, 2560, 4), "4b_o": (2560, 4096, 4), "4b_gate": (9728, 2560, 4), "4b_down": (2560, 9728, 4),
}


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("M", [33, 64, 128, 512])
def test_wide_projection_shapes_sampled(lib, name, M):
    N, K, bits = SHAPES[name]
    r = synthetic.rng(1900 + list(SHAPES).index(name) + M)
    w = synthetic.quant_weight(r, N, K, bits, STATS[bits])
    x = synthetic.activations(r, M, K)
    cols = np.unique(np.concatenate([r.choice(N, 192, replace=False), [0, N - 1]]))
    _check(lib, w, x, cols=cols, what="%s M=%d" % (name, M))
    assert lib.device_error() == 0


def test_wide_residual_in_place_and_reproducible(lib):
    """y = bf16(residual + bf16(x w^T)): the product is checked against the oracle
    elsewhere; here the residual form must equal the residual added, in bf16, to
    the GPU's own product (the product path is deterministic), in place too."""
    r = synthetic.rng(1990)
    N, K, M, bits = 640, 2048, 96, 8
    w = synthetic.quant_weight(r, N, K, bits, STATS[bits])
    x = synthetic.activations(r, M, K)
    res = synthetic.activations(r, M, N)
    dw = dev_weight(w)
    prod = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x))
    y1 = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), residual=dev_bf16(res))
    h = dev_bf16(res)
    lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), y=h, residual=h)   # in place
    torch.cuda.synchronize()
    want = quant.f32_to_bf16_bits(quant.bf16_bits_to_f32(res) + host_f32_of_bf16(prod))
    assert np.array_equal(host_f32_of_bf16(y1), quant.bf16_bits_to_f32(want))
    assert torch.equal(h, y1)
    y2 = lib.qmm_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), residual=dev_bf16(res))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)                         # split-k partials are added in a fixed order
    assert lib.device_error() == 0


def test_wide_refuses_beyond_512_rows(lib):
    from speculative_decoding_verify_qmm_gb300.binding import SVError, SV_EUNSUPPORTED
    r = synthetic.rng(1995)
    w = dev_weight(synthetic.quant_weight(r, 64, 512, 8, STATS[8]))
    x = dev_bf16(synthetic.activations(r, 513, 512))
    with pytest.raises(SVError) as e:
        lib.qmm_verify(w["wq"], w["scales"], w["biases"], 512, 8, x, workspace=lib.workspace(1 << 20))
    assert e.value.status == SV_EUNSUPPORTED
