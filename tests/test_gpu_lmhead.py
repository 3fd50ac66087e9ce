"""Vocab-head parity: logits against the oracle, row statistics exact on the GPU's logits."""

import numpy as np
import pytest
import torch

from oracle import qmm as oq
from oracle import quant
import synthetic
from tests._util import assert_close_rms, dev_bf16, dev_weight, sub_weight

pytestmark = pytest.mark.gpu


def _check_stats(logits, rmax, rsum, rarg, T):
    zmax, am, se = oq.row_stats(logits, T)
    assert np.array_equal(rmax, zmax)
    assert np.array_equal(rarg, am)
    if T > 0:
        assert np.allclose(rsum, se, rtol=2e-6, atol=0)


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny_head(lib, M, T):
    r = synthetic.rng(300 + M)
    w = synthetic.quant_weight(r, 1000, 1024, 4, synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, 1024)
    dw = dev_weight(w)
    logits, rmax, rsum, rarg = lib.lm_head_verify(dw["wq"], dw["scales"], dw["biases"], 1024, 4, dev_bf16(x), T)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    want = oq.qmm_f32(w["wq"], w["scales"], w["biases"], 1024, 4, x)
    assert_close_rms(lg, want, what="logits")
    _check_stats(lg, rmax.cpu().numpy(), rsum.cpu().numpy(), rarg.cpu().numpy(), T)
    assert lib.device_error() == 0


@pytest.mark.parametrize("K,bits,M,T", [(4096, 8, 8, 0.7), (4096, 8, 16, 0.0), (2560, 4, 32, 1.0),
                                        (5120, 8, 32, 1.0)])
def test_full_vocab_head_sampled_rows(lib, K, bits, M, T):
    """V = 151936 at the full widths; the oracle checks a sample of vocabulary rows."""
    V = 151936
    r = synthetic.rng(400 + K + M)
    w = synthetic.quant_weight(r, V, K, bits, synthetic.LARGE_8BIT if bits == 8 else synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, K)
    dw = dev_weight(w)
    logits, rmax, rsum, rarg = lib.lm_head_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), T)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    am = rarg.cpu().numpy()
    rows = np.unique(np.concatenate([r.choice(V, 3000, replace=False), am, [0, V - 1, V - 64, 64 * 1187]]))
    want = oq.qmm_f32(*[sub_weight(w, rows)[k] for k in ("wq", "scales", "biases")], K, bits, x)
    assert_close_rms(lg[:, rows], want, what="sampled logits")
    _check_stats(lg, rmax.cpu().numpy(), rsum.cpu().numpy(), am, T)
    assert lib.device_error() == 0


@pytest.mark.parametrize("M,T", [(4, 0.7), (8, 0.0)])
def test_head_beyond_4096_tiles(lib, M, T):
    """A vocabulary of more than 4096 64-row tiles (V = 263144): the per-row merge
    of the tile statistics walks its tiles in several register-held chunks.  Row
    statistics against the GPU's own logits, logits on sampled rows."""
    V, K, bits = 4112 * 64 + 40, 512, 4
    r = synthetic.rng(450 + M)
    w = synthetic.quant_weight(r, V, K, bits, synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, K)
    dw = dev_weight(w)
    logits, rmax, rsum, rarg = lib.lm_head_verify(dw["wq"], dw["scales"], dw["biases"], K, bits, dev_bf16(x), T)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    am = rarg.cpu().numpy()
    rows = np.unique(np.concatenate([r.choice(V, 2000, replace=False), am, [0, V - 1, 4096 * 64, 4096 * 64 - 1]]))
    want = oq.qmm_f32(*[sub_weight(w, rows)[k] for k in ("wq", "scales", "biases")], K, bits, x)
    assert_close_rms(lg[:, rows], want, what="sampled logits")
    _check_stats(lg, rmax.cpu().numpy(), rsum.cpu().numpy(), am, T)
    assert lib.device_error() == 0
