"""The allocation-free matmul entry point (sv_qmm_verify_noalloc).

Callers that cannot allocate device memory - a plugin inside an application
that owns all device memory, a runtime that bans cudaMalloc after start-up -
use this form; its scratch is an array built into the library.  This file is
collected last on purpose: a failure here still lets every other test run
first.  It checks, through the C ABI, that calls in a row (different shapes,
so each sees the previous one's leftovers in the shared array) match
sv_qmm_verify and the CPU oracle within the parity tolerance, and that a call needing more
scratch than the array holds is refused with a clear error.
"""

import pytest
import torch

from oracle import qmm as oq, quant
import synthetic
from speculative_decoding_verify_qmm_gb300.binding import SVError, SV_EUNSUPPORTED
from tests._util import REL_TOL, assert_close_bf16, dev_bf16, dev_weight, host_f32_of_bf16

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_form_on_two_calls(lib):
    # A long-K call first, then shorter ones: the later calls' split-tile
    # partials then sit where the first call left nonzero prepared
    # activations, so a call that did not clear its own region would fail.
    r = synthetic.rng(4242)
    cases = [(1024, 12288, 8, 16, synthetic.LARGE_8BIT), (4096, 1024, 8, 8, synthetic.LARGE_8BIT),
             (1000, 2048, 4, 17, synthetic.TINY_4BIT)]
    for N, K, bits, M, stats in cases:
        hw = synthetic.quant_weight(r, N, K, bits, stats)
        hx = synthetic.activations(r, M, K)
        w, x = dev_weight(hw), dev_bf16(hx)
        got = lib.qmm_verify_noalloc(w["wq"], w["scales"], w["biases"], K, bits, x)
        want = lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x)
        torch.cuda.synchronize()
        what = "noalloc %dx%d M=%d" % (N, K, M)
        assert_close_bf16(host_f32_of_bf16(got), host_f32_of_bf16(want), tol=REL_TOL, what=what)
        oracle = quant.bf16_bits_to_f32(oq.qmm_verify(hw["wq"], hw["scales"], hw["biases"], K, bits, hx))
        assert_close_bf16(host_f32_of_bf16(got), oracle, tol=REL_TOL, what=what + " vs oracle")
    assert lib.lib.sv_qmm_noalloc_scratch_bytes() == 4 << 20
    assert lib.device_error() == 0


def test_noalloc_refuses_calls_beyond_its_scratch(lib):
    r = synthetic.rng(4243)
    N, K, M = 64, 65536, 32
    w = dev_weight(synthetic.quant_weight(r, N, K, 8, synthetic.LARGE_8BIT))
    x = dev_bf16(synthetic.activations(r, M, K))
    with pytest.raises(SVError) as e:
        lib.qmm_verify_noalloc(w["wq"], w["scales"], w["biases"], K, 8, x)
    assert e.value.status == SV_EUNSUPPORTED
    assert "scratch" in str(e.value)
