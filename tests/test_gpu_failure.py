"""Failure detection without a GPU fault: a device-side bounded wait that
nothing completes ends at its limit, records a timeout in the device error
word (read and cleared by sv_device_error) and leaves the context usable."""

import ctypes

import pytest
import torch

from oracle import qmm as oq, quant
import synthetic
from speculative_decoding_verify_qmm_gb300 import binding
from tests._util import assert_close_bf16, dev_bf16, dev_weight, host_f32_of_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_a_timeout(lib):
    assert lib.device_error() == 0
    lib.check(lib.lib.sv_selftest_bounded_wait(20000, None))   # 20 ms
    bits = ctypes.c_uint(0)
    assert lib.lib.sv_device_error(ctypes.byref(bits)) == binding.SV_ETIMEOUT
    assert bits.value & 1                                       # the timeout bit of a wait on a full barrier
    assert lib.device_error() == 0                              # reading cleared it
    # the context still works: a projection against the oracle
    r = synthetic.rng(990)
    hw = synthetic.quant_weight(r, 200, 1024, 8, synthetic.LARGE_8BIT)
    hx = synthetic.activations(r, 3, 1024)
    w = dev_weight(hw)
    y = lib.qmm_verify(w["wq"], w["scales"], w["biases"], 1024, 8, dev_bf16(hx))
    torch.cuda.synchronize()
    want = quant.bf16_bits_to_f32(oq.qmm_verify(hw["wq"], hw["scales"], hw["biases"], 1024, 8, hx))
    assert_close_bf16(host_f32_of_bf16(y), want, what="after a timeout")
    assert lib.device_error() == 0


def test_selftest_rejects_a_limit_out_of_range(lib):
    assert lib.lib.sv_selftest_bounded_wait(0, None) == binding.SV_EINVAL
    assert lib.lib.sv_selftest_bounded_wait(2000000, None) == binding.SV_EINVAL
