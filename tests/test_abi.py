"""The C-ABI library builds, loads and exports every symbol of include/specverify.h,
and rejects bad arguments on the host before touching a device (no GPU needed)."""

import ctypes

import pytest

from speculative_decoding_verify_qmm_gb300 import binding, build


@pytest.fixture(scope="module")
def raw():
    build.build()
    return binding.load_library()


def test_every_declared_symbol_is_exported(raw):
    names = binding.header_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(raw, name), name
    assert set(names) == set(binding._SIGNATURES)


def test_status_strings(raw):
    assert raw.sv_status_string(0) == b"ok"
    assert raw.sv_status_string(1) == b"invalid argument"
    assert raw.sv_version() >= 100


P = ctypes.c_void_p


def _qmm(raw, N=64, K=512, bits=8, group=64, M=4, wq=16, x=16, y=16, ws=256, ws_bytes=1 << 20, ldx=None):
    return raw.sv_qmm_verify(P(wq), P(16), P(16), N, K, bits, group, P(x), ldx or K, M, P(y), N, None, 0,
                             P(ws), ws_bytes, None)


def test_qmm_argument_errors_on_host(raw):
    assert _qmm(raw, bits=3) == binding.SV_EUNSUPPORTED
    assert _qmm(raw, bits=16) == binding.SV_EUNSUPPORTED
    assert _qmm(raw, group=32) == binding.SV_EUNSUPPORTED
    assert _qmm(raw, K=576) == binding.SV_EUNSUPPORTED       # multiple of 64, not of 512
    assert _qmm(raw, K=100) == binding.SV_EINVAL
    assert _qmm(raw, M=513) == binding.SV_EUNSUPPORTED
    assert _qmm(raw, M=0) == binding.SV_EINVAL
    assert _qmm(raw, N=0) == binding.SV_EINVAL
    assert _qmm(raw, wq=0) == binding.SV_EINVAL
    assert _qmm(raw, wq=8) == binding.SV_EINVAL              # not 16-byte aligned
    assert _qmm(raw, x=0) == binding.SV_EINVAL
    assert _qmm(raw, ldx=100) == binding.SV_EINVAL
    assert _qmm(raw, ws=128) == binding.SV_EINVAL            # workspace not 256-byte aligned
    assert b"512" in raw.sv_last_error() or raw.sv_last_error()


def test_accept_argument_errors_on_host(raw):
    offs = (ctypes.c_int32 * 3)(0, 4, 9)
    args = dict(ldl=1000, V=1000, T=1.0)
    # m out of range, offsets not starting at zero, bad temperature, missing q/u
    assert raw.sv_spec_accept(P(16), 1000, None, None, None, P(16), 1000, P(16), 32, 1000, 1.0, P(16), P(16),
                              P(16), P(256), 1 << 20, None) == binding.SV_EINVAL
    bad = (ctypes.c_int32 * 3)(1, 4, 9)
    assert raw.sv_spec_accept_batched(2, bad, P(16), 1000, None, None, None, P(16), 1000, P(16), 1000, 1.0,
                                      P(16), P(16), P(16), P(256), 1 << 20, None) == binding.SV_EINVAL
    assert raw.sv_spec_accept_batched(2, offs, P(16), 1000, None, None, None, P(16), 1000, P(16), 1000,
                                      float("nan"), P(16), P(16), P(16), P(256), 1 << 20, None) == binding.SV_EINVAL
    assert raw.sv_spec_accept_batched(2, offs, P(16), 1000, None, None, None, None, 1000, P(16), 1000, 1.0,
                                      P(16), P(16), P(16), P(256), 1 << 20, None) == binding.SV_EINVAL
    # row statistics must be all given or all NULL for sampled accept
    assert raw.sv_spec_accept_batched(2, offs, P(16), 1000, P(16), None, None, P(16), 1000, P(16), 1000, 1.0,
                                      P(16), P(16), P(16), P(256), 1 << 20, None) == binding.SV_EINVAL
    # workspace too small
    assert raw.sv_spec_accept_batched(2, offs, P(16), 1000, None, None, None, P(16), 1000, P(16), 1000, 1.0,
                                      P(16), P(16), P(16), P(256), 16, None) == binding.SV_EINVAL
    assert raw.sv_accept_workspace_bytes(0, 4) == 0
    assert raw.sv_accept_workspace_bytes(2, 9) > 0
    del args


def test_glue_and_philox_argument_errors_on_host(raw):
    assert raw.sv_philox_uniforms(1, 0, 0, -1, P(16), None) == binding.SV_EINVAL
    assert raw.sv_philox_uniforms(1, 0, 0, 0, None, None) == binding.SV_OK      # nothing to do
    assert raw.sv_rmsnorm(P(16), 64, 0, 64, None, 1e-6, P(16), 64, None) == binding.SV_EINVAL
    assert raw.sv_rmsnorm(P(16), 32, 2, 64, None, 1e-6, P(16), 64, None) == binding.SV_EINVAL
    assert raw.sv_residual_add(None, 64, P(16), 64, 2, 64, None) == binding.SV_EINVAL
    assert raw.sv_swiglu(P(16), 64, P(16), 64, 2, 64, P(16), 10, None) == binding.SV_EINVAL


def test_bf16_ulp_helper():
    import numpy as np
    from oracle import quant
    from tests._util import bf16_ulp
    x = np.array([1.0, 1.5, 2.0, 3.0, 0.75, -6.0, 1e-3], dtype=np.float32)
    # the next bf16 value above |x| is |x| + ulp for every x exactly representable in bf16
    bits = quant.f32_to_bf16_bits(np.abs(x))
    nxt = quant.bf16_bits_to_f32((bits + 1).astype(np.uint16)).astype(np.float64)
    assert np.allclose(nxt - quant.bf16_bits_to_f32(bits), bf16_ulp(x), rtol=0, atol=0)


def test_round_plan_argument_errors_on_host(raw):
    """The plan calls reject bad models and buffers before touching the device."""
    assert raw.sv_round_plan_bytes(None) == 0
    assert raw.sv_round_plan_init(None, P(256), 1 << 20) == binding.SV_EINVAL
    layers = (binding.Layer * 1)()
    model = binding.Model(0, 1024, 1024, 2048, 1000, 8, 1e-6, layers, binding.QWeight())
    assert raw.sv_round_plan_bytes(ctypes.byref(model)) == 0              # no layers
    assert raw.sv_round_plan_init(ctypes.byref(model), P(256), 1 << 20) == binding.SV_EINVAL
    model.n_layers = 68                                                     # more than 4 * 67 + 1 phases
    assert raw.sv_round_plan_bytes(ctypes.byref(model)) == 0
    model.n_layers = 1
    assert raw.sv_round_plan_bytes(ctypes.byref(model)) == 5 * 3 * 128     # 5 projections x 3 descriptors
    assert raw.sv_round_plan_init(ctypes.byref(model), P(256), 1 << 20) == binding.SV_EINVAL  # null weights


def test_pack_sizes_and_argument_errors_on_host(raw):
    assert raw.sv_qmm_pack_bytes(1000, 1024, 8) == 16 * 2 * (64 * 512 + 2 * 64 * 8 * 2)
    assert raw.sv_qmm_pack_bytes(1024, 1024, 4) == 16 * 2 * (64 * 256 + 2 * 64 * 8 * 2)
    assert raw.sv_qmm_pack_bytes(1024, 576, 8) == 0      # K not a multiple of 512
    assert raw.sv_qmm_pack_bytes(1024, 1024, 3) == 0
    assert raw.sv_qmm_pack_bytes(0, 1024, 8) == 0
    ok = dict(wq=P(256), s=P(256), b=P(256))
    assert raw.sv_qmm_pack(None, ok["s"], ok["b"], 64, 512, 8, 64, P(256), 1 << 20, None) == binding.SV_EINVAL
    assert raw.sv_qmm_pack(ok["wq"], ok["s"], ok["b"], 64, 512, 8, 64, None, 1 << 20, None) == binding.SV_EINVAL
    assert raw.sv_qmm_pack(ok["wq"], ok["s"], ok["b"], 64, 512, 8, 64, P(264), 1 << 20, None) == binding.SV_EINVAL
    assert raw.sv_qmm_pack(ok["wq"], ok["s"], ok["b"], 64, 512, 8, 64, P(256), 16, None) == binding.SV_EINVAL
    assert raw.sv_qmm_pack(ok["wq"], ok["s"], ok["b"], 64, 512, 3, 64, P(256), 1 << 20, None) == binding.SV_EUNSUPPORTED
