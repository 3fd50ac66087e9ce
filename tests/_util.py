"""Helpers shared by the GPU parity tests (host <-> device copies, tolerance)."""

import numpy as np
import torch

from oracle import quant

REL_TOL = 1e-2   # max |gpu - oracle| <= REL_TOL * rms(oracle), fp32 accumulation on both sides


def dev_weight(w, device="cuda"):
    """Host weight dict (numpy) -> device tensors (int32 words, fp16 scales/biases)."""
    return {"wq": torch.from_numpy(w["wq"].view(np.int32)).to(device),
            "scales": torch.from_numpy(w["scales"].view(np.float16)).to(device),
            "biases": torch.from_numpy(w["biases"].view(np.float16)).to(device),
            "K": w["K"], "bits": w["bits"]}


def dev_bf16(bits_u16, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).to(device).view(torch.bfloat16)


def host_bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32_of_bf16(t):
    return quant.bf16_bits_to_f32(host_bf16_bits(t))


def assert_close_rms(got, want, tol=REL_TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    rms = np.sqrt(np.mean(want ** 2))
    err = np.abs(got - want).max() if got.size else 0.0
    assert err <= tol * rms, "%s max err %.3e > %.1e * rms %.3e" % (what, err, tol, rms)
    return err / rms if rms else 0.0


def bf16_ulp(x):
    """Unit in the last place of bf16 at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 0.0)


def assert_close_bf16(got, want, tol=REL_TOL, what="", ulps=1):
    """Parity of bf16 outputs.  Each side rounds its fp32-accumulated value to
    bf16 once; the REL_TOL * rms rule bounds the accumulation error, and one
    bf16 ulp at the element's magnitude covers a rounding that falls on the
    other side of a bf16 boundary (`ulps` such roundings for a value that
    passes through several bf16 results in turn)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    rms = np.sqrt(np.mean(want ** 2))
    excess = np.abs(got - want) - ulps * bf16_ulp(want)
    err = excess.max() if got.size else 0.0
    assert err <= tol * rms, "%s max err beyond one bf16 ulp %.3e > %.1e * rms %.3e" % (what, err, tol, rms)
    return err / rms if rms else 0.0


def sub_weight(w, rows):
    """The weight rows `rows` of a host weight dict (for sampled oracle checks)."""
    return {"wq": w["wq"][rows], "scales": w["scales"][rows], "biases": w["biases"][rows],
            "K": w["K"], "bits": w["bits"]}
