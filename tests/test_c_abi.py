"""The library from a plain C program (tests/abi_from_c.c): compiled with gcc
against include/specverify.h and linked to libspecverify.so, with no Python in
the process.  Host mode runs on any machine; the GPU mode runs one projection,
the vocab head, Philox uniforms and the sampled accept step on device memory
the program allocates itself, and its outputs are checked against the oracle."""

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import accept as oa, philox as oph, qmm as oq, quant
import synthetic
from speculative_decoding_verify_qmm_gb300 import binding, build
from tests._util import assert_close_bf16

HERE = os.path.dirname(os.path.abspath(__file__))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    build.build()
    lib_dir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_from_c")
    cmd = [gcc, "-std=c99", "-O1", "-Wall", "-Werror", "-I", os.path.dirname(binding.HEADER),
           "-I", os.path.join(CUDA, "include"), os.path.join(HERE, "abi_from_c.c"), "-o", exe,
           "-L", lib_dir, "-lspecverify", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_caller_host_checks(c_program):
    r = subprocess.run([c_program, "host"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "host checks ok" in r.stdout


@pytest.mark.gpu
def test_c_caller_runs_one_verify_step(c_program, tmp_path):
    r = synthetic.rng(4242)
    N, K, bits, M = 200, 1024, 4, 3           # ragged last tile
    V, Kh, m, seed, T = 1000, 1024, 5, 77, 0.8
    w = synthetic.quant_weight(r, N, K, bits, synthetic.TINY_4BIT)
    x = synthetic.activations(r, M, K)
    hw = synthetic.quant_weight(r, V, Kh, bits, synthetic.TINY_4BIT)
    hx = synthetic.activations(r, m + 1, Kh)
    _, q = synthetic.logits_and_draft_probs(r, m, V)
    draft = synthetic.sample_drafts(r, q)
    hdr = np.array([N, K, bits, M, V, Kh, m, seed], np.int32).tobytes() + np.float32(T).tobytes()
    blob = hdr + b"".join(np.ascontiguousarray(a).tobytes() for a in (
        w["wq"], w["scales"], w["biases"], x, hw["wq"], hw["scales"], hw["biases"], hx,
        q.astype(np.float32), draft.astype(np.int32)))
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    fin.write_bytes(blob)
    res = subprocess.run([c_program, "gpu", str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    out = fout.read_bytes()
    rows = m + 1
    o = 0

    def take(dtype, count):
        nonlocal o
        a = np.frombuffer(out, dtype=dtype, count=count, offset=o)
        o += a.nbytes
        return a

    status = take(np.int32, 4)
    assert (status == 0).all(), status
    y = take(np.uint16, M * N).reshape(M, N)
    logits = take(np.float32, rows * V).reshape(rows, V)
    row_max, row_sumexp = take(np.float32, rows), take(np.float32, rows)
    row_argmax, u = take(np.int32, rows), take(np.float32, rows)
    out_len = int(take(np.int32, 1)[0])
    out_tokens = take(np.int32, rows)
    assert o == len(out)

    # the projection and the head against the oracle
    want_y = quant.bf16_bits_to_f32(oq.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x))
    assert_close_bf16(quant.bf16_bits_to_f32(y), want_y, what="qmm from C")
    want_z = oq.qmm_f32(hw["wq"], hw["scales"], hw["biases"], Kh, bits, hx)
    rms = np.sqrt(np.mean(want_z ** 2))
    assert np.max(np.abs(logits - want_z)) <= 1e-2 * rms
    # row statistics of the GPU's own logits: argmax exact, max exact, sum-exp to fp32 rounding
    assert (row_argmax == np.argmax(logits, axis=1)).all()
    assert (row_max == logits.max(axis=1)).all()
    se = np.exp((logits.astype(np.float64) - row_max[:, None].astype(np.float64)) / T).sum(axis=1)
    assert np.allclose(row_sumexp, se, rtol=2e-6)
    # Philox uniforms bit-exact, and the accept step on the GPU's logits
    assert (u == oph.uniforms(seed, 0, 0, rows)).all()
    det = oa.sampled_accept_detail(logits, q, draft, T, u)
    assert out_len == det["out_len"]
    assert out_tokens[:out_len].tolist() == list(det["tokens"])
