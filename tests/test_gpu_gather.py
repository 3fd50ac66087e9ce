"""Gather-qmm (mixture-of-experts rows) through the C ABI against the oracle."""

import numpy as np
import pytest
import torch

from oracle import qmm as oq, quant
import synthetic
from tests._util import assert_close_bf16, dev_bf16, host_bf16_bits, host_f32_of_bf16

pytestmark = pytest.mark.gpu

STATS = {2: synthetic.TINY_2BIT, 4: synthetic.TINY_4BIT, 8: synthetic.LARGE_8BIT}


def _experts(r, E, N, K, bits):
    ws = [synthetic.quant_weight(r, N, K, bits, STATS[bits]) for _ in range(E)]
    dev = {k: torch.from_numpy(np.ascontiguousarray(np.concatenate([w[k] for w in ws])).view(
        np.int32 if k == "wq" else np.float16)).cuda() for k in ("wq", "scales", "biases")}
    return ws, dev


def _routes(r, M, E, top):
    rows, exps = [], []
    for m in range(M):
        for e in r.choice(E, top, replace=False):
            rows.append(m)
            exps.append(int(e))
    return np.array(rows, np.int32), np.array(exps, np.int32)


def _check(lib, ws, dev, x, rows, exps, E, K, bits, what):
    y = lib.gather_qmm(dev["wq"], dev["scales"], dev["biases"], E, K, bits, dev_bf16(x),
                       torch.from_numpy(rows).cuda(), torch.from_numpy(exps).cuda())
    torch.cuda.synchronize()
    want = quant.bf16_bits_to_f32(oq.gather_qmm(ws, x, rows, exps))
    assert_close_bf16(host_f32_of_bf16(y), want, what=what)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K,E,M,top", [(200, 1024, 6, 5, 3), (768, 2048, 32, 8, 4), (64, 512, 3, 1, 2)])
def test_gather_matches_oracle(lib, bits, N, K, E, M, top):
    r = synthetic.rng(1700 + bits + N + E + M)
    ws, dev = _experts(r, E, N, K, bits)
    x = synthetic.activations(r, M, K)
    rows, exps = _routes(r, M, E, top)
    perm = r.permutation(len(rows))                    # pairs in no particular order
    _check(lib, ws, dev, x, rows[perm], exps[perm], E, K, bits, "gather %s" % ((N, K, E, M, top),))
    assert lib.device_error() == 0


def test_gather_one_expert_takes_every_row(lib):
    # M = 17 rows (the 24-row padded block) all routed to expert 2, plus a few others
    r = synthetic.rng(1750)
    E, N, K, M, bits = 4, 300, 1536, 17, 8
    ws, dev = _experts(r, E, N, K, bits)
    x = synthetic.activations(r, M, K)
    rows = np.concatenate([np.arange(M), [0, 5, 16]]).astype(np.int32)
    exps = np.concatenate([np.full(M, 2), [0, 3, 0]]).astype(np.int32)
    _check(lib, ws, dev, x, rows, exps, E, K, bits, "all rows to one expert")
    # the identity routing onto one expert is the plain verify matmul
    w = ws[2]
    y_plain = lib.qmm_verify(dev["wq"][2 * N:3 * N], dev["scales"][2 * N:3 * N], dev["biases"][2 * N:3 * N], K,
                             bits, dev_bf16(x))
    y_gather = lib.gather_qmm(dev["wq"], dev["scales"], dev["biases"], E, K, bits, dev_bf16(x),
                              torch.arange(M, dtype=torch.int32, device="cuda"),
                              torch.full((M,), 2, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert_close_bf16(host_f32_of_bf16(y_gather), host_f32_of_bf16(y_plain), what="gather vs qmm_verify")
    assert lib.device_error() == 0


def test_gather_flags_bad_pairs_and_leaves_their_rows(lib):
    r = synthetic.rng(1760)
    E, N, K, M, bits = 3, 64, 512, 2, 4
    ws, dev = _experts(r, E, N, K, bits)
    x = synthetic.activations(r, M, K)
    rows = np.array([0, 1, 1, 7], np.int32)             # row 7 does not exist
    exps = np.array([2, 0, 9, 1], np.int32)             # expert 9 does not exist
    y = torch.full((4, N), 3.0, dtype=torch.bfloat16, device="cuda")
    lib.gather_qmm(dev["wq"], dev["scales"], dev["biases"], E, K, bits, dev_bf16(x),
                   torch.from_numpy(rows).cuda(), torch.from_numpy(exps).cuda(), y=y)
    torch.cuda.synchronize()
    got = host_f32_of_bf16(y)
    assert np.all(got[2:] == 3.0)
    want = quant.bf16_bits_to_f32(oq.gather_qmm(ws, x, rows[:2], exps[:2]))
    assert_close_bf16(got[:2], want, what="valid pairs")
    assert lib.device_error() == 4                      # the bad-input bit, then cleared
    assert lib.device_error() == 0
