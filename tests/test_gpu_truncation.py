"""Top-k / top-p truncation and logprobs: the CUDA path through the C ABI
against the oracle, with near-tie exemptions: a top_p cut whose prefix mass
lies within a rounding band of top_p times the total (1e-9 of it for
probability rows, whose weights both sides sum exactly in fp64; 2e-7 for
logits rows, whose weights the kernel takes from fp32 exp), a decision with
|u - p/q| < 1e-6 and a final draw with |u*Z - C_k| < 1e-6 * Z."""

import numpy as np
import pytest
import scipy.special
import torch

from oracle import accept as oa
import synthetic

pytestmark = pytest.mark.gpu

TIE = 1e-6


def _boundary_near_tie(keys, weights, top_k, top_p, band):
    """True when the top_p cut of this row sits within band * total of a prefix mass."""
    if top_p >= 1.0:
        return False
    w = np.asarray(weights, np.float64)
    V = len(w)
    order = np.lexsort((np.arange(V), -np.asarray(keys, np.float64)))
    n = V if top_k <= 0 else min(top_k, V)
    c = np.cumsum(w[order[:n]])
    return bool(np.min(np.abs(c - top_p * c[-1])) < band * c[-1])


def _target_near_tie(z, T, top_k, top_p):
    zz = np.asarray(z, np.float32)
    e = np.exp((zz.astype(np.float64) - float(zz.max())) / T)
    return _boundary_near_tie(zz, e, top_k, top_p, 2e-7)


CASES = [(0, 0.9), (50, 1.0), (40, 0.8), (1, 1.0), (0, 0.3), (5000, 0.95)]


@pytest.mark.parametrize("V", [1000, 151936])
@pytest.mark.parametrize("top_k,top_p", CASES)
def test_truncate_probs_matches_oracle(lib, V, top_k, top_p):
    r = synthetic.rng(700 + V % 97 + top_k)
    rows = 6
    q = scipy.special.softmax(r.standard_normal((rows, V)) * 2.0, axis=1).astype(np.float32)
    q[0, :] = np.float32(1.0 / V)                     # a row of ties: the lower indices win
    got = lib.truncate_probs(torch.from_numpy(q).cuda(), top_k, top_p).cpu().numpy()
    checked = 0
    for i in range(rows):
        if _boundary_near_tie(q[i], q[i].astype(np.float64), top_k, top_p, 1e-9):
            continue
        want = oa.truncate_probs(q[i], top_k, top_p)
        assert np.array_equal(got[i] > 0, want > 0), "row %d kept set" % i
        assert np.allclose(got[i], want, rtol=2e-6, atol=1e-12), "row %d values" % i
        checked += 1
    assert checked >= rows - 2
    # in place
    d = torch.from_numpy(q).cuda()
    lib.truncate_probs(d, top_k, top_p, out=d)
    assert np.array_equal(d.cpu().numpy(), got)


def _accept_case(lib, r, V, m, T, top_k, top_p):
    z = (r.standard_normal((m + 1, V)) * 2.0).astype(np.float32)
    q = scipy.special.softmax(z[:m].astype(np.float64) / T + r.standard_normal((m, V)), axis=1).astype(np.float32)
    draft = [int(r.choice(V, p=q[i].astype(np.float64) / q[i].astype(np.float64).sum())) for i in range(m)]
    u = r.random(m + 1).astype(np.float32)
    dq = torch.from_numpy(q).cuda() if m else None
    n, toks = lib.spec_accept_truncated([0, m + 1], torch.from_numpy(z).cuda(),
                                        torch.from_numpy(np.asarray(draft, np.int32)).cuda(), T, top_k, top_p,
                                        q=dq, u=torch.from_numpy(u).cuda())
    torch.cuda.synchronize()
    n = int(n[0].item())
    got = (n, toks.cpu().numpy()[:n].tolist())
    det = oa.sampled_accept_truncated_detail(z, q, draft, T, u, top_k, top_p)
    exempt = any(_target_near_tie(z[i], T, top_k, top_p) for i in range(m + 1))
    for i, rr in enumerate(det["ratios"]):
        exempt |= bool(np.isfinite(rr) and abs(float(u[i]) - rr) < TIE)
    exempt |= bool(np.min(np.abs(det["cdf"] - det["theta"])) < TIE * det["Z"])
    return got, det, exempt


@pytest.mark.parametrize("V", [1000, 151936])
@pytest.mark.parametrize("top_k,top_p", [(0, 0.9), (40, 0.8), (20, 1.0)])
def test_truncated_accept_matches_oracle(lib, V, top_k, top_p):
    r = synthetic.rng(710 + top_k)
    compared = 0
    trials = 24 if V == 1000 else 6
    for t in range(trials):
        m = [0, 1, 3, 7][t % 4]
        got, det, exempt = _accept_case(lib, r, V, m, 0.8, top_k, top_p)
        if exempt:
            continue
        assert got == (det["out_len"], det["tokens"]), (t, got, det["out_len"], det["tokens"])
        compared += 1
    assert compared >= trials - 2
    assert lib.device_error() == 0


def test_top_k_one_is_greedy(lib):
    r = synthetic.rng(720)
    for t in range(12):
        V, m = 1000, [1, 3, 7][t % 3]
        z = (r.standard_normal((m + 1, V)) * 2.0).astype(np.float32)
        am = np.argmax(z, axis=1)
        draft = np.asarray([int(am[i]) if r.random() < 0.6 else int(r.integers(0, V)) for i in range(m)], np.int32)
        q = scipy.special.softmax(r.standard_normal((m, V)), axis=1).astype(np.float32)
        u = r.random(m + 1).astype(np.float32)
        n, toks = lib.spec_accept_truncated([0, m + 1], torch.from_numpy(z).cuda(), torch.from_numpy(draft).cuda(),
                                            1.0, 1, 1.0, q=torch.from_numpy(q).cuda(), u=torch.from_numpy(u).cuda())
        torch.cuda.synchronize()
        n = int(n[0].item())
        assert (n, toks.cpu().numpy()[:n].tolist()) == oa.greedy_accept(z, draft)


@pytest.mark.parametrize("V,T", [(1000, 1.0), (151936, 0.7), (151936, 0.0)])
def test_logprobs_match_oracle(lib, V, T):
    r = synthetic.rng(730 + V % 13)
    rows, top_n = 5, 8
    z = (r.standard_normal((rows, V)) * 2.0).astype(np.float32)
    chosen = r.integers(0, V, rows).astype(np.int32)
    clp, ids, tlp = lib.logprobs(torch.from_numpy(z).cuda(), T, chosen=torch.from_numpy(chosen).cuda(), top_n=top_n)
    torch.cuda.synchronize()
    clp, ids, tlp = clp.cpu().numpy(), ids.cpu().numpy(), tlp.cpu().numpy()
    for i in range(rows):
        w_lp, w_ids, w_top = oa.logprobs(z[i], T, int(chosen[i]), top_n)
        assert abs(clp[i] - w_lp) <= 1e-5 * max(1.0, abs(w_lp))
        assert list(ids[i]) == list(w_ids)
        assert np.all(np.abs(tlp[i] - w_top) <= 1e-5 * np.maximum(1.0, np.abs(w_top)))


def test_rejections(lib):
    from speculative_decoding_verify_qmm_gb300.binding import SVError
    z = torch.zeros((2, 100), device="cuda")
    with pytest.raises(SVError):
        lib.truncate_probs(z, -1, 1.0)
    with pytest.raises(SVError):
        lib.truncate_probs(z, 0, 0.0)
    with pytest.raises(SVError):
        lib.logprobs(z, 1.0, top_n=33)


@pytest.mark.parametrize("V", [1, 2, 5, 9, 17])
def test_tiny_vocabularies_leave_slices_empty(lib, V):
    """A row is split over up to 8 CTAs: vocabularies this small leave some of
    them an empty slice (or a single token), which every call must get right."""
    r = synthetic.rng(760 + V)
    rows = 3
    q = scipy.special.softmax(r.standard_normal((rows, V)) * 2.0, axis=1).astype(np.float32)
    for top_k, top_p in [(0, 0.7), (2, 1.0), (3, 0.5), (0, 1.0)]:
        got = lib.truncate_probs(torch.from_numpy(q).cuda(), top_k, top_p).cpu().numpy()
        for i in range(rows):
            if _boundary_near_tie(q[i], q[i].astype(np.float64), top_k, top_p, 1e-9):
                continue
            want = oa.truncate_probs(q[i], top_k, top_p)
            assert np.array_equal(got[i] > 0, want > 0), (V, top_k, top_p, i)
            assert np.allclose(got[i], want, rtol=2e-6, atol=1e-12)
    z = (r.standard_normal((rows, V)) * 2.0).astype(np.float32)
    chosen = r.integers(0, V, rows).astype(np.int32)
    top_n = min(V, 8)
    clp, ids, tlp = lib.logprobs(torch.from_numpy(z).cuda(), 0.9, chosen=torch.from_numpy(chosen).cuda(), top_n=top_n)
    torch.cuda.synchronize()
    clp, ids, tlp = clp.cpu().numpy(), ids.cpu().numpy(), tlp.cpu().numpy()
    for i in range(rows):
        w_lp, w_ids, w_top = oa.logprobs(z[i], 0.9, int(chosen[i]), top_n)
        assert abs(clp[i] - w_lp) <= 1e-5 * max(1.0, abs(w_lp))
        assert list(ids[i]) == list(w_ids)
        assert np.all(np.abs(tlp[i] - w_top) <= 1e-5 * np.maximum(1.0, np.abs(w_top)))
    if V >= 2:  # the truncated accept on the same small rows (m = 1)
        got, det, exempt = _accept_case(lib, r, V, 1, 0.8, 2, 0.9)
        if not exempt:
            assert got == (det["out_len"], det["tokens"])
    assert lib.device_error() == 0
