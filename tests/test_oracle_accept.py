"""Pins for the accept-step oracle: hand-built cases, closed forms, chi-square."""

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import accept, qmm
import synthetic


def _planted(m, V, winners, r):
    """Logits whose row i has its unique maximum at winners[i]."""
    z = r.standard_normal((m + 1, V)).astype(np.float32)
    for i, w in enumerate(winners):
        z[i, w] = z[i].max() + 1.0
    return z


def test_row_stats_uniform_and_ties():
    z = np.zeros((2, 50), dtype=np.float32)
    z[1, 7] = z[1, 30] = 3.0                       # duplicate maximum: lowest index wins
    zmax, am, se = qmm.row_stats(z, 1.0)
    assert am.tolist() == [0, 7]
    assert zmax.tolist() == [0.0, 3.0]
    assert se[0] == 50.0
    assert np.allclose(qmm.target_probs(z[0], 1.0), 1 / 50)


def test_row_stats_match_scipy():
    r = synthetic.rng(20)
    z = (r.standard_normal((4, 3000)) * 2).astype(np.float32)
    for T in (0.7, 1.0, 2.5):
        zmax, _, se = qmm.row_stats(z, T)
        lse = scipy.special.logsumexp(z.astype(np.float64) / T, axis=1)
        assert np.allclose(np.log(se) + zmax.astype(np.float64) / T, lse, rtol=0, atol=1e-12)
        p = qmm.target_probs(z[1], T)
        assert np.allclose(p, scipy.special.softmax(z[1].astype(np.float64) / T), rtol=1e-12, atol=0)


@pytest.mark.parametrize("m", [0, 1, 3, 7, 15])
def test_greedy_first_mismatch_at_every_position(m):
    r = synthetic.rng(21 + m)
    V = 64
    winners = [int(t) for t in r.integers(0, V, m + 1)]
    z = _planted(m, V, winners, r)
    # all drafts right: m accepted plus the bonus token
    n, toks = accept.greedy_accept(z, winners[:m])
    assert n == m + 1 and toks == winners
    for j in range(m):
        draft = list(winners[:m])
        draft[j] = (draft[j] + 1 + int(r.integers(0, V - 1))) % V   # wrong, never the winner
        if draft[j] == winners[j]:
            draft[j] = (draft[j] + 1) % V
        for i in range(j + 1, m):                   # later drafts are irrelevant
            draft[i] = int(r.integers(0, V))
        n, toks = accept.greedy_accept(z, draft)
        assert n == j + 1
        assert toks == winners[:j] + [winners[j]]


def test_sampled_q_equal_p_always_accepts():
    r = synthetic.rng(30)
    m, V, T = 5, 40, 1.0
    z = (r.standard_normal((m + 1, V)) * 2).astype(np.float32)
    q = np.stack([qmm.target_probs(z[i], T) for i in range(m)]).astype(np.float32)
    for _ in range(200):
        draft = [int(r.integers(0, V)) for _ in range(m)]
        u = (r.random(m + 1) * 0.999).astype(np.float32)
        n, toks = accept.sampled_accept(z, q, draft, T, u)
        assert n == m + 1 and toks[:m] == draft


def test_sampled_one_hot_draft_closed_form():
    # q one-hot on d: ratio p[d], so accept iff u < p[d]; the residual is p with d removed.
    r = synthetic.rng(31)
    V, T = 12, 1.0
    z = (r.standard_normal((2, V)) * 1.5).astype(np.float32)
    p = qmm.target_probs(z[0], T)
    d = 4
    q = np.zeros((1, V), dtype=np.float32)
    q[0, d] = 1.0
    det = accept.sampled_accept_detail(z, q, [d], T, np.array([p[d] + 1e-3, 0.3], np.float32))
    assert det["reject"] == 0 and det["weights_kind"] == "residual"
    assert abs(det["Z"] - (1 - p[d])) < 1e-12
    rest = p.copy()
    rest[d] = 0
    c = np.cumsum(rest / rest.sum())
    assert det["tokens"] == [int(np.nonzero(c > np.float32(0.3))[0][0])]
    det = accept.sampled_accept_detail(z, q, [d], T, np.array([p[d] - 1e-3, 0.3], np.float32))
    assert det["reject"] == -1 and det["tokens"][0] == d and det["weights_kind"] == "bonus"


def test_sampled_zero_residual_falls_back_to_p():
    # unnormalised q >= p everywhere: ratio 5/9 < 1, residual is zero -> draw from p
    z = np.zeros((2, 2), dtype=np.float32)
    q = np.array([[0.9, 0.9]], dtype=np.float32)
    det = accept.sampled_accept_detail(z, q, [1], 1.0, np.array([0.9, 0.75], np.float32))
    assert det["reject"] == 0 and det["weights_kind"] == "p_fallback"
    assert det["tokens"] == [1] and det["out_len"] == 1


def test_inverse_cdf_edges():
    k, theta, _ = accept.inverse_cdf([0.0, 0.25, 0.0, 0.75, 0.0], 0.0)
    assert k == 1 and theta == 0.0                 # strict '>' skips the zero-weight prefix
    k, _, _ = accept.inverse_cdf([0.0, 0.25, 0.0, 0.75, 0.0], 0.25)
    assert k == 3                                  # C_1 = 0.25 is not > 0.25
    k, _, _ = accept.inverse_cdf([0.5, 0.5, 0.0], 1.0)
    assert k == 1                                  # threshold at the total: last positive weight


def _chi2_pvalue(counts, probs):
    exp = probs * counts.sum()
    return scipy.stats.chisquare(counts, exp).pvalue


def test_sampled_accept_output_follows_target_chi_square():
    """Committed tokens are distributed as the target (the lossless claim)."""
    r = synthetic.rng(40)
    V, T, m, rounds = 16, 1.0, 2, 120_000
    z = (r.standard_normal((m + 1, V)) * 1.2).astype(np.float32)
    noisy = z[:m] + r.standard_normal((m, V)).astype(np.float32)
    q = np.stack([scipy.special.softmax(noisy[i].astype(np.float64)) for i in range(m)]).astype(np.float32)
    p0, p1 = qmm.target_probs(z[0], T), qmm.target_probs(z[1], T)
    first = np.zeros(V)
    second = np.zeros(V)
    qc = [np.cumsum(q[i].astype(np.float64) / q[i].astype(np.float64).sum()) for i in range(m)]
    for _ in range(rounds):
        draft = [min(int(np.searchsorted(qc[i], r.random(), side="right")), V - 1) for i in range(m)]
        u = r.random(m + 1).astype(np.float32)
        n, toks = accept.sampled_accept(z, q, draft, T, u)
        first[toks[0]] += 1
        if n >= 2:
            second[toks[1]] += 1
    assert _chi2_pvalue(first, p0) > 1e-3
    assert _chi2_pvalue(second, p1) > 1e-3
    # the pin must be able to fail: the draft's own distribution is rejected
    assert _chi2_pvalue(first, q[0].astype(np.float64) / q[0].sum()) < 1e-3


def test_batched_equals_per_request():
    r = synthetic.rng(50)
    V, T = 30, 0.8
    ms = [3, 0, 5, 1]
    offs = np.concatenate([[0], np.cumsum([mm + 1 for mm in ms])])
    z = (r.standard_normal((offs[-1], V)) * 2).astype(np.float32)
    q = np.concatenate([scipy.special.softmax(r.standard_normal((mm, V)), axis=1) for mm in ms]).astype(np.float32)
    drafts = [list(r.integers(0, V, mm)) for mm in ms]
    us = [r.random(mm + 1).astype(np.float32) for mm in ms]
    got = accept.spec_accept_batched(z, q, drafts, offs, T, us)
    qo = 0
    for b, mm in enumerate(ms):
        want = accept.sampled_accept(z[offs[b]:offs[b + 1]], q[qo:qo + mm], drafts[b], T, us[b])
        qo += mm
        assert got[b] == want


# ----------------------------------------------------- truncation and logprobs

def test_truncation_hand_examples():
    w = np.array([0.1, 0.5, 0.1, 0.3])
    keys = w.astype(np.float32)
    assert list(accept.truncation_mask(keys, w, 0, 0.8)) == [False, True, False, True]      # 0.5 + 0.3 reaches 0.8
    assert list(accept.truncation_mask(keys, w, 0, 0.81)) == [True, True, False, True]      # the tie goes to index 0
    assert list(accept.truncation_mask(keys, w, 1, 1.0)) == [False, True, False, False]
    assert list(accept.truncation_mask(keys, w, 3, 1.0)) == [True, True, False, True]
    # top_k first, then top_p over the renormalised survivors: (0.5, 0.3) -> shares (0.625, 0.375)
    assert list(accept.truncation_mask(keys, w, 2, 0.6)) == [False, True, False, False]
    assert list(accept.truncation_mask(keys, w, 2, 0.7)) == [False, True, False, True]
    flat = np.full(6, 1 / 6)
    assert list(accept.truncation_mask(flat.astype(np.float32), flat, 2, 1.0)) == [True, True, False, False, False, False]


def test_no_truncation_is_the_plain_target():
    r = synthetic.rng(60)
    z = (r.standard_normal(50) * 2).astype(np.float32)
    assert np.allclose(accept.truncated_target_probs(z, 0.8, 0, 1.0), qmm.target_probs(z, 0.8), rtol=1e-12)
    assert np.allclose(accept.truncated_target_probs(z, 0.8, 50, 1.0), qmm.target_probs(z, 0.8), rtol=1e-12)


def test_top_k_one_sampled_accept_is_greedy():
    # the truncated target is one-hot on the argmax: sampled acceptance reduces to greedy
    r = synthetic.rng(61)
    for _ in range(200):
        V, m = 20, int(r.integers(0, 6))
        z = (r.standard_normal((m + 1, V)) * 2).astype(np.float32)
        am = np.argmax(z, axis=1)
        draft = [int(am[i]) if r.random() < 0.6 else int(r.integers(0, V)) for i in range(m)]
        q = scipy.special.softmax(r.standard_normal((m, V)), axis=1).astype(np.float32)
        u = r.random(m + 1).astype(np.float32)
        d = accept.sampled_accept_truncated_detail(z, q, draft, 1.0, u, 1, 1.0)
        assert (d["out_len"], d["tokens"]) == accept.greedy_accept(z, draft)


def test_truncated_sampled_accept_follows_truncated_target_chi_square():
    r = synthetic.rng(62)
    V, T, m, rounds, top_k, top_p = 16, 1.0, 2, 60_000, 10, 0.8
    z = (r.standard_normal((m + 1, V)) * 1.2).astype(np.float32)
    q = scipy.special.softmax(z[:m].astype(np.float64) + r.standard_normal((m, V)), axis=1).astype(np.float32)
    p0 = accept.truncated_target_probs(z[0], T, top_k, top_p)
    p1 = accept.truncated_target_probs(z[1], T, top_k, top_p)
    assert (p0 == 0).sum() >= 6                       # the truncation does remove tokens
    qc = [np.cumsum(q[i].astype(np.float64) / q[i].astype(np.float64).sum()) for i in range(m)]
    first, second = np.zeros(V), np.zeros(V)
    for _ in range(rounds):
        draft = [min(int(np.searchsorted(qc[i], r.random(), side="right")), V - 1) for i in range(m)]
        u = r.random(m + 1).astype(np.float32)
        d = accept.sampled_accept_truncated_detail(z, q, draft, T, u, top_k, top_p)
        first[d["tokens"][0]] += 1
        if d["out_len"] >= 2:
            second[d["tokens"][1]] += 1
    assert first[p0 == 0].sum() == 0 and second[p1 == 0].sum() == 0   # never outside the kept set
    keep0, keep1 = p0 > 0, p1 > 0
    assert _chi2_pvalue(first[keep0], p0[keep0]) > 1e-3
    assert _chi2_pvalue(second[keep1], p1[keep1]) > 1e-3
    # the pin can fail: the untruncated target is rejected
    full = qmm.target_probs(z[0], T)
    assert _chi2_pvalue(first, full) < 1e-3


def test_truncate_probs_rule():
    q = np.array([0.05, 0.4, 0.05, 0.3, 0.2], np.float32)
    out = accept.truncate_probs(q, 0, 0.85)                # 0.4 + 0.3 + 0.2 = 0.9 >= 0.85
    assert np.allclose(out, [0, 0.4 / 0.9, 0, 0.3 / 0.9, 0.2 / 0.9])
    out = accept.truncate_probs(q, 2, 1.0)
    assert np.allclose(out, [0, 0.4 / 0.7, 0, 0.3 / 0.7, 0])


def test_logprobs_closed_forms():
    V = 10
    lp, ids, top = accept.logprobs(np.zeros(V, np.float32), 1.0, 3, 4)
    assert lp == pytest.approx(-np.log(V)) and list(ids) == [0, 1, 2, 3]
    assert np.allclose(top, -np.log(V))
    r = synthetic.rng(63)
    z = (r.standard_normal(300) * 3).astype(np.float32)
    for T in (0.0, 0.7, 1.0):
        want = scipy.special.log_softmax(z.astype(np.float64) / (T if T > 0 else 1.0))
        lp, ids, top = accept.logprobs(z, T, 17, 5)
        assert lp == pytest.approx(want[17], rel=1e-12)
        assert list(ids) == list(np.argsort(-want, kind="stable")[:5])
        assert np.allclose(top, want[ids], rtol=1e-12)
