"""Accept-step parity: bit-exact against the oracle on identical fp32 logits, with
the near-tie exemptions of the parity rules (|u - p/q| < 1e-6 for a decision,
|u*Z - C_k| < 1e-6 * Z for the final draw)."""

import numpy as np
import pytest
import torch

from oracle import accept as oa
from oracle import philox as oph
import synthetic

pytestmark = pytest.mark.gpu

TIE = 1e-6


def _exempt(det, u):
    """True when the oracle's outcome sits within the stated tolerance of a tie."""
    for i, r in enumerate(det["ratios"]):
        if np.isfinite(r) and abs(float(u[i]) - r) < TIE:
            return True
    c = det["cdf"]
    return bool(np.min(np.abs(c - det["theta"])) < TIE * det["Z"])


def _gpu(lib, z, q, draft, T, u, stats=None):
    dz = torch.from_numpy(z).cuda()
    dq = torch.from_numpy(q).cuda() if q is not None and q.size else None
    dd = torch.from_numpy(np.asarray(draft, np.int32)).cuda()
    du = torch.from_numpy(np.asarray(u, np.float32)).cuda() if u is not None else None
    n, toks = lib.spec_accept(dz, dd, T, q=dq, u=du, stats=stats)
    torch.cuda.synchronize()
    n = int(n.item())
    return n, toks.cpu().numpy()[:n].tolist()


@pytest.mark.parametrize("m", [0, 1, 7])
def test_greedy_tiny_bit_exact(lib, m):
    r = synthetic.rng(500 + m)
    for trial in range(60):
        z, _ = synthetic.logits_and_draft_probs(r, m, 1000)
        target = np.argmax(z, axis=1)
        draft = synthetic.agreeing_drafts(r, target[:m], 1000, 0.7)
        assert _gpu(lib, z, None, draft, 0.0, None) == tuple(oa.greedy_accept(z, draft))


def _sampled_trials(lib, seed, m, V, T, trials):
    r = synthetic.rng(seed)
    exempt = 0
    for _ in range(trials):
        z, q = synthetic.logits_and_draft_probs(r, m, V)
        draft = synthetic.sample_drafts(r, q) if m else np.zeros(0, np.int32)
        u = synthetic.accept_uniforms(r, m + 1)
        det = oa.sampled_accept_detail(z, q, draft, T, u)
        got = _gpu(lib, z, q, draft, T, u)
        if got != (det["out_len"], det["tokens"]):
            assert _exempt(det, u), (got, det["out_len"], det["tokens"])
            exempt += 1
    assert exempt <= max(1, trials // 50)
    assert lib.device_error() == 0


@pytest.mark.parametrize("m", [0, 1, 7])
def test_sampled_tiny(lib, m):
    _sampled_trials(lib, 600 + m, m, 1000, 1.0, 150)


@pytest.mark.parametrize("m", [0, 3, 7, 15])
def test_sampled_full_vocab(lib, m):
    _sampled_trials(lib, 700 + m, m, 151936, 0.7, 12)


def test_sampled_rejects_often_and_resamples(lib):
    """A draft far from the target: most rounds end in a residual draw."""
    r = synthetic.rng(800)
    m, V, T = 7, 4096, 1.0
    seen_reject = 0
    for _ in range(40):
        z = (r.standard_normal((m + 1, V)) * 2).astype(np.float32)
        q = np.full((m, V), 1.0 / V, np.float32)          # uniform draft
        draft = r.integers(0, V, m).astype(np.int32)
        u = synthetic.accept_uniforms(r, m + 1)
        det = oa.sampled_accept_detail(z, q, draft, T, u)
        seen_reject += det["reject"] >= 0
        got = _gpu(lib, z, q, draft, T, u)
        assert got == (det["out_len"], det["tokens"]) or _exempt(det, u)
    assert seen_reject > 20


def test_zero_draft_probability_accepts(lib):
    r = synthetic.rng(801)
    m, V, T = 4, 512, 1.0
    z, q = synthetic.logits_and_draft_probs(r, m, V)
    draft = synthetic.sample_drafts(r, q)
    for i, d in enumerate(draft):
        q[i, d] = 0.0
    u = np.full(m + 1, 0.999, np.float32)
    n, toks = _gpu(lib, z, q, draft, T, u)
    assert n == m + 1 and toks[:m] == draft.tolist()


def test_batched_matches_oracle(lib):
    r = synthetic.rng(900)
    V, T = 151936, 1.0
    ms = [7, 7, 7, 7]
    for trial in range(4):
        offs = np.concatenate([[0], np.cumsum([mm + 1 for mm in ms])]).astype(np.int32)
        zs, qs, drafts, us = [], [], [], []
        for b, mm in enumerate(ms):
            z, q = synthetic.logits_and_draft_probs(r, mm, V)
            zs.append(z); qs.append(q)
            drafts.append(synthetic.sample_drafts(r, q))
            us.append(oph.uniforms(1234, b, trial * 8, mm + 1))   # per-request Philox stream
        Z = np.concatenate(zs); Q = np.concatenate(qs)
        want = oa.spec_accept_batched(Z, Q, drafts, offs, T, us)
        n, toks = lib.spec_accept_batched(offs.tolist(), torch.from_numpy(Z).cuda(),
                                          torch.from_numpy(np.concatenate(drafts)).cuda(), T,
                                          q=torch.from_numpy(Q).cuda(),
                                          u=torch.from_numpy(np.concatenate(us)).cuda())
        torch.cuda.synchronize()
        n = n.cpu().numpy(); toks = toks.cpu().numpy()
        for b in range(len(ms)):
            got = (int(n[b]), toks[offs[b]:offs[b] + n[b]].tolist())
            if got != tuple(want[b]) and list(got) != list(want[b]):
                det = oa.sampled_accept_detail(zs[b], qs[b], drafts[b], T, us[b])
                assert _exempt(det, us[b])
    assert lib.device_error() == 0


def test_out_of_range_draft_is_flagged(lib):
    """The kernel's own bounds check turns a bad token id into an error bit, not a fault."""
    r = synthetic.rng(901)
    z, q = synthetic.logits_and_draft_probs(r, 2, 100)
    draft = np.array([5, 100], np.int32)
    u = np.zeros(3, np.float32)
    _gpu(lib, z, q, draft, 1.0, u)
    assert lib.device_error() != 0
    assert lib.device_error() == 0          # reading clears it


def test_greedy_m31_full_vocab_every_mismatch_position(lib):
    """The warp-wide first-mismatch reduction at its widest (m = 31 drafts)."""
    r = synthetic.rng(820)
    m, V = 31, 151936
    z = (r.standard_normal((m + 1, V)) * 2).astype(np.float32)
    target = np.argmax(z, axis=1)
    for pos in [0, 1, 15, 29, 30, None]:
        draft = target[:m].astype(np.int32).copy()
        if pos is not None:
            draft[pos] = (draft[pos] + 1) % V
            draft[pos + 1:] = r.integers(0, V, m - pos - 1)   # anything after the first mismatch
        assert _gpu(lib, z, None, draft, 0.0, None) == tuple(oa.greedy_accept(z, draft))
    assert lib.device_error() == 0


def test_draft_equal_to_target_always_accepts(lib):
    """q = p (the target's own distribution, in fp32): p/q = 1 up to rounding, so
    every draft is accepted except where |u - p/q| < 1e-6."""
    r = synthetic.rng(821)
    m, V, T = 15, 151936, 1.0
    z = (r.standard_normal((m + 1, V)) * 2).astype(np.float32)
    q = np.stack([oq_target(z[i], T) for i in range(m)]).astype(np.float32)
    for _ in range(3):
        draft = np.asarray([int(r.choice(V, p=q[i].astype(np.float64) / q[i].astype(np.float64).sum()))
                            for i in range(m)], np.int32)
        u = synthetic.accept_uniforms(r, m + 1)
        det = oa.sampled_accept_detail(z, q, draft, T, u)
        got = _gpu(lib, z, q, draft, T, u)
        if got != (det["out_len"], det["tokens"]):
            assert _exempt(det, u)
        else:
            assert got[0] == m + 1                         # all accepted, then the bonus draw
    assert lib.device_error() == 0


def oq_target(z_row, T):
    from oracle import qmm as oq
    return oq.target_probs(z_row, T)


def test_small_residual_draw_is_valid(lib):
    """q = p (1 +- 1e-4), renormalised: a rejection leaves a residual max(0, p - q)
    whose total Z is ~1e-4.  Decisions are bit-exact (ratios are far from u);
    the drawn token carries positive residual weight and sits where u * Z falls
    in the oracle's cumulative weights, to within the kernel's fp32 rounding of
    p (about 1e-7 of p per token, a few 1e-4 of a Z this small)."""
    r = synthetic.rng(822)
    V, T = 32768, 1.0
    for trial in range(6):
        z = (r.standard_normal((2, V)) * 2).astype(np.float32)
        p0 = oq_target(z[0], T)
        q0 = p0 * (1.0 + 1e-4 * np.sign(r.standard_normal(V)))
        q0 = np.ascontiguousarray((q0 / q0.sum()).astype(np.float32).reshape(1, V))
        d = int(np.argmax(np.where(q0[0] > p0, p0, 0.0)))   # a likely token with q > p: p/q < 1
        draft = np.asarray([d], np.int32)
        u = np.asarray([0.99995, r.random()], np.float32)   # rejected: u > p/q ~ 1 - 1e-4
        det = oa.sampled_accept_detail(z, q0, draft, T, u)
        assert det["reject"] == 0 and det["weights_kind"] == "residual" and det["Z"] < 1e-3
        n, toks = _gpu(lib, z, q0, draft, T, u)
        assert n == 1
        k = toks[0]
        res = np.maximum(0.0, p0 - q0[0].astype(np.float64))
        assert res[k] > 0
        c = np.cumsum(res) / res.sum()
        lo, hi = (c[k - 1] if k else 0.0), c[k]
        assert lo - 2e-3 <= float(u[1]) <= hi + 2e-3, (trial, lo, float(u[1]), hi)
    assert lib.device_error() == 0
