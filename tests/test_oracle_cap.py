"""Pins for the draft-cap oracle: closed forms, simulation and limiting cases."""

import numpy as np
import pytest

from oracle import cap
import synthetic


@pytest.mark.parametrize("p", [0.0, 0.3, 0.7, 0.95, 1.0])
@pytest.mark.parametrize("c", [0, 1, 4, 15])
def test_expected_committed_geometric_closed_form(p, c):
    want = c + 1 if p == 1.0 else (1 - p ** (c + 1)) / (1 - p)
    assert cap.expected_committed(p, c) == pytest.approx(want, rel=1e-12, abs=1e-15)


def test_expected_committed_matches_simulated_rounds():
    # each draft position accepted w.p. p given all earlier ones were; the round
    # commits the accepted prefix plus one target token
    r = synthetic.rng(300)
    p, c, n = 0.7, 6, 200_000
    acc = r.random((n, c)) < p
    prefix = np.where(acc.all(axis=1), c, np.argmin(acc, axis=1))
    committed = prefix + 1
    se = committed.std() / np.sqrt(n)
    assert abs(committed.mean() - cap.expected_committed(p, c)) < 5 * se


def test_best_cap_limiting_cases():
    z = [0.0] * 8
    flat = [10.0] * 8
    # free verify width and a free drafter: the widest cap wins for any p > 0
    assert cap.best_cap(0.5, flat, z, 1.0, 7)[0] == 7
    # nothing is ever accepted: every cap commits one token, ties go to cap 0
    assert cap.best_cap(0.0, flat, z, 1.0, 7)[0] == 0
    # a cliff after width 5 (cap 4): caps beyond it cost 10x
    cliff = [10.0] * 5 + [100.0] * 3
    assert cap.best_cap(0.8, cliff, z, 0.0, 7)[0] == 4
    # a drafter that costs more than a whole plain step per draft never pays
    assert cap.best_cap(0.9, flat, [0.0] + [50.0 * k for k in range(1, 8)], 0.0, 7)[0] == 0


def test_best_cap_maximises_simulated_throughput():
    r = synthetic.rng(301)
    verify = [20.0 + 0.4 * c + (3.0 * (c - 5) if c > 5 else 0.0) for c in range(16)]
    draft = [0.0] + [1.5 + 0.8 * c for c in range(1, 16)]
    p = 0.75
    best, _ = cap.best_cap(p, verify, draft, 2.0, 15)
    n = 100_000
    rates = []
    for c in range(16):
        if c:
            acc = r.random((n, c)) < p
            prefix = np.where(acc.all(axis=1), c, np.argmin(acc, axis=1))
        else:
            prefix = np.zeros(n)
        rates.append((prefix + 1).sum() / (n * (draft[c] + 2.0 + verify[c])))
    rates = np.array(rates)
    assert rates[best] >= rates.max() * (1 - 3e-3)
    assert np.argmax(rates) in (best - 1, best, best + 1)


def test_acceptance_estimate_single_round_and_convergence():
    z = [0.0] * 8
    ctl = cap.CapController(7, [1.0] * 8, z, 0.0, alpha=1.0, probe_every=4, probe_cap=2, p0=0.5)
    ctl.update(4, 2)                       # 2 successes, 1 failure
    assert ctl.p() == pytest.approx(2 / 3)
    ctl.update(4, 4)                       # 4 successes, no failure
    assert ctl.p() == 1.0
    ctl.update(0, 0)                       # a plain step carries no information
    assert ctl.p() == 1.0
    r = synthetic.rng(302)
    p = 0.62
    ctl = cap.CapController(7, [1.0] * 8, z, 0.0, alpha=0.002, probe_every=4, probe_cap=2, p0=0.1)
    for _ in range(40_000):
        acc = r.random(5) < p
        ctl.update(5, 5 if acc.all() else int(np.argmin(acc)))
    assert abs(ctl.p() - p) < 0.03


def test_parks_when_speculation_loses_and_probes():
    verify = [10.0] * 8
    draft = [0.0] + [3.0 * k for k in range(1, 8)]   # each draft costs 30% of a plain step
    ctl = cap.CapController(7, verify, draft, 0.0, alpha=0.5, probe_every=3, probe_cap=2, p0=0.1)
    caps = [ctl.next_cap() for _ in range(7)]
    assert caps == [0, 0, 0, 2, 0, 0, 2]              # parked: plain steps plus a probe every third round
    ctl.update(2, 2)                                   # the probe accepted everything
    ctl.update(2, 2)
    assert not ctl.parked and ctl.next_cap() > 0


def test_knee():
    assert cap.knee([10, 10.2, 10.5, 10.9, 12.0, 15.0], 0.1) == 4
    assert cap.knee([10, 20], 0.1) == 1
    assert cap.knee([10] * 6, 0.0) == 6
