"""Draft-cap choice from measured verify costs and live acceptance.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see the package docstring).

What it computes, from the pages:

* mlx-dspark PyPI page, "The Apple-Silicon speedup ceiling": tokens per
  second ~ A / (drafter + overhead + slope * C) for accept length A and draft
  cap C; the verify cost term is measured, not assumed.  Here the verify cost
  of a round of width M = 1 + C is the measured curve ``verify_us[C]`` itself
  (the pages' slope * C is its linear summary), so one round costs
  ``T(C) = draft_us[C] + overhead_us + verify_us[C]``.
* mlx-dspark wiki page, "Key techniques" (hardware-aware auto-calibration):
  the controller picks the cap per round from the cached curves and a live
  acceptance EWMA, with expected_committed = 1 + sum_i p^i, and drops to a
  cap-0 "parked" mode when speculation is losing.
* PyPI page, "Tuning" (--max-draft auto): while parked it runs plain steps
  plus periodic probe rounds, so the acceptance estimate stays current.

[reading] The pages do not say how the EWMA is formed.  Here it is the
exponentially weighted maximum-likelihood estimate of a geometric acceptance
model: a round that verified C drafts and accepted a of them contributes a
successes and, when a < C, one failure; S and F are EWMAs of those counts
and p = S / (S + F).  The best cap maximises E(C) / T(C) with
E(C) = sum_{i=0}^{C} p^i (the committed target token plus the expected
accepted prefix), ties going to the smaller cap.
"""


def expected_committed(p, cap):
    """1 + p + p^2 + ... + p^cap: tokens a round of `cap` drafts commits on
    average when each draft position is accepted with probability p given
    that all earlier ones were."""
    total, term = 0.0, 1.0
    for _ in range(cap + 1):
        total += term
        term *= p
    return total


def round_us(verify_us, draft_us, overhead_us, cap):
    return draft_us[cap] + overhead_us + verify_us[cap]


def best_cap(p, verify_us, draft_us, overhead_us, max_cap):
    """argmax over C in [0, max_cap] of E(C) / T(C); the smallest C on ties."""
    best, best_rate = 0, None
    for c in range(max_cap + 1):
        rate = expected_committed(p, c) / round_us(verify_us, draft_us, overhead_us, c)
        if best_rate is None or rate > best_rate:
            best, best_rate = c, rate
    return best, best_rate


class CapController:
    """Per-round cap choice.  verify_us[C] and draft_us[C] for C = 0..max_cap."""

    def __init__(self, max_cap, verify_us, draft_us, overhead_us, alpha, probe_every, probe_cap, p0):
        self.max_cap, self.alpha = max_cap, alpha
        self.verify_us, self.draft_us, self.overhead_us = list(verify_us), list(draft_us), overhead_us
        self.probe_every, self.probe_cap = probe_every, probe_cap
        self.S, self.F = p0, 1.0 - p0          # the prior counts as one round's worth of evidence
        self.parked, self.since_probe = False, 0

    def p(self):
        tot = self.S + self.F
        return self.S / tot if tot > 0 else 0.0

    def next_cap(self):
        if self.parked:
            self.since_probe += 1
            if self.since_probe >= self.probe_every:
                self.since_probe = 0
                return self.probe_cap
            return 0
        cap, _ = best_cap(self.p(), self.verify_us, self.draft_us, self.overhead_us, self.max_cap)
        if cap == 0:
            self.parked, self.since_probe = True, 0
        return cap

    def update(self, cap, accepted):
        """Record a round that verified `cap` drafts and accepted `accepted`."""
        if cap <= 0:
            return
        a = self.alpha
        self.S = (1.0 - a) * self.S + a * accepted
        self.F = (1.0 - a) * self.F + a * (1.0 if accepted < cap else 0.0)
        if self.parked:
            cap_now, _ = best_cap(self.p(), self.verify_us, self.draft_us, self.overhead_us, self.max_cap)
            if cap_now > 0:
                self.parked = False


def knee(verify_us, tol):
    """Widest round M = 1 + C whose cost stays within (1 + tol) of width 1:
    the end of the cheap verify region (PyPI page, "Results at a glance")."""
    base = verify_us[0]
    m = 1
    for c, t in enumerate(verify_us):
        if t <= (1.0 + tol) * base:
            m = c + 1
        else:
            break
    return m
