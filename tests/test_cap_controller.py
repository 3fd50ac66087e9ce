"""The library's draft-cap controller (host code behind the C ABI) against the
cap oracle.  No GPU: these calls do no device work."""

import numpy as np
import pytest

from oracle import cap as ocap
import synthetic
from speculative_decoding_verify_qmm_gb300 import binding
from speculative_decoding_verify_qmm_gb300.binding import SVError, SV_EINVAL


@pytest.fixture(scope="module")
def clib():
    from speculative_decoding_verify_qmm_gb300 import build
    build.build()
    return binding.load_library()


def _curves(r, n):
    verify = list(np.cumsum(r.uniform(0.0, 2.0, n)) + 20.0)
    if n > 1 and r.random() < 0.5:              # sometimes a cliff past a knee
        k = int(r.integers(1, n))
        verify = [v + (30.0 if i >= k else 0.0) for i, v in enumerate(verify)]
    draft = [0.0] + list(np.cumsum(r.uniform(0.2, 3.0, n - 1)))
    return verify, draft


def test_expected_committed_matches_oracle(clib):
    for p in (0.0, 0.25, 0.7, 1.0):
        for c in (0, 1, 7, 31):
            assert clib.sv_expected_committed(p, c) == ocap.expected_committed(p, c)


def test_best_cap_matches_oracle(clib):
    r = synthetic.rng(310)
    for _ in range(300):
        n = int(r.integers(1, 33))
        verify, draft = _curves(r, n)
        p, over = float(r.random()), float(r.uniform(0, 5))
        got = binding.best_cap(clib, p, verify, draft, over)
        want = ocap.best_cap(p, verify, draft, over, n - 1)
        assert got[0] == want[0] and got[1] == want[1]


def test_controller_sequence_matches_oracle(clib):
    r = synthetic.rng(311)
    for trial in range(20):
        n = int(r.integers(2, 17))
        verify, draft = _curves(r, n)
        args = (n - 1, verify, draft, float(r.uniform(0, 3)), float(r.uniform(0.05, 1.0)),
                int(r.integers(1, 6)), int(r.integers(1, n)), float(r.random()))
        got, want = binding.CapController(clib, *args), ocap.CapController(*args)
        p_true = float(r.random())
        for _ in range(200):
            c = got.next_cap()
            assert c == want.next_cap()
            acc = r.random(c) < p_true
            a = c if acc.all() else int(np.argmin(acc))
            got.update(c, a)
            want.update(c, a)
            assert got.p() == want.p() and got.parked == want.parked


def test_knee_matches_oracle(clib):
    r = synthetic.rng(312)
    for _ in range(100):
        verify, _ = _curves(r, int(r.integers(1, 33)))
        tol = float(r.uniform(0, 0.5))
        assert binding.verify_knee(clib, verify, tol) == ocap.knee(verify, tol)


def test_rejections(clib):
    with pytest.raises(SVError) as e:
        binding.best_cap(clib, 1.5, [1.0, 2.0], [0.0, 1.0], 0.0)
    assert e.value.status == SV_EINVAL
    with pytest.raises(SVError):
        binding.best_cap(clib, 0.5, [1.0, -2.0], [0.0, 1.0], 0.0)
    with pytest.raises(SVError):
        binding.CapController(clib, 3, [1.0] * 4, [0.0] * 4, 0.0, 0.0, 1, 1, 0.5)   # alpha 0
    ctl = binding.CapController(clib, 3, [1.0] * 4, [0.0] * 4, 0.0, 0.5, 1, 1, 0.5)
    with pytest.raises(SVError):
        ctl.update(2, 3)                                                          # accepted > cap
