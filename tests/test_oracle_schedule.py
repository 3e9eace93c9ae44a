"""Pins for the oracle's prefix scheduler, Algorithm 1 (CPU only).

DSpark summary §3.2.2: a_{r,j} = prod_{i<=j} c_{r,i}; B = sum_r (1 + l_r);
tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); Theta = tau * SPS(B).  Candidates are
taken in survival order, which respects the prefix constraint and maximises
expected accepted tokens at fixed B; the search stops at the first candidate
that does not improve Theta, which finds the global maximum when Theta is
unimodal along the path.  Appendix A gives the worked counterexample.

Pins: brute-force enumeration of every allocation (l_1..l_R) in [0, gamma]^R
for tiny R and gamma; prefix monotonicity; the Appendix A numbers from
tests/golden/appendix_a.json; special cases (flat step rate -> full blocks,
c = 1 -> l = gamma, immediate stop).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix_a.json")


def _survival(c):
    return np.cumprod(np.asarray(c, dtype=np.float64), axis=1)


def _tau(a, ell):
    return sum(1.0 + a[r, :l].sum() for r, l in enumerate(ell))


def _all_allocations(R, g):
    return itertools.product(range(g + 1), repeat=R)


def test_prefix_monotonicity():
    rng = np.random.default_rng(0)
    for _ in range(50):
        R, g = rng.integers(1, 9), rng.integers(1, 17)
        c = rng.uniform(0, 1, size=(R, g)).astype(np.float32)
        c[rng.uniform(size=(R, g)) < 0.1] = 1.0
        s = oracle.schedule(c, np.ones(R * (1 + g) + 1))
        a = s["a"]
        assert (np.diff(a, axis=1) <= 0).all()
        np.testing.assert_allclose(a, _survival(c), rtol=1e-5)


@pytest.mark.parametrize("R,g", [(1, 4), (2, 3), (3, 2), (3, 4), (2, 4)])
def test_greedy_maximises_tau_at_every_batch_size(R, g):
    # A step-rate table that rises until B = R + n and then falls off a cliff
    # makes Algorithm 1 take exactly n candidates: its allocation must reach the
    # brute-force maximum of tau over all allocations with the same B.
    rng = np.random.default_rng(R * 10 + g)
    for trial in range(20):
        c = rng.uniform(0.05, 1.0, size=(R, g)).astype(np.float32)
        a = oracle.schedule(c, np.ones(R * (1 + g) + 1))["a"].astype(np.float64)
        best = {}
        for ell in _all_allocations(R, g):
            B = R + sum(ell)
            best[B] = max(best.get(B, -1.0), _tau(a, ell))
        for n in range(0, R * g + 1):
            sps = np.array([1e3 * (1 + b) if b <= R + n else 1e-6 for b in range(R * (1 + g) + 1)])
            s = oracle.schedule(c, sps)
            assert s["B"] == R + n
            assert abs(_tau(a, s["ell"]) - best[R + n]) < 1e-9
            assert abs(s["tau"] - best[R + n]) < 1e-9


@pytest.mark.parametrize("R,g", [(1, 4), (2, 3), (3, 3), (2, 4)])
def test_stops_at_global_theta_peak_when_unimodal(R, g):
    rng = np.random.default_rng(100 + R * 10 + g)
    checked = 0
    for trial in range(200):
        c = rng.uniform(0.05, 1.0, size=(R, g)).astype(np.float32)
        a = oracle.schedule(c, np.ones(R * (1 + g) + 1))["a"].astype(np.float64)
        B = np.arange(R * (1 + g) + 1, dtype=np.float64)
        sps = 1.0 / (rng.uniform(1e-3, 5e-3) + rng.uniform(1e-5, 5e-4) * B
                     + rng.uniform(0, 1e-5) * B * B)
        # Theta along Algorithm 1's path
        order = sorted(((a[r, j], j, r) for r in range(R) for j in range(g)),
                       key=lambda t: (-t[0], t[1], t[2]))
        tau, path = float(R), [R * sps[R]]
        for i, (av, _, _) in enumerate(order):
            tau += av
            path.append(tau * sps[R + i + 1])
        peak = int(np.argmax(path))
        unimodal = all(path[i] < path[i + 1] for i in range(peak)) and all(
            path[i] > path[i + 1] for i in range(peak, len(path) - 1))
        if not unimodal:
            continue
        checked += 1
        s = oracle.schedule(c, sps)
        glob = max(_tau(a, ell) * sps[R + sum(ell)] for ell in _all_allocations(R, g))
        assert abs(s["theta"] - glob) <= 1e-9 * glob
        assert abs(_tau(a, s["ell"]) * sps[R + int(s["ell"].sum())] - glob) <= 1e-9 * glob
    assert checked > 20


def test_appendix_a_counterexample_numbers():
    gold = json.load(open(GOLDEN))
    sps = np.array([0.0] + gold["sps_1_2_3"])
    for c2 in [0.9, 0.0]:
        c = np.array([[gold["a1"], c2]], dtype=np.float32)
        s = oracle.schedule(c, sps)
        # Theta_0 = 1 * SPS(1) = 1.0; Theta_1 = (1 + 0.8) * SPS(2) = 0.9 < Theta_0: stop.
        assert s["ell"].tolist() == [0]
        assert s["theta"] == pytest.approx(gold["theta0"], abs=1e-12)
        theta1 = (1.0 + float(np.float32(gold["a1"]))) * sps[2]
        assert theta1 == pytest.approx(gold["theta1"], abs=1e-7)


def test_full_blocks_under_flat_step_rate():
    rng = np.random.default_rng(5)
    R, g = 8, 16
    c = rng.uniform(0.01, 1, size=(R, g)).astype(np.float32)
    s = oracle.schedule(c, np.full(R * (1 + g) + 1, 250.0))
    assert s["ell"].tolist() == [g] * R
    s = oracle.schedule(np.ones((R, g), np.float32), np.full(R * (1 + g) + 1, 250.0))
    assert s["ell"].tolist() == [g] * R


def test_zero_survival_is_never_taken_under_flat_rate():
    c = np.array([[0.9, 0.0, 0.5], [1.0, 1.0, 1.0]], dtype=np.float32)
    s = oracle.schedule(c, np.full(10, 3.0))
    assert s["ell"].tolist() == [1, 3]


def test_steep_step_rate_takes_nothing():
    c = np.full((4, 4), 0.9, np.float32)
    sps = 1.0 / (1e-3 + 1.0 * np.arange(4 * 5 + 1))
    s = oracle.schedule(c, sps)
    assert s["ell"].tolist() == [0, 0, 0, 0]
    assert s["B"] == 4
