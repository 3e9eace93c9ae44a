"""Pins for the oracle's zero-overhead scheduler (CPU only).

DSpark summary §5.2: the serving scheduler predicts the next capacity K from
confidences two steps old -- without Algorithm 1's early stop, so that a
throughput cliff of an irregular SPS curve does not trap it in a local optimum
-- and then takes the top K current candidates by current cumulative
confidence (survival).  The capacity reading: K = the number of candidates at
the first global maximum of Theta = tau * SPS(B) along Algorithm 1's order.

Pins: brute force over every allocation (l_1..l_R) in [0, gamma]^R on tiny
cases (the capacity reaches the global Theta maximum over all allocations, and
top-K reaches the maximum tau at B = R + K); reduction to Algorithm 1 when
Theta is unimodal along the path; K never below Algorithm 1's count; and a
hand-computed cliff where Algorithm 1 stops at once and the capacity does not.
"""
import itertools

import numpy as np
import pytest

import oracle


def _tau(a, ell):
    return sum(1.0 + a[r, :l].sum() for r, l in enumerate(ell))


def _survival32(c):
    # the oracle's own survivals (sequential fp32 products), read back exactly
    return oracle.schedule(c, np.ones(c.size + c.shape[0] + 1))["a"].astype(np.float64)


def _irregular_sps(rng, n_b):
    # positive, piecewise: a smooth decay with random cliffs and plateaus
    t = 1e-3 + np.cumsum(rng.uniform(0, 4e-4, size=n_b))
    cliffs = rng.uniform(size=n_b) < 0.2
    t = t + np.cumsum(cliffs * rng.uniform(0, 3e-3, size=n_b))
    return 1.0 / t


@pytest.mark.parametrize("R,g", [(1, 4), (2, 3), (3, 2), (2, 4), (3, 3)])
def test_capacity_is_the_global_theta_maximum_over_all_allocations(R, g):
    rng = np.random.default_rng(7 * R + g)
    for trial in range(40):
        c = rng.uniform(0.05, 1.0, size=(R, g)).astype(np.float32)
        sps = _irregular_sps(rng, R * (1 + g) + 1)
        a = _survival32(c)
        best = {}
        for ell in itertools.product(range(g + 1), repeat=R):
            B = R + sum(ell)
            best[B] = max(best.get(B, -1.0), _tau(a, ell))
        theta = {B: t * sps[B] for B, t in best.items()}
        top = max(theta.values())
        cap = oracle.schedule_capacity(c, sps)
        assert cap["B"] == R + cap["K"]
        assert abs(cap["theta"] - top) <= 1e-12 * top
        # the first maximum: every smaller batch is strictly worse (beyond rounding)
        for B in range(R, cap["B"]):
            assert theta[B] < top * (1 - 1e-12)


@pytest.mark.parametrize("R,g", [(1, 4), (2, 3), (3, 3), (4, 4)])
def test_capacity_equals_algorithm1_when_theta_is_unimodal(R, g):
    rng = np.random.default_rng(300 + 10 * R + g)
    for trial in range(100):
        c = rng.uniform(0.05, 1.0, size=(R, g)).astype(np.float32)
        B = np.arange(R * (1 + g) + 1, dtype=np.float64)
        sps = 1.0 / (rng.uniform(1e-3, 5e-3) + rng.uniform(1e-5, 5e-4) * B)
        # tau is concave along the sorted order and 1/(alpha + beta B) is
        # log-concave, so Theta is unimodal along the path
        alg1 = oracle.schedule(c, sps)
        cap = oracle.schedule_capacity(c, sps)
        assert cap["K"] == alg1["n_taken"]
        assert cap["theta"] == alg1["theta"]


def test_capacity_never_below_algorithm1():
    rng = np.random.default_rng(11)
    for trial in range(300):
        R, g = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        c = rng.uniform(0.0, 1.0, size=(R, g)).astype(np.float32)
        sps = _irregular_sps(rng, R * (1 + g) + 1)
        assert oracle.schedule_capacity(c, sps)["K"] >= oracle.schedule(c, sps)["n_taken"]


def test_cliff_hand_computed():
    # One request, gamma = 4, c = 0.9 at every position: survivals 0.9, 0.81,
    # 0.729, 0.6561.  SPS(1) = 1, SPS(2..5) = 0.5 (a cliff right after B = 1).
    # Theta_0 = 1, Theta_1 = 1.9 * 0.5 = 0.95: Algorithm 1 stops at once (l = 0).
    # Along the whole path Theta_4 = (1 + 0.9 + 0.81 + 0.729 + 0.6561) * 0.5
    # = 2.04755 is the maximum, so the capacity is K = 4.
    c = np.full((1, 4), 0.9, dtype=np.float32)
    sps = np.array([0.0, 1.0, 0.5, 0.5, 0.5, 0.5])
    assert oracle.schedule(c, sps)["ell"].tolist() == [0]
    cap = oracle.schedule_capacity(c, sps)
    assert cap["K"] == 4 and cap["B"] == 5
    assert abs(cap["tau"] - 4.0951) < 1e-6
    assert abs(cap["theta"] - 2.04755) < 1e-6
    assert oracle.schedule_topk(c, cap["K"]).tolist() == [4]


@pytest.mark.parametrize("R,g", [(1, 4), (2, 3), (3, 3), (2, 4)])
def test_topk_reaches_the_best_tau_at_its_batch_size(R, g):
    rng = np.random.default_rng(500 + 10 * R + g)
    for trial in range(30):
        c = rng.uniform(0.05, 1.0, size=(R, g)).astype(np.float32)
        a = _survival32(c)
        best = {}
        for ell in itertools.product(range(g + 1), repeat=R):
            B = R + sum(ell)
            best[B] = max(best.get(B, -1.0), _tau(a, ell))
        for K in range(0, R * g + 3):
            ell = oracle.schedule_topk(c, K)
            assert ell.sum() == min(K, R * g)
            assert ((0 <= ell) & (ell <= g)).all()
            assert abs(_tau(a, ell) - best[R + min(K, R * g)]) < 1e-9


def test_topk_takes_highest_survival_first_and_ignores_old_confidences():
    # Non-anticipation: the selection sees the current confidences only
    # through their order, and the capacity only through K.
    rng = np.random.default_rng(3)
    R, g = 6, 5
    c_old = rng.uniform(0.1, 1.0, size=(R, g)).astype(np.float32)
    c_now = rng.uniform(0.1, 1.0, size=(R, g)).astype(np.float32)
    sps = _irregular_sps(rng, R * (1 + g) + 1)
    K = oracle.schedule_capacity(c_old, sps)["K"]
    ell = oracle.schedule_topk(c_now, K)
    a = _survival32(c_now)
    taken = [a[r, j] for r in range(R) for j in range(ell[r])]
    left = [a[r, j] for r in range(R) for j in range(ell[r], g)]
    if taken and left:
        assert min(taken) >= max(left)
    # the old confidences enter only through K
    c_other = rng.uniform(0.1, 1.0, size=(R, g)).astype(np.float32)
    K2 = oracle.schedule_capacity(c_other, sps)["K"]
    if K2 == K:
        assert (oracle.schedule_topk(c_now, K2) == ell).all()
