"""Pins for the oracle's Sequential Temperature Scaling and static-threshold
pruning (CPU only).

DSpark summary §3.2.1: STS calibrates the cumulative prefix survival on
held-out data with a left-to-right 1-D grid search that minimises each
position's Expected Calibration Error, the earlier positions' calibration
held fixed.  §4.3.3: a static threshold on the (calibrated) survival prunes
the verify length.

Pins: the temperature map's closed forms (T = 1 is the identity, 1/2 is fixed,
symmetry, sigmoid(z) -> sigmoid(z / T)); a hand-computed ECE; recovery of
known per-position miscalibrations from synthetic (confidence, outcome) pairs
drawn with the true acceptance probabilities; the argmin property at every
position; left-to-right independence; and the threshold's closed form for a
constant confidence.
"""
import numpy as np
import pytest

import oracle

GRID = oracle.sts_grid()
STEP = np.log(GRID[1] / GRID[0])


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def test_temper_closed_forms():
    assert GRID[60] == 1.0
    for c in [1e-6, 0.1, 0.37, 0.5, 0.8, 0.999]:
        assert oracle.temper(c, 1.0) == c
        for T in [0.3, 2.0, 7.5]:
            assert abs(oracle.temper(c, T) + oracle.temper(1 - c, T) - 1.0) < 1e-12
    for z in [-4.0, -0.5, 0.7, 3.0]:
        for T in [0.25, 1.7, 4.0]:
            assert abs(oracle.temper(_sigmoid(z), T) - _sigmoid(z / T)) < 1e-12
    assert oracle.temper(0.5, 3.0) == 0.5
    assert oracle.temper(0.0, 2.0) == 0.0 and oracle.temper(1.0, 2.0) == 1.0


def test_ece_hand_computed():
    # one position, two bins: [0, 0.5) holds 0.2 (y=0) and 0.4 (y=1): |0.2 + 0.4 - 1| = 0.4;
    # [0.5, 1] holds 0.6 and 0.9 (y=1 both): |1.5 - 2| = 0.5; ECE = 0.9 / 4 = 0.225
    c = np.array([[0.2], [0.4], [0.6], [0.9]], dtype=np.float32)
    y = np.array([[0], [1], [1], [1]], dtype=np.uint8)
    e = oracle.sts_ece(c, y, [1.0], bins=2)
    assert abs(e[0] - 0.225) < 1e-7  # the inputs are fp32-rounded


def _synthetic(rng, N, alphas):
    gam = len(alphas)
    p = rng.uniform(0.05, 0.95, size=(N, gam))
    y = (rng.uniform(size=(N, gam)) < p).astype(np.uint8)
    lp = np.log(p) - np.log1p(-p)
    c = _sigmoid(lp * np.asarray(alphas)).astype(np.float32)  # over/under-confident by alpha_k
    return c, y


def test_recovers_known_per_position_miscalibration():
    rng = np.random.default_rng(1)
    alphas = [2.0, 0.5, 1.0, 3.0]
    c, y = _synthetic(rng, 100_000, alphas)
    out = oracle.sts_calibrate(c, y, GRID)
    for k, a in enumerate(alphas):
        assert abs(np.log(out["temps"][k] / a)) <= 3 * STEP, (k, out["temps"][k], a)
    # calibrated: the error left is sampling noise
    assert (out["ece"] < 0.01).all()


def test_each_temperature_minimises_its_position_ece():
    rng = np.random.default_rng(2)
    c, y = _synthetic(rng, 5000, [1.5, 0.7, 2.5])
    out = oracle.sts_calibrate(c, y, GRID)
    for k in range(3):
        for g in GRID[::7]:
            t = out["temps"].copy()
            t[k] = g
            e = oracle.sts_ece(c, y, t)
            assert e[k] >= out["ece"][k] - 1e-12
        np.testing.assert_allclose(oracle.sts_ece(c, y, out["temps"])[k], out["ece"][k], rtol=1e-12)


def test_left_to_right():
    # the temperature of position k does not depend on the data of later positions
    rng = np.random.default_rng(3)
    c, y = _synthetic(rng, 4000, [1.5, 0.7, 2.5])
    t1 = oracle.sts_calibrate(c, y, GRID)["temps"]
    c2, y2 = c.copy(), y.copy()
    c2[:, 2] = rng.uniform(size=c.shape[0])
    y2[:, 2] = 1 - y2[:, 2]
    t2 = oracle.sts_calibrate(c2, y2, GRID)["temps"]
    assert t2[0] == t1[0] and t2[1] == t1[1]


def test_threshold_closed_form_and_monotone():
    # constant confidence p at T = 1: survival p^j, so l = floor(ln theta / ln p) (capped at gamma)
    for p in [0.9, 0.75, 0.5]:
        c = np.full((3, 12), p, dtype=np.float32)
        for theta in [0.9, 0.5, 0.2, 0.01]:
            want = min(12, int(np.floor(np.log(theta) / np.log(float(np.float32(p))) + 1e-9)))
            assert (oracle.schedule_threshold(c, theta) == want).all(), (p, theta)
    rng = np.random.default_rng(4)
    c = rng.uniform(0.3, 1.0, size=(50, 8)).astype(np.float32)
    temps = GRID[rng.integers(30, 90, size=8)]
    prev = None
    for theta in [0.0, 0.1, 0.3, 0.6, 0.9, 1.1]:
        ell = oracle.schedule_threshold(c, theta, temps)
        if theta == 0.0:
            assert (ell == 8).all()
        if theta > 1.0:
            assert (ell == 0).all()
        if prev is not None:
            assert (ell <= prev).all()
        prev = ell
