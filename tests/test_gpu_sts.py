"""GPU-vs-oracle parity of Sequential Temperature Scaling and the static-threshold
scheduler through the C-ABI.

The temperature map runs in fp32 on the GPU and fp64 in the oracle, so a
chosen temperature may differ only where the oracle's own ECEs of the two
choices (same earlier temperatures) are within TIE of each other -- after such
a position the later ones are not compared; a threshold length may differ only
where the oracle's survival is within TIE of theta at the deciding position.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_05_gb300 as dspark

pytestmark = pytest.mark.gpu

TIE = 1e-6


def _synthetic(rng, N, alphas):
    p = rng.uniform(0.05, 0.95, size=(N, len(alphas)))
    y = (rng.uniform(size=p.shape) < p).astype(np.uint8)
    lp = np.log(p) - np.log1p(-p)
    c = (1.0 / (1.0 + np.exp(-lp * np.asarray(alphas)))).astype(np.float32)
    return c, y


def _gpu(c, y, grid, bins=15):
    dev = torch.device("cuda")
    out = dspark.dspark_sts_calibrate(torch.from_numpy(c).to(dev), torch.from_numpy(y).to(dev),
                                      torch.from_numpy(grid).to(dev), bins)
    torch.cuda.synchronize()
    return out["temps"].cpu().numpy(), out["ece"].cpu().numpy()


@pytest.mark.parametrize("N,alphas,bins", [(20000, [2.0, 0.5, 1.0, 3.0], 15),
                                           (200000, [1.3, 0.8, 2.2, 0.6, 1.0, 1.7, 0.9, 2.8], 15),
                                           (3000, [1.0, 2.0], 7)])
def test_sts_matches_the_oracle(N, alphas, bins):
    rng = np.random.default_rng(N)
    c, y = _synthetic(rng, N, alphas)
    grid = oracle.sts_grid()
    t_gpu, e_gpu = _gpu(c, y, grid, bins)
    ref = oracle.sts_calibrate(c, y, grid, bins)
    for k in range(len(alphas)):
        if t_gpu[k] != ref["temps"][k]:
            t = ref["temps"].copy()
            e_ref = oracle.sts_ece(c, y, t, bins)[k]
            t[k] = t_gpu[k]
            e_alt = oracle.sts_ece(c, y, t, bins)[k]
            assert abs(e_alt - e_ref) < TIE, (k, t_gpu[k], ref["temps"][k], e_alt, e_ref)
            break
        assert abs(e_gpu[k] - ref["ece"][k]) < TIE, (k, e_gpu[k], ref["ece"][k])
    # the GPU's temperatures are a good calibration by the oracle's own measure
    assert (oracle.sts_ece(c, y, t_gpu, bins) <= ref["ece"] + TIE).all()


@pytest.mark.parametrize("with_temps", [False, True])
def test_threshold_matches_the_oracle(with_temps):
    rng = np.random.default_rng(5 + with_temps)
    R, g = 4096, 12
    c = rng.uniform(0.5, 1.0, size=(R, g)).astype(np.float32)
    c[rng.uniform(size=(R, g)) < 0.02] = 1.0
    temps = oracle.sts_grid()[rng.integers(40, 80, size=g)] if with_temps else None
    dev = torch.device("cuda")
    for theta in [0.9, 0.5, 0.2, 0.05]:
        got = dspark.dspark_schedule_threshold(
            torch.from_numpy(c).to(dev), theta,
            None if temps is None else torch.from_numpy(temps).to(dev))["ell"].cpu().numpy()
        want = oracle.schedule_threshold(c, theta, temps)
        bad = np.nonzero(got != want)[0]
        for r in bad:
            a = np.cumprod([oracle.temper(float(v), 1.0 if temps is None else temps[j])
                            for j, v in enumerate(c[r])])
            j = min(got[r], want[r])  # the position where they decide differently
            assert abs(a[j] - theta) < TIE, (r, got[r], want[r], a[j], theta)
        assert len(bad) <= 2
