"""GPU-vs-oracle parity of the zero-overhead scheduling calls through the C-ABI
(dspark_schedule_capacity -> dspark_schedule_topk): the capacity K, its
diagnostics and the selected lengths l_r are bit-exact, on random and
workload confidences with smooth and irregular (cliff) step-rate tables."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

pytestmark = pytest.mark.gpu


def _irregular_sps(rng, n_b):
    t = 1e-3 + np.cumsum(rng.uniform(0, 4e-4, size=n_b))
    cliffs = rng.uniform(size=n_b) < 0.2
    t = t + np.cumsum(cliffs * rng.uniform(0, 3e-3, size=n_b))
    return 1.0 / t


def _gpu_capacity_topk(c_old, c_now, sps, extra_k=()):
    dev = torch.device("cuda")
    co = torch.from_numpy(c_old).to(dev)
    cn = torch.from_numpy(c_now).to(dev)
    s = torch.from_numpy(sps).to(dev)
    cap = dspark.dspark_schedule_capacity(co, s)
    sel = dspark.dspark_schedule_topk(cn, cap["K"])  # K stays on the device
    out = {"K": int(cap["K"].item()), "diag": cap["diag"].cpu().numpy(), "ell": sel["ell"].cpu().numpy()}
    out["extra"] = {}
    for k in extra_k:
        kk = torch.tensor([k], dtype=torch.int32, device=dev)
        out["extra"][k] = dspark.dspark_schedule_topk(cn, kk)["ell"].cpu().numpy()
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(cap["workspace"]) == 0
    assert dspark.dspark_read_device_status(sel["workspace"]) == 0
    return out


@pytest.mark.parametrize("R,g", [(1, 4), (3, 5), (130, 4), (512, 16), (1024, 16)])
def test_capacity_and_topk_match_the_oracle(R, g):
    rng = np.random.default_rng(R + 100 * g)
    for trial in range(3):
        c_old = rng.uniform(0.0, 1.0, size=(R, g)).astype(np.float32)
        c_now = rng.uniform(0.0, 1.0, size=(R, g)).astype(np.float32)
        c_old[rng.uniform(size=(R, g)) < 0.05] = 1.0  # survival ties
        sps = _irregular_sps(rng, R * (1 + g) + 1)
        n = R * g
        got = _gpu_capacity_topk(c_old, c_now, sps, extra_k=(0, 1, n // 2, n, n + 7))
        ref = oracle.schedule_capacity(c_old, sps)
        assert got["K"] == ref["K"]
        assert got["diag"][0] == ref["B"] and got["diag"][3] == ref["K"]
        assert got["diag"][1] == ref["tau"] and got["diag"][2] == ref["theta"]
        assert (got["ell"] == oracle.schedule_topk(c_now, ref["K"])).all()
        for k, ell in got["extra"].items():
            assert (ell == oracle.schedule_topk(c_now, k)).all(), k


@pytest.mark.parametrize("name", ["verify_r512_g16_v151936", "serving_r1024_g16_v129280"])
def test_capacity_on_workload_confidences(name):
    w = workload.WORKLOADS[name]
    inp = workload.generate(w.resized(name=w.name, V=8), seed=0, device="cpu")
    c = inp["conf"].numpy()
    sps = inp["sps"].numpy()
    got = _gpu_capacity_topk(c, c, sps)
    ref = oracle.schedule_capacity(c, sps)
    assert got["K"] == ref["K"] and got["diag"][2] == ref["theta"]
    assert (got["ell"] == oracle.schedule_topk(c, ref["K"])).all()
    # both workloads' tables make Theta unimodal along the path: ZOS's
    # capacity is then Algorithm 1's count
    assert ref["K"] == oracle.schedule(c, sps)["n_taken"]


def test_throughput_cliff():
    # Algorithm 1 stops at once (l = 0); the capacity looks past the cliff (K = 4).
    c = np.full((1, 4), 0.9, dtype=np.float32)
    sps = np.array([0.0, 1.0, 0.5, 0.5, 0.5, 0.5])
    got = _gpu_capacity_topk(c, c, sps)
    assert got["K"] == 4 and got["ell"].tolist() == [4]
    dev = torch.device("cuda")
    alg1 = dspark.dspark_schedule(torch.from_numpy(c).to(dev), torch.from_numpy(sps).to(dev))
    assert alg1["ell"].cpu().tolist() == [0]
