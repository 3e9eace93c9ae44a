"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: the GPU runs the whole round; the oracle recomputes a sample
of requests one by one (first, middle, last and random ones) and the whole
schedule.  Properties that hold at any size are checked on every request."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

from parity import compare_draft, compare_verify, f64, oracle_target_bias, torch_bias_rows

pytestmark = pytest.mark.gpu

FULL = ["verify_r512_g16_v151936", "qwen3_r64_g16_v151936", "largevocab_r256_g8_v262144",
        "serving_r1024_g16_v129280"]


def sampled_requests(R, n_random=2, seed=0):
    rng = np.random.default_rng(seed)
    s = {0, R // 2, R - 1, *rng.integers(0, R, size=n_random).tolist()}
    return sorted(s)


def round_sampled(w, seed, req, weights_seed=None):
    """One full-size round on the GPU; the oracle recomputes requests `req` and the
    whole schedule.  Returns what the comparisons need."""
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=seed, device=dev, weights_seed=weights_seed)
    gd = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], w.T, seed)
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    x0 = inp["x0"].cpu().numpy()
    od = oracle.draft(f64(inp["U"][req]), W1, W2, x0[req], w.T, seed, req_ids=req)
    ob = oracle_target_bias(W1, W2, x0[req], od["x"])
    where = {r: i for i, r in enumerate(req)}

    def bias_rows(i):
        if i in where:
            return torch.from_numpy(ob[where[i]]).to(dev)
        return torch_bias_rows(inp["W1"], inp["W2"], inp["x0"][i:i + 1], gd["x"][i:i + 1])[0]

    Z = workload.target_logits(w, inp["U"], seed, bias_rows=bias_rows)
    gs = dspark.dspark_schedule(inp["conf"], inp["sps"])
    gv = dspark.dspark_verify(gd["x"], gd["logp"], gd["lse"], gd["scores"], Z, gs["ell"], w.T, seed)
    torch.cuda.synchronize()
    for ws in (gd["workspace"], gs["workspace"], gv["workspace"]):
        assert dspark.dspark_read_device_status(ws) == 0

    osch = oracle.schedule(inp["conf"].cpu().numpy(), inp["sps"].cpu().numpy())
    ell = gs["ell"].cpu().numpy()
    assert (ell == osch["ell"]).all()
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z[req]), osch["ell"][req], w.T,
                       seed, req_ids=req)

    take = lambda t: t[req].cpu().numpy()
    gds = {k: take(gd[k]) for k in ["x", "logp", "lse"]}
    exempt = compare_draft(gds, od, w.dtype, scores_ref=od["scores"], scores_gpu=take(gd["scores"]))
    assert len(exempt) <= 1
    gvs = {k: take(gv[k]) for k in ["n_acc", "tokens", "n_emit", "cstar", "lse_t"]}
    compare_verify(gvs, ov, osch["ell"][req], w.dtype, skip=exempt)
    return inp, gd, gs, gv, ell


def check_structure(w, gd, gv, ell):
    """Properties that hold on every request at any size."""
    x = gd["x"].cpu().numpy()
    tok = gv["tokens"].cpu().numpy()
    n = gv["n_acc"].cpu().numpy()
    assert ((x >= 0) & (x < w.V)).all()
    assert (n >= 0).all() and (n <= ell).all()
    assert (gv["n_emit"].cpu().numpy() == n + 1).all()
    for i in range(w.R):
        assert (tok[i, :n[i]] == x[i, :n[i]]).all()
        assert 0 <= tok[i, n[i]] < w.V
        assert (tok[i, n[i] + 1:] == -1).all()


@pytest.mark.parametrize("name", FULL)
def test_full_size_round_sampled(name):
    w = workload.WORKLOADS[name]
    inp, gd, gs, gv, ell = round_sampled(w, 0, sampled_requests(w.R))
    check_structure(w, gd, gv, ell)
    # p^d is normalised on every row (sampled rows of the scores tensor)
    pd = torch.exp(gd["scores"][:: max(1, w.R // 8)] - gd["lse"][:: max(1, w.R // 8), :, None]).sum(-1)
    assert torch.allclose(pd, torch.ones_like(pd), atol=1e-4)


@pytest.mark.parametrize("seed", range(10))
def test_serving_round_per_seed(seed):
    # The serving workload's report runs 100 rounds with seeds 0..99, each on
    # its own U, x0, c and target logits (the draft head's weights from seed 0,
    # as in bench.py --seeds).  Seeds 0..9 at full size: two sampled requests
    # per seed against the oracle, the whole schedule bit-exact, and the
    # output structure on every request.
    w = workload.WORKLOADS["serving_r1024_g16_v129280"]
    req = sorted(set(np.random.default_rng(100 + seed).integers(0, w.R, size=2).tolist()))
    inp, gd, gs, gv, ell = round_sampled(w, seed, req, weights_seed=0)
    check_structure(w, gd, gv, ell)
    assert 0 < ell.sum() < w.R * w.gamma  # the serving schedule trims: mixed prefix lengths
