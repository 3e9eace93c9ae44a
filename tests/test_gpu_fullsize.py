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


@pytest.mark.parametrize("name", FULL)
def test_full_size_round_sampled(name):
    w = workload.WORKLOADS[name]
    seed = 0
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=seed, device=dev)
    gd = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], w.T, seed)
    req = sampled_requests(w.R)
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

    # every request: output structure
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
    # p^d is normalised on every row (sampled rows of the scores tensor)
    pd = torch.exp(gd["scores"][:: max(1, w.R // 8)] - gd["lse"][:: max(1, w.R // 8), :, None]).sum(-1)
    assert torch.allclose(pd, torch.ones_like(pd), atol=1e-4)
