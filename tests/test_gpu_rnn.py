"""GPU-vs-oracle parity of the RNN-head draft (dspark_draft_sample_rnn) through
the C-ABI.

The state runs in fp32 on the GPU and in fp64 in the oracle, and both round it
to bf16 for the contraction.  Where the two states straddle a bf16 rounding
boundary one element of A differs by one bf16 step (at most 2^-8 for |h| < 1),
which moves the bias by at most 2^-8 * max|W2| (about 4e-4 for these weights).
The scores get an exact allowance on top of the Markov draft's tolerance (2e-3
relative): for every state element whose oracle value lies within H_EPS of a
bf16 rounding midpoint (so that the fp32 state may round the other way), one
bf16 step times |W2[a, v]| / T.  A drafted token may differ from the oracle's
only where the oracle's Gumbel margin is below twice the position's largest
allowance (two keys moving apart), and never where it is 1e-3 or more.
H_EPS = 2e-5 bounds the fp32 state's error: an r-term fp32 sum (r <= 256,
terms below 0.15 here) plus tanhf, carried through a contractive Wh.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

from parity import compare_draft, f64

pytestmark = pytest.mark.gpu

RNN_TIE = 1e-3
H_EPS = 2e-5
W = workload.WORKLOADS
CASES = [
    W["qwen3_r64_g16_v151936"].resized(name="rnn_r130_g4_v2056_r64", R=130, gamma=4, V=2056, r=64),
    W["serving_r1024_g16_v129280"].resized(name="rnn_r257_g3_v4096_r128", R=257, gamma=3, V=4096, r=128),
    W["verify_r512_g16_v151936"].resized(name="rnn_r64_g8_v3000_r256", R=64, gamma=8, V=3000, r=256),
]


def _straddle_allowance(h, W2, T):
    """[n, gamma, V]: sum over the state elements within H_EPS of a bf16 midpoint of
    (the bf16 step there) * |W2[a, v]| / T."""
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    lo, hi = to_bf16(h - H_EPS), to_bf16(h + H_EPS)
    step = np.abs(hi - lo)  # 0 unless h - H_EPS and h + H_EPS round apart
    return np.einsum("nga,av->ngv", step, np.abs(W2)) / T


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_rnn_draft_matches_the_oracle(w):
    seed = 3
    inp = workload.generate(w, seed=seed, device="cpu")
    rin = workload.rnn_inputs(w, seed=seed, device="cpu")
    od = oracle.draft_rnn(f64(inp["U"]), f64(inp["W1"]), f64(inp["W2"]), f64(rin["Wh"]), f64(rin["Q"]),
                          inp["x0"].numpy(), w.T, seed, want_state=True)
    extra = _straddle_allowance(od["h"], f64(inp["W2"]), w.T)
    tie = np.maximum(RNN_TIE, 2 * extra.max(axis=-1))
    dev = torch.device("cuda")
    gd = dspark.dspark_draft_sample_rnn(inp["U"].to(dev), inp["W1"].to(dev), inp["W2"].to(dev),
                                        rin["Wh"].to(dev), rin["Q"].to(dev), inp["x0"].to(dev), w.T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(gd["workspace"]) == 0
    g = {k: v.cpu().numpy() for k, v in gd.items() if k != "workspace"}
    exempt = compare_draft(g, od, w.dtype, scores_ref=od["scores"], scores_gpu=g["scores"], tie=tie,
                           score_extra=extra)
    assert len(exempt) <= max(1, w.R // 50), exempt
    # the recurrence matters: the Markov draft of the same inputs picks other tokens
    mk = dspark.dspark_draft_sample(inp["U"].to(dev), inp["W1"].to(dev), inp["W2"].to(dev),
                                    inp["x0"].to(dev), w.T, seed)
    assert (mk["x"].cpu().numpy() != g["x"]).any()


@pytest.mark.parametrize("name", ["verify_r512_g16_v151936", "qwen3_r64_g16_v151936"])
def test_rnn_draft_full_size_sampled(name):
    # The RNN draft at a workload's full size, in the launch configuration the
    # benchmark times (bench.py --head rnn): the oracle recomputes a sample of
    # requests one by one (first, middle, last and two random ones); every row's
    # p^d is normalised and every token is in range.
    w = W[name]
    seed = 0
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=seed, device=dev)
    rin = workload.rnn_inputs(w, seed=seed, device=dev)
    gd = dspark.dspark_draft_sample_rnn(inp["U"], inp["W1"], inp["W2"], rin["Wh"], rin["Q"], inp["x0"], w.T,
                                        seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(gd["workspace"]) == 0
    rng = np.random.default_rng(0)
    req = sorted({0, w.R // 2, w.R - 1, *rng.integers(0, w.R, size=2).tolist()})
    od = oracle.draft_rnn(f64(inp["U"][req]), f64(inp["W1"]), f64(inp["W2"]), f64(rin["Wh"]), f64(rin["Q"][req]),
                          inp["x0"].cpu().numpy()[req], w.T, seed, req_ids=req, want_state=True)
    extra = _straddle_allowance(od["h"], f64(inp["W2"]), w.T)
    tie = np.maximum(RNN_TIE, 2 * extra.max(axis=-1))
    take = lambda t: t[req].cpu().numpy()
    g = {k: take(gd[k]) for k in ["x", "logp", "lse"]}
    exempt = compare_draft(g, od, w.dtype, scores_ref=od["scores"], scores_gpu=take(gd["scores"]), tie=tie,
                           score_extra=extra)
    assert len(exempt) <= 1, exempt
    x = gd["x"].cpu().numpy()
    assert ((x >= 0) & (x < w.V)).all()
    step = max(1, w.R // 8)
    pd = torch.exp(gd["scores"][::step] - gd["lse"][::step, :, None]).sum(-1)
    assert torch.allclose(pd, torch.ones_like(pd), atol=1e-4)
