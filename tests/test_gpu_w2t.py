"""The draft with the head's second factor given in the tensor cores' layout
(dspark_transpose_w2 once, then dspark_draft_sample_w2t / _rnn_w2t) gives the
same outputs, bit for bit, as the calls that take W2 as stored and transpose
it themselves; and one case against the oracle directly."""
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

from parity import compare_draft, f64

pytestmark = pytest.mark.gpu

W = workload.WORKLOADS
CASES = [
    W["qwen3_r64_g16_v151936"].resized(name="w2t_r64_g3_v2056_r64", R=64, gamma=3, V=2056, r=64),
    W["serving_r1024_g16_v129280"].resized(name="w2t_r257_g2_v4096_r128", R=257, gamma=2, V=4096, r=128),
    W["verify_r512_g16_v151936"].resized(name="w2t_r130_g4_v3000_r256", R=130, gamma=4, V=3000, r=256),
]
KEYS = ("x", "logp", "lse", "scores")


def test_transpose_w2_is_the_transpose():
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(5)
    for r, V in [(64, 8), (128, 1000), (256, 4104)]:
        W2 = torch.randn(r, V, generator=g).to(torch.bfloat16).to(dev)
        W2T = dspark.dspark_transpose_w2(W2)
        torch.cuda.synchronize()
        assert W2T.shape == (V, r)
        assert torch.equal(W2T.cpu(), W2.cpu().t().contiguous())


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_draft_w2t_equals_draft(w):
    dev = torch.device("cuda")
    seed = 7
    g = {k: v.to(dev) for k, v in workload.generate(w, seed=seed, device="cpu").items()}
    ref = dspark.dspark_draft_sample(g["U"], g["W1"], g["W2"], g["x0"], w.T, seed)
    W2T = dspark.dspark_transpose_w2(g["W2"])
    out = dspark.dspark_draft_sample_w2t(g["U"], g["W1"], W2T, g["x0"], w.T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(out["workspace"]) == 0
    for k in KEYS:
        assert torch.equal(out[k], ref[k]), k


def test_draft_w2t_matches_the_oracle():
    w = CASES[2]
    seed = 11
    inp = workload.generate(w, seed=seed, device="cpu")
    od = oracle.draft(f64(inp["U"]), f64(inp["W1"]), f64(inp["W2"]), inp["x0"].numpy(), w.T, seed)
    dev = torch.device("cuda")
    g = {k: v.to(dev) for k, v in inp.items()}
    W2T = dspark.dspark_transpose_w2(g["W2"])
    gd = dspark.dspark_draft_sample_w2t(g["U"], g["W1"], W2T, g["x0"], w.T, seed)
    torch.cuda.synchronize()
    gd = {k: gd[k].cpu().numpy() for k in KEYS}
    exempt = compare_draft(gd, od, w.dtype, scores_ref=od["scores"], scores_gpu=gd["scores"])
    assert len(exempt) <= max(1, w.R // 50), exempt


def test_rnn_draft_w2t_equals_rnn_draft():
    w = CASES[1]
    seed = 3
    dev = torch.device("cuda")
    g = {k: v.to(dev) for k, v in workload.generate(w, seed=seed, device="cpu").items()}
    rin = {k: v.to(dev) for k, v in workload.rnn_inputs(w, seed=seed, device="cpu").items()}
    ref = dspark.dspark_draft_sample_rnn(g["U"], g["W1"], g["W2"], rin["Wh"], rin["Q"], g["x0"], w.T, seed)
    W2T = dspark.dspark_transpose_w2(g["W2"])
    out = dspark.dspark_draft_sample_rnn_w2t(g["U"], g["W1"], W2T, rin["Wh"], rin["Q"], g["x0"], w.T,
                                             seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(out["workspace"]) == 0
    for k in KEYS:
        assert torch.equal(out[k], ref[k]), k


def test_draft_w2t_equals_draft_full_vocab():
    # The serving workload's shapes (R = 1024 requests, V = 129,280, r = 256) at two
    # positions: eight row tiles of 19 column slots each over 1,010 vocab tiles.
    w = W["serving_r1024_g16_v129280"].resized(gamma=2)
    dev = torch.device("cuda")
    seed = 4
    g = {k: v.to(dev) for k, v in workload.generate(w, seed=seed, device="cpu").items()}
    ref = dspark.dspark_draft_sample(g["U"], g["W1"], g["W2"], g["x0"], w.T, seed)
    W2T = dspark.dspark_transpose_w2(g["W2"])
    out = dspark.dspark_draft_sample_w2t(g["U"], g["W1"], W2T, g["x0"], w.T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(out["workspace"]) == 0
    for k in KEYS:
        assert torch.equal(out[k], ref[k]), k
