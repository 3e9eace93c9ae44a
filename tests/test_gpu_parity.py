"""GPU-vs-oracle parity through the C-ABI (dspark_draft_sample -> dspark_schedule
-> dspark_verify) on seeded synthetic workloads.

Small cases run the oracle on every request: several vocab tiles, a ragged
last tile, ragged 128-row blocks, both dtypes, T = 1 and T = 0.7, and
schedules that keep full blocks, trim everything, or mix.  Integer outputs
are bit-exact except documented near ties (tests/parity.py); floats within
1e-5 absolute (fp32 path) or 2e-3 relative (bf16 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

from parity import TIE, close, compare_draft, compare_verify, f64, oracle_target_bias

pytestmark = pytest.mark.gpu

W = workload.WORKLOADS
TINY = W["tiny_r4_g4_v1024"]
QWEN = W["qwen3_r64_g16_v151936"]
SERV = W["serving_r1024_g16_v129280"]
LARGE = W["largevocab_r256_g8_v262144"]

SMALL_CASES = [
    TINY,
    TINY.resized(name="tiny_T07_r9_v1000", R=9, V=1000, T=0.7),
    QWEN.resized(name="bf16_full_blocks_r130_g3_v1000_r64", R=130, gamma=3, V=1000, r=64),
    SERV.resized(name="bf16_mixed_r130_g4_v2056_r256", R=130, gamma=4, V=2056, r=256),
    LARGE.resized(name="bf16_T07_trimmed_r5_g2_v2056", R=5, gamma=2, V=2056),
    QWEN.resized(name="bf16_minimal_r1_g1_v8", R=1, gamma=1, V=8, r=64),
    SERV.resized(name="bf16_r257_g2_v4096_r128", R=257, gamma=2, V=4096, r=128),
]


def run_case(w, seed=0):
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=seed, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
    bias = oracle_target_bias(W1, W2, inp["x0"].numpy(), od["x"]) if w.z_bias else None
    Z = workload.target_logits(w, inp["U"], seed,
                               bias_rows=(lambda i: torch.from_numpy(bias[i])) if w.z_bias else None)
    osch = oracle.schedule(inp["conf"].numpy(), inp["sps"].numpy())
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), osch["ell"], w.T, seed)

    g = {k: v.to(dev) for k, v in inp.items()}
    gd = dspark.dspark_draft_sample(g["U"], g["W1"], g["W2"], g["x0"], w.T, seed)
    gs = dspark.dspark_schedule(g["conf"], g["sps"])
    gv = dspark.dspark_verify(gd["x"], gd["logp"], gd["lse"], gd["scores"], Z.to(dev), gs["ell"], w.T,
                              seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(gd["workspace"]) == 0
    assert dspark.dspark_read_device_status(gs["workspace"]) == 0
    assert dspark.dspark_read_device_status(gv["workspace"]) == 0
    cpu = lambda d: {k: v.cpu().numpy() for k, v in d.items() if isinstance(v, torch.Tensor) and k != "workspace"}
    return inp, Z, od, osch, ov, cpu(gd), cpu(gs), cpu(gv)


@pytest.mark.parametrize("w", SMALL_CASES, ids=lambda w: w.name)
def test_round_parity_small(w):
    inp, Z, od, osch, ov, gd, gs, gv = run_case(w)
    exempt = compare_draft(gd, od, w.dtype, scores_ref=od["scores"], scores_gpu=gd["scores"])
    assert len(exempt) <= max(1, w.R // 50), exempt
    assert (gs["ell"] == osch["ell"]).all()
    assert gs["diag"][0] == osch["B"] and gs["diag"][3] == osch["n_taken"]
    assert gs["diag"][1] == osch["tau"] and gs["diag"][2] == osch["theta"]
    ex_v = compare_verify(gv, ov, osch["ell"], w.dtype, skip=exempt)
    assert len(ex_v) <= max(1, w.R // 50) + len(exempt)
    # structure of the outputs
    for i in range(w.R):
        n = gv["n_acc"][i]
        assert 0 <= n <= gs["ell"][i]
        assert (gv["tokens"][i, :n] == gd["x"][i, :n]).all()
        assert 0 <= gv["tokens"][i, n] < w.V
        assert (gv["tokens"][i, n + 1:] == -1).all()
        assert np.isnan(gv["cstar"][i, gs["ell"][i]:]).all()


@pytest.mark.parametrize("R,gamma,V", [(40, 6, 3000 - 3000 % 8), (6, 3, 262144), (5, 2, 344064)],
                         ids=["v2992", "v262144", "v344064"])
def test_verify_parity_on_oracle_draft(R, gamma, V):
    # Verify alone, fed the oracle's draft outputs (rounded to fp32), with a
    # random schedule: every scheduled row is tested and its c* compared, at
    # vocabularies from a few tiles of the row loop to beyond 2^18.
    w = QWEN.resized(name="verify_only", R=R, gamma=gamma, V=V, r=64)
    seed = 5
    inp = workload.generate(w, seed=seed, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
    bias = oracle_target_bias(W1, W2, inp["x0"].numpy(), od["x"])
    Z = workload.target_logits(w, inp["U"], seed, bias_rows=lambda i: torch.from_numpy(bias[i]))
    ell = np.random.default_rng(0).integers(0, w.gamma + 1, size=w.R).astype(np.int32)
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), ell, w.T, seed)
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    gv = dspark.dspark_verify(t(od["x"], torch.int32), t(od["logp"], torch.float32),
                              t(od["lse"], torch.float32), t(od["scores"], torch.float32), Z.to(dev),
                              t(ell, torch.int32), w.T, seed)
    gv = {k: v.cpu().numpy() for k, v in gv.items() if isinstance(v, torch.Tensor) and k != "workspace"}
    ex = compare_verify(gv, ov, ell, w.dtype)
    assert len(ex) <= 1
    assert ell.sum() > 0
    if R >= 40:
        assert ov["n_acc"].sum() > 0 and (ov["n_acc"] < ell).any()  # both outcomes exercised


@pytest.mark.parametrize("R,V", [(1300, 1000), (700, 40008)], ids=["r1300_v1000", "r700_v40008"])
def test_verify_draw_four_groups_per_thread(R, V):
    # Enough requests that the draw takes four 32-id groups per thread (and, on
    # bonus rows, stages each warp's bf16 target rows in shared memory with one
    # bulk copy), with V % 32 = 8: the last group of a row holds 8 ids and the
    # last warp's copy is short.  gamma = 1 and a random schedule in {0, 1} mix
    # bonus draws from row 1 and row 2 with residual draws from row 1.
    w = QWEN.resized(name="draw_gpt4", R=R, gamma=1, V=V, r=64)
    seed = 11
    inp = workload.generate(w, seed=seed, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
    bias = oracle_target_bias(W1, W2, inp["x0"].numpy(), od["x"])
    Z = workload.target_logits(w, inp["U"], seed, bias_rows=lambda i: torch.from_numpy(bias[i]))
    ell = np.random.default_rng(1).integers(0, 2, size=w.R).astype(np.int32)
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), ell, w.T, seed)
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    gv = dspark.dspark_verify(t(od["x"], torch.int32), t(od["logp"], torch.float32),
                              t(od["lse"], torch.float32), t(od["scores"], torch.float32), Z.to(dev),
                              t(ell, torch.int32), w.T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(gv["workspace"]) == 0
    gv = {k: v.cpu().numpy() for k, v in gv.items() if isinstance(v, torch.Tensor) and k != "workspace"}
    ex = compare_verify(gv, ov, ell, w.dtype)
    assert len(ex) <= max(1, R // 200), ex
    # both draws exercised (a short last group read past the copied bytes
    # would carry garbage mass and win stage 1 far more often than the oracle)
    assert (ov["n_acc"] < ell).any() and (ov["n_acc"] == ell).any()


@pytest.mark.parametrize("name", workload.ORDER)
def test_schedule_parity_full_size(name):
    w = W[name]
    inp = workload.generate(w.resized(name=w.name, V=8), seed=0, device="cpu")  # conf/sps only
    osch = oracle.schedule(inp["conf"].numpy(), inp["sps"].numpy())
    gs = dspark.dspark_schedule(inp["conf"].cuda(), inp["sps"].cuda())
    ell = gs["ell"].cpu().numpy()
    diag = gs["diag"].cpu().numpy()
    assert (ell == osch["ell"]).all()
    assert diag[0] == osch["B"] and diag[1] == osch["tau"] and diag[2] == osch["theta"]


def test_schedule_ties_and_edges():
    rng = np.random.default_rng(3)
    cases = []
    for R, g in [(1, 1), (1, 64), (256, 64), (16384, 1), (1000, 16), (3, 7)]:
        c = rng.uniform(0, 1, size=(R, g)).astype(np.float32)
        c[rng.uniform(size=(R, g)) < 0.2] = 1.0  # equal survivals along a request
        c[rng.uniform(size=(R, g)) < 0.05] = 0.0
        if R > 2:
            c[1] = c[0]  # identical requests: ties broken by request id
        B = np.arange(R * (1 + g) + 1, dtype=np.float64)
        for sps in [np.full(B.shape, 250.0), 1.0 / (1e-3 + 2e-5 * B), 1.0 / (6e-3 + 1e-5 * B + 4e-9 * B * B)]:
            cases.append((c, sps))
    for c, sps in cases:
        osch = oracle.schedule(c, sps)
        gs = dspark.dspark_schedule(torch.from_numpy(c).cuda(), torch.from_numpy(sps).cuda())
        assert (gs["ell"].cpu().numpy() == osch["ell"]).all()
        assert gs["diag"].cpu().numpy()[2] == osch["theta"]


def test_device_status_flags_bad_inputs():
    dev = torch.device("cuda")
    c = torch.tensor([[0.5, float("nan")], [1.5, -0.1]], dtype=torch.float32, device=dev)
    sps = torch.full((7,), 10.0, dtype=torch.float64, device=dev)
    gs = dspark.dspark_schedule(c, sps)
    assert dspark.dspark_read_device_status(gs["workspace"]) & 1
    osch = oracle.schedule(c.cpu().numpy(), sps.cpu().numpy())
    assert (gs["ell"].cpu().numpy() == osch["ell"]).all()
    w = TINY
    inp = workload.generate(w, seed=0, device=dev)
    x0 = inp["x0"].clone()
    x0[1] = w.V + 5
    gd = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], x0, w.T, 0)
    assert dspark.dspark_read_device_status(gd["workspace"]) & 1
    ell = torch.tensor([0, 9, -1, 2], dtype=torch.int32, device=dev)
    Z = torch.randn(w.R, w.gamma + 1, w.V, device=dev)
    gv = dspark.dspark_verify(gd["x"], gd["logp"], gd["lse"], gd["scores"], Z, ell, w.T, 0)
    assert dspark.dspark_read_device_status(gv["workspace"]) & 1
    tok = gv["tokens"].cpu().numpy()
    assert ((tok >= -1) & (tok < w.V)).all()


def test_host_errors_raise():
    dev = torch.device("cuda")
    w = TINY
    inp = workload.generate(w, seed=0, device=dev)
    with pytest.raises(dspark.DSparkError):
        dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], 0.0, 0)
    with pytest.raises(dspark.DSparkError):
        dspark.dspark_schedule(inp["conf"], inp["sps"][:5])


def test_replay_is_deterministic():
    w = SMALL_CASES[3]
    a = run_case(w, seed=11)
    b = run_case(w, seed=11)
    for k in ["x", "logp", "lse"]:
        assert (a[5][k] == b[5][k]).all()
    for k in ["tokens", "n_acc", "cstar"]:
        assert np.array_equal(a[7][k], b[7][k], equal_nan=True)


def test_target_equal_to_draft_accepts_every_token():
    # The degenerate case p^t = p^d ([summary] §3, rejection sampling): every
    # scheduled token is accepted (ln u < 0 = ln p^t - ln p^d) and
    # c* = sum min(p^d, p^t) = 1.  fp32 path, fed the oracle's draft, with the
    # target rows j <= gamma equal to the oracle's draft scores times T; the
    # bonus row is an ordinary logit row, so the bonus draw is compared too.
    w = TINY.resized(name="tiny_same_r64_g4_v1024", R=64, T=0.8)
    seed = 9
    inp = workload.generate(w, seed=seed, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
    Z = np.empty((w.R, w.gamma + 1, w.V), dtype=np.float32)
    Z[:, : w.gamma] = (od["scores"] * w.T).astype(np.float32)
    Z[:, w.gamma] = inp["U"][:, -1].numpy()
    ell = np.full(w.R, w.gamma, dtype=np.int32)
    ell[::7] = np.arange(len(ell[::7])) % (w.gamma + 1)  # some shorter prefixes
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], Z.astype(np.float64), ell, w.T, seed)
    assert (ov["n_acc"] == ell).all()
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    gv = dspark.dspark_verify(t(od["x"], torch.int32), t(od["logp"], torch.float32),
                              t(od["lse"], torch.float32), t(od["scores"], torch.float32),
                              t(Z, torch.float32), t(ell, torch.int32), w.T, seed)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in gv.items() if isinstance(v, torch.Tensor) and k != "workspace"}
    assert (g["n_acc"] == ell).all()
    assert (g["n_emit"] == ell + 1).all()
    for i in range(w.R):
        assert np.abs(g["cstar"][i, : ell[i]] - 1.0).max(initial=0.0) < 1e-5
        assert np.isnan(g["cstar"][i, ell[i]:]).all()
    assert (g["tokens"] == ov["tokens"]).all()  # accepted drafts, then the bonus draw from p^t


def test_stream_probe_converts_exactly():
    # The bandwidth probe bench.py times: out = float(in), every element.
    dev = torch.device("cuda")
    x = (torch.randn(8 * 100003, device=dev) * 3).to(torch.bfloat16)
    y = torch.full(x.shape, float("nan"), device=dev)
    dspark.dspark_stream_probe(x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, x.float())
