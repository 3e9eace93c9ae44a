"""dspark_verify_noalloc: the verify entry point for callers that cannot
allocate device memory (for example an engine whose device memory is all
pre-assigned to fixed pools, or code that must not trigger a synchronising
cudaMalloc in the middle of a round).  It keeps its scratch in a static device
array instead of a caller workspace.

Checked here through the C-ABI: on two calls in a row it must give what
dspark_verify gives on the same inputs (integers exactly, floats within the
parity tolerances), and it must refuse problems whose scratch would not fit.
This file is collected last so that a failure here comes after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_draft_05_gb300 as dspark
from speculative_decoding_draft_05_gb300 import binding, workload

pytestmark = pytest.mark.gpu

F32_ATOL = 1e-5   # fp32 path
BF16_RTOL = 2e-3  # bf16-input path


def _lib():
    L = binding.load()
    P, I, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    L.dspark_verify_noalloc.argtypes = [P, P, P, P, P, I, P, I, I, I, F, U64, P, P, P, P, P, P]
    L.dspark_verify_noalloc.restype = I
    return L


def _noalloc(L, d, Z, ell, T, seed):
    R, g = d["x"].shape
    V = d["scores"].shape[2]
    dev = Z.device
    out = dict(n_acc=torch.full((R,), -7, dtype=torch.int32, device=dev),
               tokens=torch.full((R, g + 1), -7, dtype=torch.int32, device=dev),
               n_emit=torch.full((R,), -7, dtype=torch.int32, device=dev),
               cstar=torch.full((R, g), 7.0, device=dev),
               lse_t=torch.full((R, g + 1), 7.0, device=dev))
    code = binding.DSPARK_BF16 if Z.dtype == torch.bfloat16 else binding.DSPARK_F32
    st = L.dspark_verify_noalloc(
        d["x"].data_ptr(), d["logp"].data_ptr(), d["lse"].data_ptr(), d["scores"].data_ptr(),
        Z.data_ptr(), code, ell.data_ptr(), R, g, V, T, seed, out["n_acc"].data_ptr(),
        out["tokens"].data_ptr(), out["n_emit"].data_ptr(), out["cstar"].data_ptr(),
        out["lse_t"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, L.dspark_last_error().decode()
    return out


def _compare(a, b, dtype):
    for k in ["n_acc", "tokens", "n_emit"]:
        assert torch.equal(a[k], b[k]), k
    for k in ["cstar", "lse_t"]:
        x, y = a[k].double().cpu().numpy(), b[k].double().cpu().numpy()
        assert (np.isnan(x) == np.isnan(y)).all(), k
        m = ~np.isnan(y)
        if dtype == "f32":
            assert np.abs(x[m] - y[m]).max(initial=0.0) <= F32_ATOL, k
        else:
            assert (np.abs(x[m] - y[m]) <= BF16_RTOL * np.abs(y[m]) + 1e-6).all(), k


@pytest.mark.parametrize("w", [
    workload.WORKLOADS["tiny_r4_g4_v1024"],
    workload.WORKLOADS["serving_r1024_g16_v129280"].resized(name="noalloc_bf16_r130_g4_v2056", R=130,
                                                            gamma=4, V=2056),
], ids=lambda w: w.name)
def test_noalloc_verify_matches_workspace_verify_twice(w):
    L = _lib()
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=3, device=dev)
    d = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], w.T, 3)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    Z = inp["U"].float()
    Z = torch.cat([Z, Z[:, -1:]], dim=1) + 3.0 * torch.randn(w.R, w.gamma + 1, w.V, device=dev, generator=gen)
    Z = Z.to(w.torch_dtype).contiguous()
    ell = torch.full((w.R,), w.gamma, dtype=torch.int32, device=dev)
    ell[::3] = 0  # bonus-only requests beside full blocks
    for call, seed in enumerate([3, 4]):  # two calls in a row on the shared static scratch
        ref = dspark.dspark_verify(d["x"], d["logp"], d["lse"], d["scores"], Z, ell, w.T, seed)
        got = _noalloc(L, d, Z, ell, w.T, seed)
        torch.cuda.synchronize()
        _compare(got, ref, w.dtype)
    assert (ref["n_acc"] < ell).any()  # rejections (residual draws) were exercised


def test_noalloc_verify_matches_the_oracle_twice():
    # Self-standing parity: the no-alloc entry point fed the oracle's draft
    # outputs (rounded to fp32) and target logits built along the oracle's
    # tokens, against the oracle's verify, on two calls in a row.
    import oracle
    from parity import compare_verify, f64, oracle_target_bias

    w = workload.WORKLOADS["serving_r1024_g16_v129280"].resized(name="noalloc_oracle_r40_g4_v2056", R=40,
                                                               gamma=4, V=2056, r=64)
    inp = workload.generate(w, seed=5, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    L = _lib()
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    ell = np.random.default_rng(1).integers(0, w.gamma + 1, size=w.R).astype(np.int32)
    for seed in (5, 6):
        od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
        bias = oracle_target_bias(W1, W2, inp["x0"].numpy(), od["x"])
        Z = workload.target_logits(w, inp["U"], seed, bias_rows=lambda i: torch.from_numpy(bias[i]))
        ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), ell, w.T, seed)
        d = dict(x=t(od["x"], torch.int32), logp=t(od["logp"], torch.float32),
                 lse=t(od["lse"], torch.float32), scores=t(od["scores"], torch.float32))
        got = _noalloc(L, d, Z.to(dev), t(ell, torch.int32), w.T, seed)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in got.items()}
        ex = compare_verify(g, ov, ell, w.dtype)
        assert len(ex) <= 1


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = _lib()
    R, g, V = 40000, 16, 1024  # more than 4 R (3 g + 1) bytes > 4 MiB of scratch
    p = 256  # never dereferenced: the size check comes before any device work
    st = L.dspark_verify_noalloc(p, p, p, p, p, binding.DSPARK_BF16, p, R, g, V, 1.0, 0, p, p, p, p, None,
                                 None)
    assert st == 2
    assert b"static array" in L.dspark_last_error()
