"""Verify over packed target logits (dspark_verify_packed) through the C-ABI.

An engine that lets requests verify different lengths emits the target rows
of all requests back to back; request r's rows for positions 1..l_r+1 start
at row_offsets[r].  The packed call must give exactly the outputs of the
padded call on the same rows -- and so match the oracle run on the padded
layout -- while never touching rows it was not given: the test pads every
request with a random number of extra NaN rows, which any stray read would
spread into the outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

from parity import compare_verify, f64, oracle_target_bias

pytestmark = pytest.mark.gpu

W = workload.WORKLOADS


def _inputs(w, seed):
    inp = workload.generate(w, seed=seed, device="cpu")
    W1, W2 = f64(inp["W1"]), f64(inp["W2"])
    od = oracle.draft(f64(inp["U"]), W1, W2, inp["x0"].numpy(), w.T, seed)
    bias = oracle_target_bias(W1, W2, inp["x0"].numpy(), od["x"]) if w.z_bias else None
    Z = workload.target_logits(w, inp["U"], seed,
                               bias_rows=(lambda i: torch.from_numpy(bias[i])) if w.z_bias else None)
    return od, Z


def _pack(Z, ell, rng):
    """Zp, row offsets [R + 1]: request r's rows 1..l_r+1, then 0-2 NaN rows."""
    R, g1, V = Z.shape
    rows, offsets = [], [0]
    for r in range(R):
        rows.append(Z[r, : ell[r] + 1])
        extra = int(rng.integers(0, 3))
        if extra:
            rows.append(torch.full((extra, V), float("nan"), dtype=Z.dtype))
        offsets.append(offsets[-1] + ell[r] + 1 + extra)
    return torch.cat(rows).contiguous(), np.array(offsets, dtype=np.int32)


CASES = [
    (W["qwen3_r64_g16_v151936"].resized(name="packed_bf16_r40_g6_v2992", R=40, gamma=6, V=2992, r=64), 5),
    (W["tiny_r4_g4_v1024"].resized(name="packed_f32_r9_g4_v1000", R=9, V=1000), 1),
    (W["qwen3_r64_g16_v151936"].resized(name="packed_bf16_r6_g3_v262144", R=6, gamma=3, V=262144, r=64), 2),
]


@pytest.mark.parametrize("w,seed", CASES, ids=[c[0].name for c in CASES])
def test_packed_verify_matches_padded_and_oracle(w, seed):
    od, Z = _inputs(w, seed)
    rng = np.random.default_rng(seed)
    ell = rng.integers(0, w.gamma + 1, size=w.R).astype(np.int32)
    ell[0] = w.gamma  # a full block, and (below) a request with nothing scheduled
    ell[-1] = 0
    Zp, offsets = _pack(Z, ell, rng)
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    args = (t(od["x"], torch.int32), t(od["logp"], torch.float32), t(od["lse"], torch.float32),
            t(od["scores"], torch.float32))
    dense = dspark.dspark_verify(*args, Z.to(dev), t(ell, torch.int32), w.T, seed)
    packed = dspark.dspark_verify_packed(*args, Zp.to(dev), t(offsets, torch.int32), t(ell, torch.int32),
                                         w.T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(packed["workspace"]) == 0
    host = lambda d: {k: v.cpu().numpy() for k, v in d.items() if isinstance(v, torch.Tensor) and k != "workspace"}
    gd, gp = host(dense), host(packed)
    for k in ("n_acc", "n_emit", "tokens"):
        assert (gd[k] == gp[k]).all(), k
    for k in ("cstar", "lse_t"):
        assert np.array_equal(gd[k], gp[k], equal_nan=True), k
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), ell, w.T, seed)
    assert len(compare_verify(gp, ov, ell, w.dtype)) <= 1


def test_packed_offsets_that_miss_rows_are_flagged():
    w = CASES[0][0].resized(name="packed_short", R=8, gamma=4, V=1000)
    od, Z = _inputs(w, 3)
    ell = np.full(w.R, 2, dtype=np.int32)
    Zp, offsets = _pack(Z, ell, np.random.default_rng(0))
    offsets[5] = offsets[4] + 1  # request 4 now has one row where it needs three
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    out = dspark.dspark_verify_packed(t(od["x"], torch.int32), t(od["logp"], torch.float32),
                                      t(od["lse"], torch.float32), t(od["scores"], torch.float32),
                                      Zp.to(dev), t(offsets, torch.int32), t(ell, torch.int32), w.T, 3)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(out["workspace"]) & 1  # DSPARK_DEV_BAD_INPUT
