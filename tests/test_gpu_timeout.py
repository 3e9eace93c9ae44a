"""The bounded device waits of the tensor-core draft, made to run out.

Every mbarrier wait in the draft kernel gives up after a limit of SM clocks:
the role that timed out raises the CTA's abort flag, the other roles see it and
leave, copies already issued are waited for, tensor memory is freed and the
call's device status word gets DSPARK_DEV_TIMEOUT.  The diagnostic entry point
dspark_selftest_draft_timeout runs draft step 1 with the W2 operand loads
withheld (nothing will ever complete the contraction's first wait) and a short
limit, so this path runs on purpose, on a small grid, without any fault.
Afterwards the context must still be usable: an ordinary draft on the same
inputs runs clean and matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_05_gb300 as dspark
from speculative_decoding_draft_05_gb300 import binding, workload

from parity import f64

pytestmark = pytest.mark.gpu


def test_draft_wait_timeout_sets_status_and_context_survives():
    w = workload.WORKLOADS["qwen3_r64_g16_v151936"].resized(name="timeout_r130_g1_v1000_r64", R=130,
                                                             gamma=1, V=1000, r=64)
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=0, device=dev)
    ws = binding.dspark_selftest_draft_timeout(inp["U"], inp["W1"], inp["W2"], inp["x0"],
                                               wait_cycles=200_000)
    torch.cuda.synchronize()
    status = dspark.dspark_read_device_status(ws)
    assert status & binding.DEV_TIMEOUT, status
    assert not status & binding.DEV_BAD_INPUT, status

    # the context survives: the same workspace, an ordinary draft, a clean status
    gd = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], w.T, 0, workspace=ws)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(ws) == 0
    od = oracle.draft(f64(inp["U"]), f64(inp["W1"]), f64(inp["W2"]), inp["x0"].cpu().numpy(), w.T, 0)
    x = gd["x"].cpu().numpy()
    differ = x != od["x"]
    assert (od["margin"][differ] < 1e-5).all()
    assert differ.sum() <= 1


def test_selftest_rejects_bad_limits():
    w = workload.WORKLOADS["qwen3_r64_g16_v151936"].resized(name="timeout_args", R=4, gamma=1, V=1000,
                                                             r=64)
    inp = workload.generate(w, seed=0, device=torch.device("cuda"))
    for bad in (0, 999, 5_000_000_000):
        with pytest.raises(dspark.DSparkError):
            binding.dspark_selftest_draft_timeout(inp["U"], inp["W1"], inp["W2"], inp["x0"], wait_cycles=bad)
