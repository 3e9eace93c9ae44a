"""The library keeps no state between calls, so a draft and a schedule issued on
two streams at once (as an engine overlaps them: the schedule reads only the
confidences and the step-rate table) give exactly the results of the same calls
issued one after the other, and the verify that waits for both is unchanged."""
import pytest
import torch

from speculative_decoding_draft_05_gb300 import workload
import speculative_decoding_draft_05_gb300 as dspark

pytestmark = pytest.mark.gpu

W = workload.WORKLOADS


def _schedule(inp, scheduler):
    if scheduler == "zos":
        cap = dspark.dspark_schedule_capacity(inp["conf"], inp["sps"])
        return dspark.dspark_schedule_topk(inp["conf"], cap["K"])
    return dspark.dspark_schedule(inp["conf"], inp["sps"])


def _round(w, inp, Z, side=None, W2T=None, scheduler="alg1", host=True):
    dev = torch.device("cuda")
    main = torch.cuda.current_stream()
    if side is not None:
        side.wait_stream(main)
        with torch.cuda.stream(side):
            sch = _schedule(inp, scheduler)
    if W2T is not None:
        d = dspark.dspark_draft_sample_w2t(inp["U"], inp["W1"], W2T, inp["x0"], w.T, 11)
    else:
        d = dspark.dspark_draft_sample(inp["U"], inp["W1"], inp["W2"], inp["x0"], w.T, 11)
    if side is None:
        sch = _schedule(inp, scheduler)
    else:
        main.wait_stream(side)
    v = dspark.dspark_verify(d["x"], d["logp"], d["lse"], d["scores"], Z, sch["ell"], w.T, 11)
    torch.cuda.synchronize(dev)
    out = {k: (t.cpu() if host else t) for k, t in list(d.items()) + list(sch.items()) + list(v.items())
           if isinstance(t, torch.Tensor) and k != "workspace"}
    return out


@pytest.mark.parametrize("w", [W["qwen3_r64_g16_v151936"].resized(name="streams_r200_g6_v4096", R=200, gamma=6,
                                                                  V=4096, r=128)], ids=lambda w: w.name)
def test_draft_and_schedule_on_two_streams_match_serial(w):
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=5, device=dev)
    Z = workload.target_logits(w, inp["U"], 5, bias_rows=lambda i: torch.zeros(w.gamma + 1, w.V, device=dev))
    serial = _round(w, inp, Z)
    side = torch.cuda.Stream(dev)
    for _ in range(3):
        overlapped = _round(w, inp, Z, side)
        assert serial.keys() == overlapped.keys()
        for k in serial:
            assert torch.equal(serial[k].nan_to_num(), overlapped[k].nan_to_num()), k


@pytest.mark.parametrize("scheduler", ["alg1", "zos"])
def test_full_size_round_on_two_streams_matches_serial(scheduler):
    # The serving workload at full size: 16 tensor-core draft steps on every SM
    # while the scheduler's kernels (16,384 candidates) share the SMs beside
    # them, the draft reading a W2^T prepared once.
    w = W["serving_r1024_g16_v129280"]
    dev = torch.device("cuda")
    inp = workload.generate(w, seed=2, device=dev)
    Z = workload.target_logits(w, inp["U"], 2, bias_rows=lambda i: torch.zeros(w.gamma + 1, w.V, device=dev))
    W2T = dspark.dspark_transpose_w2(inp["W2"])
    serial = _round(w, inp, Z, W2T=W2T, scheduler=scheduler, host=False)
    side = torch.cuda.Stream(dev)
    for _ in range(2):
        overlapped = _round(w, inp, Z, side, W2T=W2T, scheduler=scheduler, host=False)
        assert serial.keys() == overlapped.keys()
        for k in serial:
            assert torch.equal(serial[k].nan_to_num(), overlapped[k].nan_to_num()), k
        del overlapped
