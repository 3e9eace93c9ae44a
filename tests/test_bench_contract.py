"""bench.py keeps the JSON-line contract: the reference arm (the oracle on the
host, runnable here) and our arm (on a GPU) each print one line with the keys
the measurement needs, in consistent units."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "tiny_r4_g4_v1024", "--steps", "3", "--warmup", "3"], 300)
    assert d["impl"] == "reference"
    assert d["metric"] and d["unit"] == "positions/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_r4_g4_v1024"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    d = _run(["--workload", "qwen3_r64_g16_v151936", "--R", "8", "--gamma", "4", "--steps", "3", "--warmup", "3",
              "--no-cpu-baseline"], 600)
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"]:
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("qwen3_r64_g16_v151936") and "l2" in d["config"]
    assert d["config"]["w2_layout"] == "transposed at setup"
    assert "prepare" not in d["kernels"]  # no per-round transpose
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    pl = rf["pipelined"]  # the draft step's period inside a whole draft call
    assert pl["draft_call_us"] > 0 and pl["draft_call_us_at_2"] > 0
    assert abs(pl["frac"] - pl["achieved"] / rf["peak"]) < 1e-9
    sp = rf["stream_probe"]
    assert sp["elements"] == 8 * 151936 and sp["gbs"] > 0 and sp["us"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    kr = d["kernels_roofline"]
    for k in ("verify_rows", "verify_draw"):  # full blocks at this workload: both run
        assert kr[k]["bytes_per_launch"] > 0 and kr[k]["us_per_launch"] > 0
        assert abs(kr[k]["frac"] - kr[k]["achieved_gbs"] / rf["peak"]) < 1e-9
    assert kr["verify_rows"]["rows"] == 8 * 4
    assert kr["verify_emit"]["us_per_launch"] > 0
    vp = d["verify_rows_probe"]
    assert vp["requests"] == 8 and vp["rows"] == 32 and vp["bytes_per_launch"] == 32 * 151936 * 6
    assert vp["us_per_launch"] > 0 and vp["frac"] > 0


@pytest.mark.gpu
def test_seeds_mode_line():
    # The serving report: rounds with seeds 0..N-1, each on its own inputs.
    d = _run(["--workload", "serving_r1024_g16_v129280", "--R", "16", "--seeds", "3", "--warmup", "3"], 600)
    assert d["steps"] == 3 and d["config"]["seeds"] == 3 and d["value"] > 0
    assert d["accepted_tokens_per_s"] > 0 and 3 * 16 <= d["emitted_tokens"] <= 3 * 16 * 17
    assert d["ms_per_round"]["min"] <= d["ms_per_step"] <= d["ms_per_round"]["max"] + 1e-9


@pytest.mark.gpu
def test_plain_w2_layout_line():
    # W2 passed as stored: every round's draft call transposes it itself.
    d = _run(["--workload", "qwen3_r64_g16_v151936", "--R", "8", "--gamma", "4", "--steps", "3", "--warmup", "3",
              "--no-cpu-baseline", "--w2-layout", "plain"], 600)
    assert d["config"]["w2_layout"] == "plain" and d["value"] > 0
    assert d["kernels"]["prepare"]["launches"] == 3
