#!/usr/bin/env python
"""Benchmark of the DSpark per-round sampling path on GB300.

One step = one full round (dspark_draft_sample -> dspark_schedule ->
dspark_verify) over one batch of synthetic input already resident in HBM.
Metric: draft+verify positions/s = R * gamma / round time (whole job over all
ranks).  Default workload: R = 512 requests, gamma = 16, V = 151936, r = 256,
bf16 inputs (verify_r512_g16_v151936).  The draft head's weights stay fixed
across rounds, so its W2 is transposed once at setup into the layout the
tensor-core draft reads (dspark_transpose_w2) and every round calls
dspark_draft_sample_w2t; --w2-layout plain passes W2 as stored instead and each
round's draft call transposes it (a read and a write of r V bf16).

Also reported on the same JSON line:
  roofline      the dominant kernel (the draft contraction + epilogue) timed with
                CUDA events on its own launch stream over a second timed region
                of the same K steps (the first, which gives the value, runs
                without per-launch events), algorithmic bytes per launch /
                average launch time vs the measured HBM copy bandwidth;
  e2e           the same metric through the C-ABI with pinned HOST buffers: every
                step copies that step's inputs host->device and reads the result
                (tokens, counts, c*, l) back;
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload on
                this host's cores (rank 0, N = 1 only);
  clocks        nvidia-smi SM clocks and throttle reasons sampled during the
                timed region.

--impl reference times the CPU oracle as the reference arm (rank 0 only).
Multi-GPU (torchrun): every rank runs an independent replica (the path has no
data-path collective); time = max over ranks; value = all ranks' positions / time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_draft_05_gb300 import workload  # noqa: E402

METRIC = "draft+verify positions/s"
DEFAULT_WORKLOAD = "verify_r512_g16_v151936"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DRAFT_TILE_SOURCES = ["speculative_decoding_draft_05_gb300/csrc/draft.cu",
                      "speculative_decoding_draft_05_gb300/csrc/draft_tc.cu"]


# ----------------------------------------------------------------------------- helpers
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for rel in DRAFT_TILE_SOURCES + ["speculative_decoding_draft_05_gb300/csrc/common.cuh",
                                     "speculative_decoding_draft_05_gb300/csrc/ptx.cuh"]:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """dram bytes per draft-tile launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "draft_tile_dram.txt")
    if not os.path.exists(p):
        return None
    fields = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_digest") != source_digest():
        return None
    if fields.get("workload") != workload_name:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in [("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")]:
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- the round
class Round:
    """Device buffers of one round and the three C-ABI calls on one stream."""

    def __init__(self, w: workload.Workload, seed: int, device, scheduler: str = "alg1",
                 verify_layout: str = "padded", head: str = "markov", w2_layout: str = "transposed"):
        import speculative_decoding_draft_05_gb300 as dspark

        self.dspark = dspark
        self.w, self.seed, self.device = w, seed, device
        self.scheduler = scheduler
        self.packed = verify_layout == "packed"
        self.rnn = workload.rnn_inputs(w, seed=seed, device=device) if head == "rnn" else None
        inp = workload.generate(w, seed=seed, device=device)
        self.inp = inp
        # The head's second factor in the tensor cores' K-major layout, written once
        # here as the weights are loaded (they stay fixed across rounds); each round's
        # draft then reads it as is.  w2_layout "plain": every draft call transposes W2.
        self.w2t = None
        if (w2_layout == "transposed" and w.dtype == "bf16" and w.r % 64 == 0 and w.r <= 256
                and w.V % 8 == 0):
            self.w2t = dspark.dspark_transpose_w2(inp["W2"])
        R, g, V = w.R, w.gamma, w.V
        f32, i32 = torch.float32, torch.int32
        self.x = torch.empty(R, g, dtype=i32, device=device)
        self.logp = torch.empty(R, g, dtype=f32, device=device)
        self.lse = torch.empty(R, g, dtype=f32, device=device)
        self.scores = torch.empty(R, g, V, dtype=f32, device=device)
        self.ell = torch.empty(R, dtype=i32, device=device)
        self.diag = torch.empty(4, dtype=torch.float64, device=device)
        self.n_acc = torch.empty(R, dtype=i32, device=device)
        self.tokens = torch.empty(R, g + 1, dtype=i32, device=device)
        self.n_emit = torch.empty(R, dtype=i32, device=device)
        self.cstar = torch.empty(R, g, dtype=f32, device=device)
        self.lse_t = torch.empty(R, g + 1, dtype=f32, device=device)
        u8 = torch.uint8
        ws_draft = (dspark.draft_rnn_workspace_bytes(R, g, V, w.r) if head == "rnn"
                    else dspark.draft_workspace_bytes(R, g, V, w.r, w.torch_dtype))
        self.ws_d = torch.empty(ws_draft, dtype=u8, device=device)
        self.ws_s = torch.empty(dspark.schedule_workspace_bytes(R, g), dtype=u8, device=device)
        self.ws_s2 = torch.empty(dspark.schedule_workspace_bytes(R, g), dtype=u8, device=device)
        self.K = torch.empty(1, dtype=i32, device=device)
        # The schedule reads only the confidences and the step-rate table, not the
        # drafted tokens, so it runs on a side stream beside the draft.
        self.side = torch.cuda.Stream(device) if torch.cuda.is_available() else None
        self.ws_v = torch.empty(dspark.verify_workspace_bytes(R, g, V), dtype=u8, device=device)
        # Target logits: the workload's target stand-in carries the Markov bias
        # along the draft's own tokens; run the (deterministic) draft once, untimed.
        self.draft()
        torch.cuda.synchronize(device)
        self.Z = self._target_logits()
        torch.cuda.synchronize(device)
        if self.packed:
            # An engine's packed target output: request r's rows 1..l_r+1 back
            # to back.  l does not change between rounds here (the workload's
            # confidences and step rates are fixed), so the rows are packed once.
            self.schedule()
            rows = (1 + self.ell.long())
            self.offsets = torch.cat([torch.zeros(1, dtype=torch.long, device=device),
                                      torch.cumsum(rows, 0)]).to(torch.int32)
            req = torch.repeat_interleave(torch.arange(R, device=device), rows)
            pos = torch.arange(int(rows.sum().item()), device=device) - self.offsets[:-1].long()[req]
            self.Zp = self.Z[req, pos].contiguous()
            del self.Z
            torch.cuda.synchronize(device)

    def _target_logits(self, seed=None, out=None):
        w, inp = self.w, self.inp
        seed = self.seed if seed is None else seed
        if not w.z_bias:
            return workload.target_logits(w, inp["U"], seed, out=out)
        W1f = inp["W1"].float()
        W2f = inp["W2"].float()
        x0, x = inp["x0"], self.x

        def bias_rows(i):
            prev = torch.cat([x0[i:i + 1].long(), x[i].long()])
            return W1f[prev] @ W2f

        return workload.target_logits(w, inp["U"], seed, bias_rows=bias_rows, out=out)

    def reseed(self, seed: int):
        """New round inputs for `seed` (untimed): U, x0 and c drawn from that seed,
        the draft head's weights kept, and the target stand-in rebuilt along the
        draft's tokens under that seed's Philox key.  Buffers are reused."""
        new = workload.generate(self.w, seed=seed, device=self.device, weights_seed=self.seed)
        for k in ("U", "x0", "conf"):
            self.inp[k].copy_(new[k])
        del new
        self.draft(seed)
        torch.cuda.synchronize(self.device)
        self._target_logits(seed, out=self.Z)
        torch.cuda.synchronize(self.device)

    def draft(self, seed=None, U=None, W1=None, W2=None, x0=None, Wh=None, Q=None):
        """The draft call; W2 is the head's second factor in this round's layout
        (W2^T [V, r] where it was transposed at setup, else W2 [r, V])."""
        i = self.inp
        seed = self.seed if seed is None else seed
        U = i["U"] if U is None else U
        W1 = i["W1"] if W1 is None else W1
        W2 = (self.w2t if self.w2t is not None else i["W2"]) if W2 is None else W2
        x0 = i["x0"] if x0 is None else x0
        kw = dict(x=self.x, logp=self.logp, lse=self.lse, scores=self.scores, workspace=self.ws_d)
        d = self.dspark
        if self.rnn is not None:
            Wh = self.rnn["Wh"] if Wh is None else Wh
            Q = self.rnn["Q"] if Q is None else Q
            if self.w2t is not None:
                d.dspark_draft_sample_rnn_w2t(U, W1, W2, Wh, Q, x0, self.w.T, seed, **kw)
            else:
                d.dspark_draft_sample_rnn(U, W1, W2, Wh, Q, x0, self.w.T, seed, **kw)
        elif self.w2t is not None:
            d.dspark_draft_sample_w2t(U, W1, W2, x0, self.w.T, seed, **kw)
        else:
            d.dspark_draft_sample(U, W1, W2, x0, self.w.T, seed, **kw)

    def schedule(self, conf=None, sps=None):
        d = self.dspark
        conf = self.inp["conf"] if conf is None else conf
        sps = self.inp["sps"] if sps is None else sps
        if self.scheduler == "zos":
            # Zero-overhead scheduling: capacity from the confidences of two
            # rounds back -- the same tensor here, the workload's confidences
            # being fixed -- then the top K of the current ones.
            d.dspark_schedule_capacity(conf, sps, K=self.K, diag=self.diag, workspace=self.ws_s)
            d.dspark_schedule_topk(conf, self.K, ell=self.ell, workspace=self.ws_s2)
        else:
            d.dspark_schedule(conf, sps, ell=self.ell, diag=self.diag, workspace=self.ws_s)

    def step(self, seed=None, inputs=None):
        """One round; `seed` keys the round's Philox draws (default: the input seed);
        `inputs` is a list like input_tensors() (default: the resident inputs)."""
        ins = self.input_tensors() if inputs is None else inputs
        U, W1, W2, x0, conf, sps, Z = ins[:7]
        d = self.dspark
        seed = self.seed if seed is None else seed
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)  # the round's inputs are in place
        with torch.cuda.stream(self.side):
            self.schedule(conf, sps)
        if self.rnn is not None:
            self.draft(seed, U, W1, W2, x0, ins[-2], ins[-1])
        else:
            self.draft(seed, U, W1, W2, x0)
        main.wait_stream(self.side)  # verify needs l
        if self.packed:
            d.dspark_verify_packed(self.x, self.logp, self.lse, self.scores, Z, ins[7], self.ell,
                                   self.w.T, seed, n_acc=self.n_acc, tokens=self.tokens,
                                   n_emit=self.n_emit, cstar=self.cstar, lse_t=self.lse_t,
                                   workspace=self.ws_v)
        else:
            d.dspark_verify(self.x, self.logp, self.lse, self.scores, Z, self.ell, self.w.T, seed,
                            n_acc=self.n_acc, tokens=self.tokens, n_emit=self.n_emit,
                            cstar=self.cstar, lse_t=self.lse_t, workspace=self.ws_v)

    def input_tensors(self):
        i = self.inp
        ins = [i["U"], i["W1"], i["W2"] if self.w2t is None else self.w2t, i["x0"], i["conf"], i["sps"]]
        ins += [self.Zp, self.offsets] if self.packed else [self.Z]
        if self.rnn is not None:
            ins += [self.rnn["Wh"], self.rnn["Q"]]
        return ins

    def result_tensors(self):
        return [self.tokens, self.n_emit, self.n_acc, self.cstar, self.ell]


def draft_tile_bytes(w: workload.Workload) -> int:
    """Algorithmic bytes of one draft-contraction launch (one position k):
    U_k read (R*V*e) + scores write (R*V*4) + W2 read (r*V*e) + A_k read (R*r*e)."""
    e = 4 if w.dtype == "f32" else 2
    return w.R * w.V * (e + 4) + w.r * w.V * e + w.R * w.r * e


def round_bytes(w: workload.Workload, ell, transpose: bool = True) -> int:
    """Algorithmic HBM bytes of one round: the W2 transpose (read + write) where the
    round does it, gamma draft steps, and verify -- the Z rows of the scheduled
    positions and of the drawn token (sum(l) + R rows) and the draft scores of the
    scheduled rows."""
    e = 4 if w.dtype == "f32" else 2
    rows = int(ell.sum().item())
    return ((2 * w.r * w.V * e if transpose else 0) + w.gamma * draft_tile_bytes(w)
            + (rows + w.R) * w.V * e + rows * w.V * 4)


def draft_tile_flops(w: workload.Workload) -> int:
    return 2 * w.R * w.r * w.V


def verify_rows_bytes(w: workload.Workload, rows: int) -> int:
    """Algorithmic bytes of the verify row kernel over `rows` scheduled rows: each
    row's target logits once from HBM (its second pass hits L2) and its draft
    scores once."""
    e = 4 if w.dtype == "f32" else 2
    return rows * w.V * (e + 4)


def verify_draw_bytes(w: workload.Workload, residual_rows: int) -> int:
    """Algorithmic bytes of the draw (stage 1): one target row per request, plus the
    draft scores of the rows drawn from a residual."""
    e = 4 if w.dtype == "f32" else 2
    return w.R * w.V * e + residual_rows * w.V * 4


def draft_step_period(rnd, w, device, seed, hbm_peak, reps: int = 10) -> dict:
    """Per-step period of the draft in a whole draft call, from CUDA events around
    the call at gamma and at 2 positions: (t_gamma - t_2) / (gamma - 2).  The two
    calls share the call's fixed costs (resets, the final combine)."""
    d = rnd.dspark
    R, V, r = w.R, w.V, w.r
    U2 = rnd.inp["U"][:, :2, :].contiguous()
    out2 = dict(x=torch.empty(R, 2, dtype=torch.int32, device=device),
                logp=torch.empty(R, 2, dtype=torch.float32, device=device),
                lse=torch.empty(R, 2, dtype=torch.float32, device=device),
                scores=torch.empty(R, 2, V, dtype=torch.float32, device=device),
                workspace=torch.empty(d.draft_workspace_bytes(R, 2, V, r, torch.bfloat16),
                                      dtype=torch.uint8, device=device))
    i = rnd.inp

    def call2():
        if rnd.w2t is not None:
            d.dspark_draft_sample_w2t(U2, i["W1"], rnd.w2t, i["x0"], w.T, seed, **out2)
        else:
            d.dspark_draft_sample(U2, i["W1"], i["W2"], i["x0"], w.T, seed, **out2)

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps / 1e3

    t_full = timed(lambda: rnd.draft(seed))
    t_two = timed(call2)
    del U2, out2
    step = (t_full - t_two) / (w.gamma - 2)
    nbytes = draft_tile_bytes(w)
    return {"method": "draft call alone with CUDA events at gamma and at 2 positions; "
                      "per step = difference / (gamma - 2); not part of value",
            "draft_call_us": t_full * 1e6, "draft_call_us_at_2": t_two * 1e6,
            "per_step_us": step * 1e6, "achieved": nbytes / step / 1e9,
            "frac": nbytes / step / 1e9 / hbm_peak}


def kernel_rooflines(w, prof, rows_per_round: int, residual_per_round: float, hbm_peak: float,
                     rnn: bool):
    """Per-kernel algorithmic bytes per launch / event-timed launch / measured HBM
    peak, for the verify kernels and (RNN head) the state update."""
    out = {}

    def entry(kind, nbytes, extra):
        ms, n = prof.get(kind, (0.0, 0))
        if n <= 0 or ms <= 0:
            return
        t = ms / n / 1e3
        out[kind] = dict(extra, bytes_per_launch=int(nbytes), us_per_launch=t * 1e6,
                         achieved_gbs=nbytes / t / 1e9, frac=nbytes / t / 1e9 / hbm_peak, bound="hbm")

    entry("verify_rows", verify_rows_bytes(w, rows_per_round), {"rows": rows_per_round})
    entry("verify_draw", verify_draw_bytes(w, residual_per_round),
          {"residual_rows": residual_per_round, "bonus_rows": w.R - residual_per_round})
    ms, n = prof.get("verify_emit", (0.0, 0))
    if n > 0:  # one CTA per request: latency-bound, reported as time only
        out["verify_emit"] = {"us_per_launch": ms / n * 1e3, "bound": "latency"}
    if rnn:
        # h_{k-1} read, h_k written (fp32), the A rows written (bf16), Wh, Q_k
        e = 2
        nbytes = w.R * w.r * (4 + 4 + e + 4) + w.r * w.r * e
        entry("rnn_state", nbytes, {"note": "latency/instruction-bound: 2 R r^2 FLOP per step"})
    return out


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample_round(w, inp_cpu, req, seed, nthreads, scheduler="alg1", head="markov"):
    """Time one oracle round on the requests `req` (draft + full schedule + verify)."""
    import oracle

    f64 = lambda t: t.to(torch.float64).numpy()
    W1, W2 = inp_cpu["W1_64"], inp_cpu["W2_64"]
    x0 = inp_cpu["x0"].numpy()[req]
    t0 = time.perf_counter()
    if head == "rnn":
        rin = workload.rnn_inputs(w, seed=seed, device="cpu")
        od = oracle.draft_rnn(f64(inp_cpu["U"][req]), W1, W2, f64(rin["Wh"]), f64(rin["Q"][req]), x0, w.T,
                              seed, req_ids=req, nthreads=nthreads)
    else:
        od = oracle.draft(f64(inp_cpu["U"][req]), W1, W2, x0, w.T, seed, req_ids=req, nthreads=nthreads)
    t_draft = time.perf_counter() - t0
    t0 = time.perf_counter()
    conf = inp_cpu["conf"].numpy()
    if scheduler == "zos":
        ell = oracle.schedule_topk(conf, oracle.schedule_capacity(conf, inp_cpu["sps"].numpy())["K"])
    else:
        ell = oracle.schedule(conf, inp_cpu["sps"].numpy())["ell"]
    t_sched = time.perf_counter() - t0
    # Target stand-in for the sampled requests, from the oracle's own draft (untimed).
    # Verify reads rows j <= l_r + 1 only, so only those get the Markov bias (the
    # others are never read); the bias rows are kept compact, one request at a time.
    ls = np.asarray(ell)[req]
    if w.z_bias:
        prev = np.concatenate([x0[:, None], od["x"]], axis=1)  # [n, gamma + 1]
        first = np.concatenate([[0], np.cumsum(ls + 1)])
        rows = np.concatenate([prev[i, : ls[i] + 1] for i in range(len(req))])
        compact = oracle.markov_bias(W1, W2, rows)

        def bias_rows(i):
            b = torch.zeros(w.gamma + 1, w.V, dtype=torch.float64)
            b[: ls[i] + 1] = torch.from_numpy(compact[first[i]:first[i + 1]])
            return b

        Z = workload.target_logits(w, inp_cpu["U"][req], seed, bias_rows=bias_rows, requests=req)
    else:
        Z = workload.target_logits(w, inp_cpu["U"][req], seed, requests=req)
    t0 = time.perf_counter()
    ov = oracle.verify(od["x"], od["logp"], od["lse"], od["scores"], f64(Z), ls, w.T, seed,
                       req_ids=req, nthreads=nthreads)
    t_rest = time.perf_counter() - t0 + t_sched
    return t_draft + t_rest, int(ov["n_emit"].sum())


def oracle_inputs(w, seed, device):
    inp = workload.generate(w, seed=seed, device=device)
    cpu = {k: v.cpu() for k, v in inp.items()}
    cpu["W1_64"] = cpu["W1"].to(torch.float64).numpy()
    cpu["W2_64"] = cpu["W2"].to(torch.float64).numpy()
    return cpu


def sample_size(w, inp, seed, nthreads, target_s=28.0, scheduler="alg1", head="markov"):
    """Requests per oracle sample: about target_s seconds of wall time on nthreads
    (the timed round plus building its target stand-in), scaled from a probe of
    one request per thread (the host's speed is not assumed)."""
    n0 = max(1, min(w.R, nthreads))
    t0 = time.perf_counter()
    oracle_sample_round(w, inp, list(range(n0)), seed, nthreads, scheduler, head)
    wall = time.perf_counter() - t0
    return int(max(1, min(w.R, round(target_s * n0 / max(wall, 1e-6)))))


def cpu_baseline(w, seed, device, nthreads):
    import oracle

    oracle.build()
    inp = oracle_inputs(w, seed, device)
    n = sample_size(w, inp, seed, nthreads)
    req = list(range(n))
    t, _ = oracle_sample_round(w, inp, req, seed, nthreads)
    return {"value": n * w.gamma / t, "unit": "positions/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} of {w.R} requests (all {w.gamma} positions, full V) + the full schedule; "
                      f"{t:.1f} s"}


# ----------------------------------------------------------------------------- arms
def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    nthreads = os.cpu_count() or 1
    device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    inp = oracle_inputs(w, args.seed, device)
    n = sample_size(w, inp, args.seed, nthreads, target_s=100.0 / max(1, args.steps + args.warmup),
                    scheduler=args.scheduler, head=args.head)
    req = list(range(n))
    for _ in range(args.warmup):
        oracle_sample_round(w, inp, req, args.seed, nthreads, args.scheduler, args.head)
    times = []
    emitted = 0
    for _ in range(args.steps):
        t, e = oracle_sample_round(w, inp, req, args.seed, nthreads, args.scheduler, args.head)
        times.append(t)
        emitted += e
    tot = sum(times)
    value = n * w.gamma * args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "positions/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload.describe(w), seed=args.seed, scheduler=args.scheduler,
                           head=args.head, sample_requests=n),
            "cpu_baseline": {"value": value, "unit": "positions/s", "cores": nthreads,
                             "kind": "oracle",
                             "sample": f"{n} of {w.R} requests per step (all positions, full V) "
                                       f"+ the full schedule"},
            "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "accepted_tokens_per_s": emitted / tot}
    print(json.dumps(line), flush=True)


def run_seeds(args, w, rank, world, local):
    """Rounds with seeds 0..N-1, each on its own inputs (U, x0, c and the target
    stand-in regenerated untimed on the device; the draft head's weights from
    seed 0), one round timed per seed with CUDA events.  Reports summed
    positions over summed round time, and accepted tokens/s (emitted tokens,
    the bonus or correction token included, over the same time)."""
    import speculative_decoding_draft_05_gb300 as dspark

    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the library has no CPU path")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    dspark.binding.load()
    stream = torch.cuda.current_stream(device)
    rnd = Round(w, 0, device, scheduler=args.scheduler, verify_layout="padded", head=args.head,
                w2_layout=args.w2_layout)
    for i in range(args.warmup):
        rnd.step(0)
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_seed = []
    emitted = 0
    with ClockSampler(local) as clocks:
        for sd in range(args.seeds):
            if sd > 0:
                rnd.reseed(sd)
            barrier(world)
            torch.cuda.synchronize(device)
            ev0.record(stream)
            rnd.step(sd)
            ev1.record(stream)
            torch.cuda.synchronize(device)
            per_seed.append(ev0.elapsed_time(ev1))
            emitted += int(rnd.n_emit.sum().item())
            for ws in (rnd.ws_d, rnd.ws_s, rnd.ws_v):
                assert dspark.dspark_read_device_status(ws) == 0, f"device status at seed {sd}"
    ms = max_over_ranks(sum(per_seed), world, device)
    positions = w.R * w.gamma * len(per_seed) * world
    value = positions / (ms / 1e3)
    accepted = sum_over_ranks(float(emitted), world, device) / (ms / 1e3)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
                "steps": len(per_seed), "warmup": args.warmup, "ms_per_step": ms / len(per_seed),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
                "mode": f"seeds 0..{len(per_seed) - 1}, one round each on its own inputs",
                "config": dict(workload.describe(w), seeds=len(per_seed), scheduler=args.scheduler,
                               head=args.head, weights_seed=0,
                               w2_layout="transposed at setup" if rnd.w2t is not None else "plain",
                               l2="inputs larger than L2 (regenerated between rounds)"),
                "accepted_tokens_per_s": accepted, "emitted_tokens": emitted,
                "ms_per_round": {"min": min(per_seed), "median": statistics.median(per_seed),
                                 "max": max(per_seed)},
                "clocks": clocks.summary()}
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_ours(args, w, rank, world, local):
    import speculative_decoding_draft_05_gb300 as dspark

    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the library has no CPU path")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    dspark.binding.load()
    stream = torch.cuda.current_stream(device)
    rnd = Round(w, args.seed, device, scheduler=args.scheduler, verify_layout=args.verify_layout,
                head=args.head, w2_layout=args.w2_layout)
    seeds = [args.seed + i for i in range(args.steps)]  # one Philox key per round
    for i in range(args.warmup):
        rnd.step(args.seed + i)
    torch.cuda.synchronize(device)
    assert dspark.dspark_read_device_status(rnd.ws_d) == 0

    # ---- device-timed regions: the K steps as they run (the value), then the
    # same K steps with the library's per-launch events on (the kernel times
    # and the roofline), so that event records do not weigh on the value.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(device)
        ev0.record(stream)
        for sd in seeds:
            rnd.step(sd)
        ev1.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        dspark.dspark_profile_start()
        ev2.record(stream)
        for sd in seeds:
            rnd.step(sd)
        ev3.record(stream)
        torch.cuda.synchronize(device)
        prof = dspark.dspark_profile_stop()
        barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world, device)
    ms_prof = max_over_ranks(ev2.elapsed_time(ev3), world, device)
    positions = w.R * w.gamma * args.steps * world
    value = positions / (ms_max / 1e3)
    # tokens emitted by those rounds (deterministic: replay the same seeds, untimed)
    emitted = 0
    residual_rows = 0
    for sd in seeds:
        rnd.step(sd)
        emitted += int(rnd.n_emit.sum().item())
        residual_rows += int((rnd.n_acc < rnd.ell).sum().item())
    accepted = sum_over_ranks(float(emitted), world, device) / (ms_max / 1e3)

    # ---- e2e through the C-ABI with pinned host buffers: every step copies its
    # inputs host->device and reads its result back; step i+1's copies (two
    # copy streams, chunked) overlap step i's compute on double-buffered inputs.
    host_in = [t.cpu().pin_memory() for t in rnd.input_tensors()]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in rnd.result_tensors()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e2e_steps = max(3, min(args.steps, 10))
    sets = [rnd.input_tensors(), [t.clone() for t in rnd.input_tensors()]]
    copy_streams = [torch.cuda.Stream(device), torch.cuda.Stream(device)]
    chunk = 256 << 20

    def issue_copies(dst_set):
        n = 0
        for dst, src in zip(dst_set, host_in):
            flat_d, flat_s = dst.view(-1), src.view(-1)
            step_el = max(1, chunk // dst.element_size())
            for o in range(0, flat_d.numel(), step_el):
                with torch.cuda.stream(copy_streams[n % 2]):
                    flat_d[o:o + step_el].copy_(flat_s[o:o + step_el], non_blocking=True)
                n += 1
        evs = []
        for cs in copy_streams:
            ev = torch.cuda.Event()
            ev.record(cs)
            evs.append(ev)
        return evs

    barrier(world)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cs in copy_streams:
        cs.wait_event(e0)
    copied = issue_copies(sets[0])
    done = [None, None]
    for i, sd in enumerate(seeds[:e2e_steps]):
        for ev in copied:
            stream.wait_event(ev)
        nxt = None
        if i + 1 < e2e_steps:
            if done[(i + 1) % 2] is not None:  # that set's previous round must be finished
                for cs in copy_streams:
                    cs.wait_event(done[(i + 1) % 2])
            nxt = issue_copies(sets[(i + 1) % 2])
        rnd.step(sd, inputs=sets[i % 2])
        for dst, src in zip(host_out, rnd.result_tensors()):
            dst.copy_(src, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream)
        done[i % 2] = ev
        copied = nxt
    e1.record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    del sets
    e2e_ms = max(e0.elapsed_time(e1), 1e3 * wall)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = w.R * w.gamma * e2e_steps * world / (e2e_ms / 1e3)

    # ---- roofline of the dominant kernel (draft contraction + fused epilogue)
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    tile_ms, tile_n = prof["draft_tile"]
    avg_tile_s = tile_ms / max(1, tile_n) / 1e3
    achieved = draft_tile_bytes(w) / avg_tile_s / 1e9
    roofline = {"bound": "hbm", "kernel": "draft_tile", "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_src,
                "traffic": recorded_traffic(w.name),
                "algorithmic_bytes_per_launch": draft_tile_bytes(w),
                "avg_launch_ms": avg_tile_s * 1e3,
                "tensor": {"achieved_tflops": draft_tile_flops(w) / avg_tile_s / 1e12,
                           "peak_tflops": bf16_peak,
                           "frac": draft_tile_flops(w) / avg_tile_s / 1e12 / bf16_peak}}
    # Ceiling for the draft step's traffic mix: a contiguous stream of one step's
    # elements, bf16 in and fp32 out (U -> the scores buffer), timed the same way.
    if w.dtype == "bf16":
        n_el = w.R * w.V
        src, dst = rnd.inp["U"].view(-1)[:n_el], rnd.scores.view(-1)[:n_el]
        for _ in range(3):
            dspark.dspark_stream_probe(src, dst)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        for _ in range(20):
            dspark.dspark_stream_probe(src, dst)
        p1.record()
        torch.cuda.synchronize(device)
        t_probe = p0.elapsed_time(p1) / 20 / 1e3
        roofline["stream_probe"] = {"elements": n_el, "us": t_probe * 1e6,
                                    "gbs": 6 * n_el / t_probe / 1e9,
                                    "draft_step_us": avg_tile_s * 1e6,
                                    "probe_over_draft": t_probe / avg_tile_s}
    # The draft step in its own launch configuration: consecutive steps are
    # programmatic dependents and overlap, which per-launch events prevent.  The
    # draft call is timed alone at gamma and at 2 positions (same R, V, weights);
    # the difference over gamma - 2 is the period of one step inside the call.
    if w.dtype == "bf16" and args.head == "markov" and w.gamma > 2:
        roofline["pipelined"] = draft_step_period(rnd, w, device, args.seed, hbm_peak)
    k_roof = kernel_rooflines(w, prof, int(rnd.ell.sum().item()), residual_rows / len(seeds), hbm_peak,
                              args.head == "rnn")
    # Full-block verify over this round's own buffers, outside the timed regions:
    # the first (up to) 64 requests with l = gamma, so that the row kernel streams
    # every position even where the workload's schedule keeps nothing.
    vprobe = None
    if not rnd.packed:
        n = min(64, w.R)
        ell_full = torch.full((n,), w.gamma, dtype=torch.int32, device=device)
        vo = dict(n_acc=torch.empty_like(rnd.n_acc[:n]), tokens=torch.empty_like(rnd.tokens[:n]),
                  n_emit=torch.empty_like(rnd.n_emit[:n]), cstar=torch.empty_like(rnd.cstar[:n]),
                  lse_t=torch.empty_like(rnd.lse_t[:n]), workspace=rnd.ws_v)
        args_v = (rnd.x[:n], rnd.logp[:n], rnd.lse[:n], rnd.scores[:n], rnd.Z[:n], ell_full, w.T, args.seed)
        for _ in range(2):
            dspark.dspark_verify(*args_v, **vo)
        torch.cuda.synchronize(device)
        dspark.dspark_profile_start()
        for _ in range(5):
            dspark.dspark_verify(*args_v, **vo)
        vp = dspark.dspark_profile_stop()
        ms_r, n_r = vp["verify_rows"]
        t_r = ms_r / max(1, n_r) / 1e3
        nb = verify_rows_bytes(w, n * w.gamma)
        vprobe = {"requests": n, "rows": n * w.gamma, "bytes_per_launch": nb, "us_per_launch": t_r * 1e6,
                  "achieved_gbs": nb / t_r / 1e9, "frac": nb / t_r / 1e9 / hbm_peak, "peak": hbm_peak,
                  "note": "extra call outside the timed regions; not part of value"}
    rb = round_bytes(w, rnd.ell, transpose=rnd.w2t is None and w.dtype == "bf16")
    round_roof = {"bound": "hbm", "algorithmic_bytes": rb,
                  "achieved": rb / (ms_max / args.steps / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                  "frac": rb / (ms_max / args.steps / 1e3) / 1e9 / hbm_peak}
    kernels = {k: {"ms_per_launch": v[0] / max(1, v[1]), "launches": v[1],
                   "share": v[0] / max(1e-9, sum(x[0] for kk, x in prof.items() if not kk.startswith("_")))}
               for k, v in prof.items() if not k.startswith("_") and v[1] > 0}
    launches = sum(v[1] for k, v in prof.items() if not k.startswith("_"))

    out = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out = cpu_baseline(w, args.seed, device, os.cpu_count() or 1)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
                "ms_per_step_with_kernel_events": ms_prof / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
                if w.dtype == "bf16" else "f32", "data": "synthetic",
                "config": dict(workload.describe(w), seed=args.seed, scheduler=args.scheduler,
                               verify_layout=args.verify_layout, head=args.head,
                               w2_layout="transposed at setup" if rnd.w2t is not None else "plain",
                               parallelism="replicas" if world > 1 else "single",
                               l2="inputs larger than L2 (U %.2f GB, scores %.2f GB, Z %.2f GB > 129 MB)" % (
                                   w.R * w.gamma * w.V * (2 if w.dtype == "bf16" else 4) / 1e9,
                                   w.R * w.gamma * w.V * 4 / 1e9,
                                   rnd.input_tensors()[6].numel() * rnd.input_tensors()[6].element_size() / 1e9)),
                "roofline": roofline, "round_roofline": round_roof, "kernels_roofline": k_roof,
                "verify_rows_probe": vprobe, "cpu_baseline": out,
                "e2e": {"value": e2e_value, "unit": "positions/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": e2e_steps},
                "gpu_launches": launches, "clocks": clocks.summary(),
                "accepted_tokens_per_s": accepted, "mean_ell": float(rnd.ell.float().mean().item()),
                "mean_emitted": float(rnd.n_emit.float().mean().item()), "kernels": kernels}
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workload.ORDER)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scheduler", choices=["alg1", "zos"], default="alg1",
                    help="alg1: Algorithm 1 (default); zos: zero-overhead capacity + top-K")
    ap.add_argument("--head", choices=["markov", "rnn"], default="markov",
                    help="draft head: markov (default) or the RNN head")
    ap.add_argument("--verify-layout", choices=["padded", "packed"], default="padded",
                    help="target logits padded [R, gamma+1, V] (default) or packed rows + offsets")
    ap.add_argument("--w2-layout", choices=["transposed", "plain"], default="transposed",
                    help="the head's W2: transposed once at setup into the tensor cores' layout "
                         "(default; weights stay fixed across rounds) or passed as stored, "
                         "each draft call transposing it")
    ap.add_argument("--R", type=int, default=None, help="override the workload's request count")
    ap.add_argument("--gamma", type=int, default=None, help="override the workload's draft length")
    ap.add_argument("--seeds", type=int, default=0,
                    help="N > 0: N rounds with seeds 0..N-1, each on its own regenerated inputs "
                         "(the serving workload's 100-seed report)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_info()
    w = workload.WORKLOADS[args.workload]
    over = {k: v for k, v in (("R", args.R), ("gamma", args.gamma)) if v is not None}
    if over:
        w = w.resized(**over)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if args.seeds > 0:
        run_seeds(args, w, rank, world, local)
        return
    run_ours(args, w, rank, world, local)


if __name__ == "__main__":
    main()
