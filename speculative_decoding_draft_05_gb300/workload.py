"""Seeded synthetic inputs for the DSpark per-round sampling path.

This module only draws random tensors with the shapes, dtypes and value
distributions of the five workloads below.  It holds none of the method's
arithmetic: the Markov bias that the target logits of the bf16 workloads carry
is computed by the caller (the oracle in the tests, the library's own draft
outputs in the benchmark) and passed in to :func:`target_logits`.

Workloads (R requests, gamma draft positions, vocabulary V, Markov rank r):

==============================  ====  =====  =======  ===  =====  ====
name                            R     gamma  V        r    dtype  T
==============================  ====  =====  =======  ===  =====  ====
tiny_r4_g4_v1024                4     4      1024     16   f32    1.0
qwen3_r64_g16_v151936           64    16     151936   256  bf16   1.0
verify_r512_g16_v151936         512   16     151936   256  bf16   1.0
largevocab_r256_g8_v262144      256   8      262144   256  bf16   0.7
serving_r1024_g16_v129280       1024  16     129280   256  bf16   1.0
==============================  ====  =====  =======  ===  =====  ====

Distributions (per workload):
* U (backbone logits, [R, gamma, V]): N(0, 2^2) tiny; N(0, 3^2) + Zipf(1.1)
  offset for qwen3/verify/serving; N(0, 4^2) for largevocab.  The Zipf offset
  is the log of a Zipf(1.1) pmf over rank v+1, -1.1 ln(v+1), shared by all rows.
* W1 [V, r], W2 [r, V]: N(0, 0.1^2) tiny, N(0, 0.02^2) otherwise.
* x0 [R]: uniform in [0, V).
* Target logits Z [R, gamma+1, V] = padded U + noise (+ Markov bias B along the
  draft's own tokens for the bf16 workloads).  Row gamma+1 pads U with a fresh
  row of U's distribution.  Noise at position k ~ N(0, sigma_k^2) with
  sigma_k = 0.3k (tiny), 0.15k (qwen3, verify), 0.2k (largevocab),
  0.1 + 0.12k (serving).
* Confidence c [R, gamma] (float32): 0.9*0.85^(k-1) (tiny); 0.8 (qwen3);
  sigmoid(N(2 - 0.25k, 0.5^2)) (verify); 0.95*0.8^(k-1)*U(0.8, 1)
  (largevocab); sigmoid(N(2.5 - 0.3k, 0.7^2)) (serving).
* Step-rate table SPS[B] (float64, B = 0..R(1+gamma)): 1/(1e-3 + 2e-5 B)
  (tiny); flat 1/4e-3 (qwen3, so the scheduler keeps full blocks);
  1/(4e-3 + 1.5e-5 max(0, B-256)) (verify, largevocab);
  1/(6e-3 + 1e-5 B + 4e-9 B^2) (serving).

Every tensor is drawn from a torch.Generator on ``device`` seeded from
(seed, tensor name[, request]); per-request tensors are drawn one request at a
time so that any subset of requests can be regenerated identically on the same
device type.  CPU and CUDA generators give different streams: a test that needs
the same inputs on both sides generates them once and copies them.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Callable, Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    r: int
    dtype: str  # "f32" or "bf16": dtype of U, W1, W2 and Z
    T: float
    u_std: float
    zipf: bool
    w_std: float
    noise: Callable[[int], float]  # sigma_k for position k (1-based)
    z_bias: bool  # target logits carry the Markov bias along the draft tokens
    conf: str  # confidence law, see module docstring
    sps: str  # step-rate law, see module docstring

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def positions(self) -> int:
        return self.R * self.gamma

    def resized(self, **kw) -> "Workload":
        """Same distributions, other sizes (parity cases spanning tiles and ragged tails)."""
        name = kw.pop("name", None) or (self.name + "_" + "_".join(f"{k}{v}" for k, v in kw.items()))
        return dataclasses.replace(self, name=name, **kw)


def _sigma_lin(a: float, b: float) -> Callable[[int], float]:
    return lambda k: a + b * k


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_r4_g4_v1024", 4, 4, 1024, 16, "f32", 1.0, 2.0, False, 0.1,
                 _sigma_lin(0.0, 0.3), False, "geom_0.9_0.85", "lin_1e-3_2e-5"),
        Workload("qwen3_r64_g16_v151936", 64, 16, 151936, 256, "bf16", 1.0, 3.0, True, 0.02,
                 _sigma_lin(0.0, 0.15), True, "const_0.8", "flat_4e-3"),
        Workload("verify_r512_g16_v151936", 512, 16, 151936, 256, "bf16", 1.0, 3.0, True, 0.02,
                 _sigma_lin(0.0, 0.15), True, "sigmoid_2_0.25_0.5", "knee_4e-3_1.5e-5_256"),
        Workload("largevocab_r256_g8_v262144", 256, 8, 262144, 256, "bf16", 0.7, 4.0, False, 0.02,
                 _sigma_lin(0.0, 0.2), True, "geomU_0.95_0.8", "knee_4e-3_1.5e-5_256"),
        Workload("serving_r1024_g16_v129280", 1024, 16, 129280, 256, "bf16", 1.0, 3.0, True, 0.02,
                 _sigma_lin(0.1, 0.12), True, "sigmoid_2.5_0.3_0.7", "quad_6e-3_1e-5_4e-9"),
    ]
}

# Short aliases in the order the workloads are listed above.
ORDER = list(WORKLOADS)


def _gen(device, seed: int, tag: str, request: Optional[int] = None) -> torch.Generator:
    key = zlib.crc32(tag.encode()) & 0xFFFFFFFF
    s = (int(seed) * 0x9E3779B1 + key * 0x85EBCA77 + (0 if request is None else (request + 1) * 0xC2B2AE3D))
    g = torch.Generator(device=device)
    g.manual_seed(s & 0x7FFFFFFFFFFFFFFF)
    return g


def zipf_offset(V: int, device) -> torch.Tensor:
    """log of a Zipf(1.1) pmf over rank v+1, without its normalising constant."""
    return -1.1 * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))


def _draw_logit_rows(w: Workload, n_rows: int, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(n_rows, w.V, generator=gen, device=device, dtype=torch.float32) * w.u_std
    if w.zipf:
        x += zipf_offset(w.V, device)
    return x


def confidence(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    k = torch.arange(1, w.gamma + 1, dtype=torch.float64, device=device)
    g = _gen(device, seed, "conf")
    if w.conf == "geom_0.9_0.85":
        c = (0.9 * 0.85 ** (k - 1)).expand(w.R, w.gamma)
    elif w.conf == "const_0.8":
        c = torch.full((w.R, w.gamma), 0.8, dtype=torch.float64, device=device)
    elif w.conf.startswith("sigmoid_"):
        _, mu0, slope, sd = w.conf.split("_")
        z = torch.randn(w.R, w.gamma, generator=g, device=device, dtype=torch.float64)
        c = torch.sigmoid(float(mu0) - float(slope) * k + float(sd) * z)
    elif w.conf == "geomU_0.95_0.8":
        u = torch.rand(w.R, w.gamma, generator=g, device=device, dtype=torch.float64)
        c = 0.95 * 0.8 ** (k - 1) * (0.8 + 0.2 * u)
    else:
        raise ValueError(w.conf)
    eps = 2.0 ** -24
    return c.clamp(eps, 1.0 - eps).to(torch.float32).contiguous()


def step_rate_table(w: Workload, device="cpu") -> torch.Tensor:
    """SPS[B] in steps/s for B = 0..R(1+gamma), float64."""
    B = torch.arange(0, w.R * (1 + w.gamma) + 1, dtype=torch.float64, device=device)
    if w.sps == "lin_1e-3_2e-5":
        t = 1e-3 + 2e-5 * B
    elif w.sps == "flat_4e-3":
        t = torch.full_like(B, 4e-3)
    elif w.sps == "knee_4e-3_1.5e-5_256":
        t = 4e-3 + 1.5e-5 * torch.clamp(B - 256, min=0)
    elif w.sps == "quad_6e-3_1e-5_4e-9":
        t = 6e-3 + 1e-5 * B + 4e-9 * B * B
    else:
        raise ValueError(w.sps)
    return (1.0 / t).contiguous()


def rnn_inputs(w: Workload, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """Inputs of the RNN draft head: Wh [r, r] ~ N(0, (0.5 / sqrt(r))^2) in the
    workload dtype (a contractive recurrence), and the backbone hidden state
    projected into the head's space, Q [R, gamma, r] ~ N(0, 0.5^2) (float32)."""
    g = _gen(device, seed, "rnn")
    Wh = (torch.randn(w.r, w.r, generator=g, device=device) * (0.5 / w.r ** 0.5)).to(w.torch_dtype)
    Q = torch.randn(w.R, w.gamma, w.r, generator=g, device=device) * 0.5
    return dict(Wh=Wh.contiguous(), Q=Q.contiguous())


def generate(w: Workload, seed: int = 0, device="cpu",
             weights_seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """U, W1, W2, x0, conf, sps for workload ``w`` (dtype ``w.torch_dtype`` for U/W1/W2).

    The draft head's weights W1, W2 come from ``weights_seed`` when it is given
    (a serving run keeps one head while every round draws new U, x0 and c),
    else from ``seed``."""
    dt = w.torch_dtype
    U = torch.empty(w.R, w.gamma, w.V, dtype=dt, device=device)
    for r in range(w.R):
        U[r] = _draw_logit_rows(w, w.gamma, _gen(device, seed, "U", r), device).to(dt)
    gw = _gen(device, seed if weights_seed is None else weights_seed, "W")
    W1 = (torch.randn(w.V, w.r, generator=gw, device=device) * w.w_std).to(dt).contiguous()
    W2 = (torch.randn(w.r, w.V, generator=gw, device=device) * w.w_std).to(dt).contiguous()
    x0 = torch.randint(0, w.V, (w.R,), generator=_gen(device, seed, "x0"), device=device,
                       dtype=torch.int64).to(torch.int32)
    return dict(U=U, W1=W1, W2=W2, x0=x0, conf=confidence(w, seed, device),
                sps=step_rate_table(w, device))


def target_base_rows(w: Workload, U_r: torch.Tensor, seed: int, request: int) -> torch.Tensor:
    """fp32 [gamma+1, V]: U of one request padded with a fresh row, plus position noise."""
    device = U_r.device
    g = _gen(device, seed, "Z", request)
    base = torch.empty(w.gamma + 1, w.V, dtype=torch.float32, device=device)
    base[: w.gamma] = U_r.to(torch.float32)
    base[w.gamma] = _draw_logit_rows(w, 1, g, device)[0].to(w.torch_dtype).to(torch.float32)
    sig = torch.tensor([w.noise(k) for k in range(1, w.gamma + 2)], dtype=torch.float32,
                       device=device)
    base += torch.randn(w.gamma + 1, w.V, generator=g, device=device) * sig[:, None]
    return base


def target_logits(w: Workload, U: torch.Tensor, seed: int,
                  bias_rows: Optional[Callable[[int], torch.Tensor]] = None,
                  requests=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Z [n, gamma+1, V] in w's dtype for the listed requests (default: all).

    ``U`` holds the rows of those requests in the same order.  For the bf16
    workloads ``bias_rows(i)`` must return the fp32 Markov bias [gamma+1, V]
    of the i-th listed request along (x0, x_1, ..., x_gamma); the sum is rounded
    once to the workload dtype.
    """
    reqs = list(range(U.shape[0])) if requests is None else list(requests)
    if out is None:
        out = torch.empty(len(reqs), w.gamma + 1, w.V, dtype=w.torch_dtype, device=U.device)
    for i, r in enumerate(reqs):
        base = target_base_rows(w, U[i], seed, r)
        if w.z_bias:
            if bias_rows is None:
                raise ValueError(f"{w.name}: target logits need the Markov bias along the draft")
            base += bias_rows(i).to(base.device, torch.float32)
        out[i] = base.to(w.torch_dtype)
    return out


def describe(w: Workload) -> dict:
    return dict(workload=w.name, R=w.R, gamma=w.gamma, V=w.V, r=w.r, dtype=w.dtype,
                temperature=w.T)


def bytes_per_round(w: Workload, verify_rows: int) -> int:
    """Algorithmic bytes of one round (draft U read + scores write + W2 per step + verify rows)."""
    e = 4 if w.dtype == "f32" else 2
    draft = w.R * w.gamma * w.V * (e + 4) + w.gamma * w.r * w.V * e
    return draft + verify_rows * w.V * e


def flops_per_round(w: Workload) -> int:
    return 2 * w.R * w.r * w.V * w.gamma


def isclose_sps(a: float, b: float) -> bool:
    return math.isclose(a, b, rel_tol=1e-12)
