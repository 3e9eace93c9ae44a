"""Residual draws where the target and the draft nearly agree.

Standard rejection sampling ("DSpark ... 요약 설명", opening bullets: the target
verifies the drafted block so that its own distribution is preserved) draws the
token after the first rejection from norm(max(0, p^t - p^d)).  A good drafter
makes p^t and p^d agree closely, so that residual is a small difference of two
nearly equal numbers.  These tests build exactly that regime at the Qwen3
vocabulary (V = 151,936) and check the GPU's residual draw against the oracle
on every request:

* verify inputs: synthetic fp32 draft log-scores s (N(0, 3^2) plus the Zipf(1.1)
  offset), their fp64 log-normaliser lse, and per row a drafted token x_j whose
  draft probability lies in [1e-5, 1e-4];
* target rows Z_j = T s_j + N(0, sigma^2) in fp32 (sigma = 1e-3 or 1e-4), with
  Z_j[x_j] lowered by 6 T so that x_j is rejected (acceptance e^-6 ~ 0.25%);
* the first rejection then draws from a residual whose relative size
  (p^t - p^d) / p^d is of order sigma for about half the vocabulary.

Parity rule.  Tokens are bit-exact except where the oracle's fp64 margin
between the two choices (two groups of 32 ids at stage 1 of the two-level
draw, or two ids of one group at stage 2) is within the fp32 evaluation error
the GPU's keys can carry there.  The GPU forms delta = ln p^t - ln p^d = (z/T - s) - (LSE^t - lse)
and the log-residual ln p^t + ln(1 - e^-delta); an error e_L in its fp32 LSE^t
moves delta by e_L and the key by about e_L / delta, which at delta ~ 1e-4 is far
above the 1e-5 near-tie.  The test first bounds e_L (|LSE^t_gpu - LSE^t_oracle|
<= EPS_L on every row), then allows a token difference only within the key
error that this bound and fp32 rounding imply, and only on a few requests.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import speculative_decoding_draft_05_gb300 as dspark

from parity import TIE

pytestmark = pytest.mark.gpu

V = 151936
EPS_L = 4e-6  # |LSE^t_gpu - LSE^t_oracle| bound asserted on every scheduled row
U24 = 2.0 ** -23


def build_inputs(R, gamma, T, sigma, seed):
    rng = np.random.default_rng(seed)
    zipf = -1.1 * np.log(np.arange(V) + 1.0)
    s = (rng.normal(0.0, 3.0, size=(R, gamma, V)) + zipf).astype(np.float32)
    lse = logsumexp(s.astype(np.float64), axis=-1).astype(np.float32)
    pd = np.exp(s.astype(np.float64) - lse.astype(np.float64)[..., None])
    x = np.empty((R, gamma), np.int32)
    for i in range(R):
        for j in range(gamma):
            pool = np.flatnonzero((pd[i, j] >= 1e-5) & (pd[i, j] <= 1e-4))
            x[i, j] = rng.choice(pool)
    logp = (np.take_along_axis(s, x[..., None], -1)[..., 0].astype(np.float64)
            - lse.astype(np.float64)).astype(np.float32)
    Z = np.empty((R, gamma + 1, V), np.float32)
    Z[:, :gamma] = (T * s.astype(np.float64) + rng.normal(0.0, sigma, size=s.shape)).astype(np.float32)
    Z[:, gamma] = (rng.normal(0.0, 3.0, size=(R, V)) + zipf).astype(np.float32)
    # Reject x_j at row 1 for even requests and at row 2 for odd ones (row 1 is
    # then accepted with probability ~1, p^t(x_1) ~ p^d(x_1)).
    for i in range(R):
        j = 0 if (i % 2 == 0 or gamma == 1) else 1
        Z[i, j, x[i, j]] = np.float32(T * (float(s[i, j, x[i, j]]) - 6.0))
    ell = np.full(R, gamma, np.int32)
    return s, lse, x, logp, Z, ell


def residuals(s, lse, Z, Lt_o, i, row, T):
    """fp64 residual p^t - p^d of the whole row (request i, row), as the oracle forms it."""
    pt = np.exp(Z[i, row - 1].astype(np.float64) / T - Lt_o)
    pd = np.exp(s[i, row - 1].astype(np.float64) - float(lse[i, row - 1]))
    return pt - pd


def oracle_key(res, i, row, v, seed):
    """The oracle's fp64 stage-2 key of token v (log residual + its Gumbel)."""
    if not res[v] > 0:
        return -np.inf
    return np.log(res[v]) + oracle.gumbel(oracle.rng_word(seed, i, row, oracle.PURPOSE_RESAMPLE, v))


def oracle_group_key(res, i, row, j, seed):
    """The oracle's fp64 stage-1 key of group j (log residual mass + its Gumbel)."""
    seg = res[32 * j: 32 * j + 32]
    pos = seg[seg > 0]
    if pos.size == 0:
        return -np.inf
    return np.log(pos.sum()) + oracle.gumbel(oracle.rng_word(seed, i, row, oracle.PURPOSE_RESAMPLE_GROUP, j))


def key_allowance(s, lse, Z, Lt_o, i, row, v, T, seed):
    """Bound on |GPU key - oracle key| of token v from EPS_L and fp32 rounding
    (the log-weight's error plus the Gumbel term's rounding)."""
    z, sv, ld = float(Z[i, row - 1, v]) / T, float(s[i, row - 1, v]), float(lse[i, row - 1])
    a = z - Lt_o
    delta = (z - sv) - (Lt_o - ld)
    e_delta = EPS_L + U24 * (abs(z - sv) + abs(Lt_o - ld) + abs(delta) + abs(z))
    if delta - e_delta <= 0:
        return np.inf  # the sign of this residual is not fixed by fp32
    l1 = np.log(-np.expm1(-delta))
    G = oracle.gumbel(oracle.rng_word(seed, i, row, oracle.PURPOSE_RESAMPLE, v))
    e = (EPS_L + U24 * (abs(a) + abs(z)) + e_delta / (delta - e_delta)
         + 2 * U24 * (2 + abs(l1) + abs(G)) + U24 * abs(a + l1 + G))
    return 2.0 * e


@pytest.mark.parametrize("sigma", [1e-3, 1e-4], ids=["sigma1e-3", "sigma1e-4"])
def test_residual_draw_near_cancellation(sigma):
    R, gamma, T, seed = 256, 2, 1.0, 31
    s, lse, x, logp, Z, ell = build_inputs(R, gamma, T, sigma, seed)
    ov = oracle.verify(x, logp.astype(np.float64), lse.astype(np.float64), s.astype(np.float64),
                       Z.astype(np.float64), ell, T, seed)
    # the construction: nearly every request rejects and draws from a residual
    assert (ov["n_acc"] < ell).mean() > 0.95
    assert (ov["stop_kind"][ov["n_acc"] < ell] == 1).all()

    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    gv = dspark.dspark_verify(t(x), t(logp), t(lse), t(s), t(Z), t(ell), T, seed)
    torch.cuda.synchronize()
    assert dspark.dspark_read_device_status(gv["workspace"]) == 0
    g = {k: v.cpu().numpy() for k, v in gv.items() if isinstance(v, torch.Tensor) and k != "workspace"}

    # LSE^t of every scheduled row within EPS_L of the oracle's
    err_L = np.abs(g["lse_t"][:, :gamma].astype(np.float64) - ov["lse_t"][:, :gamma])
    assert err_L.max() <= EPS_L, f"LSE^t error {err_L.max():.3g} > {EPS_L}"
    # accept decisions bit-exact (margins are ~6 nats here)
    assert (g["n_acc"] == ov["n_acc"]).all()
    assert (g["n_emit"] == g["n_acc"] + 1).all()

    exempt = []
    for i in range(R):
        if (g["tokens"][i] == ov["tokens"][i]).all():
            continue
        n = int(ov["n_acc"][i])
        assert (g["tokens"][i, :n] == ov["tokens"][i, :n]).all() and (g["tokens"][i, n + 1:] == -1).all()
        if n == ell[i]:  # a bonus draw from p^t: the ordinary near-tie rule
            assert ov["res_margin"][i] < TIE, (i, ov["res_margin"][i])
            exempt.append(i)
            continue
        row = n + 1
        vo, vg = int(ov["tokens"][i, n]), int(g["tokens"][i, n])
        Lt_o = float(ov["lse_t"][i, row - 1])
        res = residuals(s, lse, Z, Lt_o, i, row, T)
        jo, jg = vo // 32, vg // 32
        if jo != jg:
            # stage 1 chose another group: a group key's error is at most its
            # ids' largest key error (its log-mass is a weighted mean of theirs)
            def group_allow(j):
                return max(key_allowance(s, lse, Z, Lt_o, i, row, v, T, seed)
                           for v in range(32 * j, min(V, 32 * j + 32)) if res[v] > 0)
            ko = oracle_group_key(res, i, row, jo, seed)
            kg = oracle_group_key(res, i, row, jg, seed)
            allow = group_allow(jo) + group_allow(jg) + TIE
            what = f"group {jg} vs the oracle's group {jo}"
        else:
            ko = oracle_key(res, i, row, vo, seed)
            kg = oracle_key(res, i, row, vg, seed)
            allow = (key_allowance(s, lse, Z, Lt_o, i, row, vo, T, seed)
                     + key_allowance(s, lse, Z, Lt_o, i, row, vg, T, seed) + TIE)
            what = f"token {vg} vs the oracle's token {vo} in group {jo}"
        assert ko - kg <= allow, (
            f"request {i}: gpu {what}: oracle keys {kg:.6f} / {ko:.6f}, gap {ko - kg:.3g} "
            f"beyond the fp32 allowance {allow:.3g}")
        exempt.append(i)
    assert len(exempt) <= max(2, R // 32), exempt
    keep = np.array([i not in exempt for i in range(R)])
    # c* of the scheduled rows: both distributions nearly agree, so c* ~ 1 - p^d(x)
    cs_err = np.abs(g["cstar"][keep].astype(np.float64) - ov["cstar"][keep]).max()
    assert cs_err <= 1e-5, cs_err
