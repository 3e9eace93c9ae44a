"""Pins for the oracle's verification step (CPU only).

Standard rejection sampling (DSpark summary, opening bullets and §3; DSpark
notes "배경"; Leviathan et al. 2023, Chen et al. 2023) and the soft label of
DSpark summary §3.2.1.

Pins:
* closed form: c* = sum_v min(p^d, p^t) = 1 - 1/2 |p^d - p^t|_1, and the
  empirical acceptance frequency of a drafted token equals that value
  (binomial 5-sigma band);
* output law: the first emitted token follows p^t (chi-square, tiny V); with a
  prefix-dependent target (Z_j built from the drafted x_{j-1} per trial), the
  second emitted token given an accepted first token follows the target's
  transition row;
* Appendix A: a retroactive scheduler (test-only, global argmax of Theta with
  the c_2 the sampled x_1 implies) gives the output law (0.85, 0.15), the
  causal Algorithm 1 gives the target (0.7, 0.3) -- numbers from
  tests/golden/appendix_a.json;
* special cases: l = 0 emits one token from p^t; p^d = p^t accepts every
  scheduled token with c* = 1.
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix_a.json")


def _draft_fixed(n, logits_rows, seed, T=1.0):
    """Draft with fixed per-position logits (W = 0): s_k = logits_rows[k] / T."""
    g, V = logits_rows.shape
    U = np.repeat(logits_rows[None], n, axis=0)
    W1 = np.zeros((V, 1))
    W2 = np.zeros((1, V))
    return oracle.draft(U, W1, W2, np.zeros(n, np.int32), T, seed)


def test_soft_label_closed_forms():
    rng = np.random.default_rng(0)
    n, g, V = 3, 4, 64
    d = _draft_fixed(n, rng.normal(0, 2, size=(g, V)), seed=1)
    Z = rng.normal(0, 2, size=(n, g + 1, V))
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.full(n, g), 1.0, seed=1)
    pd = np.exp(d["scores"] - d["lse"][..., None])
    pt = special.softmax(Z[:, :g], axis=2)
    np.testing.assert_allclose(v["cstar"], np.minimum(pd, pt).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(v["cstar"], 1 - 0.5 * np.abs(pd - pt).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(v["lse_t"][:, :g], special.logsumexp(Z[:, :g], axis=2), atol=1e-12)


def test_acceptance_frequency_matches_closed_form():
    rng = np.random.default_rng(1)
    n, V = 100000, 8
    draft_logits = rng.normal(0, 1.0, size=(1, V))
    d = _draft_fixed(n, draft_logits, seed=3)
    Z = np.repeat(rng.normal(0, 1.0, size=(1, 2, V))[None], n, axis=0)[:, 0]
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.ones(n, np.int32), 1.0, seed=3)
    c = float(v["cstar"][0, 0])
    freq = v["n_acc"].mean()
    assert abs(freq - c) < 5 * np.sqrt(c * (1 - c) / n), (freq, c)
    np.testing.assert_allclose(v["cstar"][:, 0], c, atol=1e-14)


@pytest.mark.parametrize("V", [8, 80])
@pytest.mark.parametrize("ell", [0, 1, 3])
def test_first_emitted_token_follows_target(ell, V):
    rng = np.random.default_rng(10 + ell)
    n, g = 60000, 3
    d = _draft_fixed(n, rng.normal(0, 1.2, size=(g, V)), seed=5)
    Zrow = rng.normal(0, 1.2, size=(g + 1, V))
    Z = np.repeat(Zrow[None], n, axis=0)
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.full(n, ell), 1.0, seed=5)
    first = v["tokens"][:, 0]
    assert (first >= 0).all()
    pt = special.softmax(Zrow[0])
    assert stats.chisquare(np.bincount(first, minlength=V), pt * n).pvalue > 1e-4
    if ell == 0:
        assert (v["n_emit"] == 1).all() and (v["n_acc"] == 0).all()
        assert np.isnan(v["cstar"]).all()
    assert (v["n_emit"] == v["n_acc"] + 1).all()
    assert (v["n_acc"] <= ell).all()


def test_prefix_dependent_target_chain():
    # Target: a Markov chain with transition logits Tt[prev].  Draft: another
    # Markov chain (the Markov head with W1 W2 = Td).  Per trial the test builds
    # Z_j = Tt[x_{j-1}] from the drafted tokens (x_0 = anchor), as a target model
    # conditioned on the drafted prefix would.
    rng = np.random.default_rng(20)
    n, g, V = 80000, 3, 6
    Td = rng.normal(0, 1.0, size=(V, V))
    Tt = rng.normal(0, 1.0, size=(V, V))
    W1 = Td  # rank V factorisation W1 @ I = Td
    W2 = np.eye(V)
    x0 = np.full(n, 2, dtype=np.int32)
    d = oracle.draft(np.zeros((n, g, V)), W1, W2, x0, 1.0, seed=8)
    prev = np.concatenate([x0[:, None], d["x"]], axis=1)  # [n, g+1]
    Z = Tt[prev]
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.full(n, g), 1.0, seed=8)
    P = special.softmax(Tt, axis=1)
    y = v["tokens"]
    assert stats.chisquare(np.bincount(y[:, 0], minlength=V), P[2] * n).pvalue > 1e-4
    two = v["n_emit"] >= 2
    for a in range(V):
        sel = two & (y[:, 0] == a)
        if sel.sum() < 3000:
            continue
        cnt = np.bincount(y[sel, 1], minlength=V)
        assert stats.chisquare(cnt, P[a] * sel.sum()).pvalue > 1e-4, a


def test_appendix_a_retroactive_scheduler_biases_output():
    gold = json.load(open(GOLDEN))
    n = 100000
    pd, pt = np.array(gold["draft_first_position"]), np.array(gold["target_first_position"])
    sps = np.array([0.0] + gold["sps_1_2_3"])
    a1 = gold["a1"]
    # Draft: first position (0.5, 0.5); second position arbitrary.
    d = _draft_fixed(n, np.log(np.array([pd, [0.5, 0.5]])), seed=21)
    Z = np.repeat(np.log(np.array([pt, [0.5, 0.5], [0.5, 0.5]]))[None], n, axis=0)

    def retroactive_ell(x1):
        # c_2 depends on the sampled first token: 0.9 after token 0 ("A"), 0 after token 1 ("B").
        c2 = 0.9 if x1 == 0 else 0.0
        thetas = [1.0 * sps[1], (1 + a1) * sps[2], (1 + a1 + a1 * c2) * sps[3]]
        return int(np.argmax(thetas))

    ell_retro = np.array([retroactive_ell(x) for x in d["x"][:, 0]], dtype=np.int32)
    assert set(np.unique(ell_retro)) <= {0, 2}
    assert retroactive_ell(0) == gold["retroactive_ell_if_c2"]["0.9"]
    assert retroactive_ell(1) == gold["retroactive_ell_if_c2"]["0.0"]
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, ell_retro, 1.0, seed=21)
    law = np.bincount(v["tokens"][:, 0], minlength=2) / n
    assert abs(law[0] - gold["retroactive_output_law"][0]) < 5 * np.sqrt(0.85 * 0.15 / n)
    # Causal Algorithm 1 stops at Theta_1 < Theta_0 before looking at c_2: l = 0.
    ell_causal = np.array([oracle.schedule(np.array([[a1, 0.9 if x == 0 else 0.0]], np.float32), sps)
                           ["ell"][0] for x in d["x"][:200, 0]])
    assert (ell_causal == 0).all()
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.zeros(n, np.int32), 1.0, seed=21)
    counts = np.bincount(v["tokens"][:, 0], minlength=2)
    assert stats.chisquare(counts, np.array(gold["causal_output_law"]) * n).pvalue > 1e-4
    assert stats.chisquare(counts, np.array(gold["retroactive_output_law"]) * n).pvalue < 1e-6


def test_identical_draft_and_target_accepts_everything():
    rng = np.random.default_rng(30)
    n, g, V = 500, 5, 32
    rows = rng.normal(0, 2, size=(g, V))
    d = _draft_fixed(n, rows, seed=31)
    Z = np.concatenate([np.repeat(rows[None], n, axis=0), rng.normal(size=(n, 1, V))], axis=1)
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.full(n, g), 1.0, seed=31)
    assert (v["n_acc"] == g).all() and (v["n_emit"] == g + 1).all()
    np.testing.assert_allclose(v["cstar"], 1.0, atol=1e-12)
    assert (v["tokens"][:, :g] == d["x"]).all()


def test_temperature_applies_to_target():
    rng = np.random.default_rng(40)
    n, V, T = 60000, 8, 0.7
    Zrow = rng.normal(0, 1.0, size=(2, V))
    d = _draft_fixed(n, rng.normal(size=(1, V)), seed=41, T=T)
    Z = np.repeat(Zrow[None], n, axis=0)
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.zeros(n, np.int32), T, seed=41)
    pt = special.softmax(Zrow[0] / T)
    assert stats.chisquare(np.bincount(v["tokens"][:, 0], minlength=V), pt * n).pvalue > 1e-4


def _two_level(lw, seed, req, pos, pg, pe):
    """The two-level Gumbel-max as the header states it: groups of 32 ids by
    log-mass + G(seed, req, pos, pg, group), then ids of the winning group by
    log-weight + G(seed, req, pos, pe, id); fp32 keys, ties to the lowest."""
    V = len(lw)
    gkey = []
    for j in range((V + 31) // 32):
        seg = lw[32 * j: 32 * j + 32]
        if np.all(seg == -np.inf):
            gkey.append(-np.inf)
        else:
            gkey.append(special.logsumexp(seg) + oracle.gumbel(oracle.rng_word(seed, req, pos, pg, j)))
    j = int(np.argmax(np.float32(gkey)))
    seg = range(32 * j, min(V, 32 * j + 32))
    ekey = [lw[v] + oracle.gumbel(oracle.rng_word(seed, req, pos, pe, v)) if lw[v] > -np.inf else -np.inf
            for v in seg]
    return 32 * j + int(np.argmax(np.float32(ekey)))


def test_random_stream_layout_of_each_decision():
    # The counter layout is a convention both sides implement from the header:
    # draft draws use groups (seed, request, k, DRAFT_GROUP, j) then ids
    # (seed, request, k, DRAFT, v), the accept test uses (seed, request, j,
    # ACCEPT, 0) and the resample/bonus draw uses groups (seed, request, row,
    # RESAMPLE_GROUP, j) then ids (seed, request, row, RESAMPLE, v).  Rebuild
    # each decision from those streams (V = 80: two full groups and a short one).
    rng = np.random.default_rng(50)
    n, g, V, seed = 6, 2, 80, 77
    rows = rng.normal(0, 1.5, size=(g, V))
    d = _draft_fixed(n, rows, seed=seed)
    Z = rng.normal(0, 1.5, size=(n, g + 1, V))
    req_ids = np.arange(100, 100 + n)
    d = oracle.draft(np.repeat(rows[None], n, axis=0), np.zeros((V, 1)), np.zeros((1, V)),
                     np.zeros(n, np.int32), 1.0, seed, req_ids=req_ids)
    for i, req in enumerate(req_ids):
        for k in range(1, g + 1):
            x = _two_level(rows[k - 1], seed, req, k, oracle.PURPOSE_DRAFT_GROUP, oracle.PURPOSE_DRAFT)
            assert d["x"][i, k - 1] == x
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.zeros(n, np.int32), 1.0, seed,
                      req_ids=req_ids)
    for i, req in enumerate(req_ids):
        tok = _two_level(Z[i, 0], seed, req, 1, oracle.PURPOSE_RESAMPLE_GROUP, oracle.PURPOSE_RESAMPLE)
        assert v["tokens"][i, 0] == tok
    v = oracle.verify(d["x"], d["logp"], d["lse"], d["scores"], Z, np.full(n, g), 1.0, seed,
                      req_ids=req_ids)
    for i, req in enumerate(req_ids):
        u1 = oracle.uniform(oracle.rng_word(seed, req, 1, oracle.PURPOSE_ACCEPT, 0))
        lse_t = special.logsumexp(Z[i, 0])
        acc = np.float32(np.log(u1)) < np.float32((Z[i, 0, d["x"][i, 0]] - lse_t) - d["logp"][i, 0])
        assert (v["n_acc"][i] >= 1) == bool(acc)
        row = v["n_acc"][i] + 1
        if v["n_acc"][i] < g:  # residual draw at the first rejected row
            pt = special.softmax(Z[i, row - 1])
            pd = np.exp(d["scores"][i, row - 1] - d["lse"][i, row - 1])
            res = pt - pd
            lw = np.where(res > 0, np.log(np.where(res > 0, res, 1.0)), -np.inf)
        else:  # bonus draw at row g + 1
            lw = Z[i, g]
        tok = _two_level(lw, seed, req, row, oracle.PURPOSE_RESAMPLE_GROUP, oracle.PURPOSE_RESAMPLE)
        assert v["tokens"][i, v["n_acc"][i]] == tok
