"""Pins for the oracle's semi-autoregressive draft (CPU only).

What pins it (DSpark summary §3.1; DSpark notes "DSpark 핵심 기술 1"):
* the Markov bias is a plain matrix product W1[prev] @ W2 -- checked against
  numpy's matmul (a library routine), including which previous token each
  position conditions on (x_0 = anchor for k = 1, x_{k-1} after);
* local normalisation: lse_k is scipy's logsumexp of s_k, sum exp(s - lse) = 1,
  logp_k = s_k(x_k) - lse_k;
* the sampling law: x_k follows softmax(s_k) (chi-square over many
  independent Philox streams), and x_2 | x_1 follows softmax(s_2(x_1)) -- at
  vocabularies of one 32-id group and of several (the two-level draw first
  picks a group by its log-mass, then an id inside it; a wrong group mass or
  a draw confined to the wrong group changes the law).
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _inputs(rng, n, g, V, r, u_std=2.0, w_std=0.3):
    U = rng.normal(0, u_std, size=(n, g, V))
    W1 = rng.normal(0, w_std, size=(V, r))
    W2 = rng.normal(0, w_std, size=(r, V))
    x0 = rng.integers(0, V, size=n).astype(np.int32)
    return U, W1, W2, x0


def test_markov_bias_is_matmul():
    rng = np.random.default_rng(0)
    V, r = 300, 24
    W1 = rng.normal(size=(V, r))
    W2 = rng.normal(size=(r, V))
    prev = rng.integers(0, V, size=17)
    B = oracle.markov_bias(W1, W2, prev)
    np.testing.assert_allclose(B, W1[prev] @ W2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_scores_normaliser_and_conditioning(T):
    rng = np.random.default_rng(1)
    n, g, V, r = 5, 4, 200, 16
    U, W1, W2, x0 = _inputs(rng, n, g, V, r)
    d = oracle.draft(U, W1, W2, x0, T, seed=3)
    prev = np.concatenate([x0[:, None], d["x"][:, :-1]], axis=1)
    expect_s = (U + np.einsum("nkr,rv->nkv", W1[prev], W2)) / T
    np.testing.assert_allclose(d["scores"], expect_s, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(d["lse"], special.logsumexp(expect_s, axis=2), rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(np.exp(d["scores"] - d["lse"][..., None]).sum(axis=2), 1.0, atol=1e-12)
    s_at_x = np.take_along_axis(d["scores"], d["x"][..., None], axis=2)[..., 0]
    np.testing.assert_allclose(d["logp"], s_at_x - d["lse"], atol=1e-13)
    assert ((d["x"] >= 0) & (d["x"] < V)).all()


@pytest.mark.parametrize("V", [8, 80])
def test_draft_first_position_law(V):
    # identical rows for every request; request ids give independent Philox streams
    rng = np.random.default_rng(2)
    n, r = 40000, 4
    U1, W1, W2, _ = _inputs(rng, 1, 1, V, r, u_std=1.0)
    U = np.repeat(U1, n, axis=0)
    x0 = np.full(n, 3, dtype=np.int32)
    d = oracle.draft(U, W1, W2, x0, 1.0, seed=7, want_scores=False)
    p = special.softmax(U1[0, 0] + W1[3] @ W2)
    counts = np.bincount(d["x"][:, 0], minlength=V)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


@pytest.mark.parametrize("V", [6, 40])
def test_draft_second_position_conditional_law(V):
    rng = np.random.default_rng(3)
    n, r = 60000 if V < 32 else 120000, 3
    U1, W1, W2, _ = _inputs(rng, 1, 2, V, r, u_std=0.7, w_std=0.8)
    U = np.repeat(U1, n, axis=0)
    x0 = np.zeros(n, dtype=np.int32)
    d = oracle.draft(U, W1, W2, x0, 1.0, seed=9, want_scores=False)
    x1, x2 = d["x"][:, 0], d["x"][:, 1]
    for a in range(V):
        sel = x1 == a
        if sel.sum() < 2000 * max(1, V // 8):
            continue
        p = special.softmax(U1[0, 1] + W1[a] @ W2)
        counts = np.bincount(x2[sel], minlength=V)
        assert stats.chisquare(counts, p * sel.sum()).pvalue > 1e-4, a


def test_seed_and_request_change_the_stream():
    rng = np.random.default_rng(4)
    U, W1, W2, x0 = _inputs(rng, 64, 3, 512, 8)
    U[:] = U[0]
    x0[:] = x0[0]
    a = oracle.draft(U, W1, W2, x0, 1.0, seed=0, want_scores=False)["x"]
    b = oracle.draft(U, W1, W2, x0, 1.0, seed=1, want_scores=False)["x"]
    assert len({tuple(row) for row in a}) > 32  # different requests draw differently
    assert (a != b).any()
    again = oracle.draft(U, W1, W2, x0, 1.0, seed=0, want_scores=False)["x"]
    assert (a == again).all()  # counter-based: replayable
