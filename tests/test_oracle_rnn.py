"""Pins for the oracle's RNN-head draft (CPU only).

DSpark summary §3.1: the alternative sequential head keeps a state across the
block and also takes the backbone's hidden state.  The reading is an Elman
recurrence in the Markov head's rank-r space:
    h_0 = 0,  h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k),  B_k = bf16(h_k) W2.

Pins: the bf16 rounding against torch's fp32 -> bf16 conversion; reduction to
the (separately pinned) Markov draft when the state and the backbone input
vanish (Wh = 0, Q = 0: the head is then the Markov head with W1' =
bf16(tanh(W1))); and a constructed recurrence in which only the state of step
1, carried through Wh[0, 1], can make step 2 pick a marked token.
"""
import numpy as np
import torch

import oracle


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(size=2000), rng.uniform(-1, 1, size=2000),
                        [0.0, 1.0, -1.0, 0.5, 2.0 ** -10, 1 - 2.0 ** -9]]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(x)) for x in v])
    assert (got == want).all()


def test_reduces_to_the_markov_head_without_state_and_backbone_input():
    rng = np.random.default_rng(1)
    n, g, V, r = 5, 4, 200, 16
    U = rng.normal(0, 2, size=(n, g, V))
    W1 = rng.normal(0, 0.8, size=(V, r))
    W2 = rng.normal(0, 0.5, size=(r, V))
    x0 = rng.integers(0, V, size=n)
    rnn = oracle.draft_rnn(U, W1, W2, np.zeros((r, r)), np.zeros((n, g, r)), x0, 1.0, 7)
    W1p = np.vectorize(oracle.round_bf16)(np.tanh(W1))
    mk = oracle.draft(U, W1p, W2, x0, 1.0, 7)
    assert (rnn["x"] == mk["x"]).all()
    for k in ("logp", "lse", "scores"):
        assert np.array_equal(rnn[k], mk[k]), k


def test_state_is_carried_through_wh():
    # r = 2, V = 8.  W1 is zero except W1[x0] = (5, 0), so h_1 = (tanh 5, 0).
    # Wh[0, 1] = 3 moves it to h_2 = (0, tanh(3 tanh 5)) ~ (0, 0.995) whatever
    # x_1 is (W1[x_1] = 0 unless x_1 = x0).  W2's row 1 puts +40 on token 6 and
    # row 0 is zero, so step 1 sees no bias and step 2 must pick token 6.
    V, r, x0 = 8, 2, 3
    rng = np.random.default_rng(2)
    W1 = np.zeros((V, r))
    W1[x0, 0] = 5.0
    W2 = np.zeros((r, V))
    W2[1, 6] = 40.0
    Wh = np.zeros((r, r))
    Wh[0, 1] = 3.0
    for seed in range(20):
        U = rng.normal(0, 1, size=(1, 2, V))
        out = oracle.draft_rnn(U, W1, W2, Wh, np.zeros((1, 2, r)), [x0], 1.0, seed)
        if out["x"][0, 0] != x0:
            assert out["x"][0, 1] == 6
        # without the carried state step 2 has no bias: token 6 only by chance
        flat = oracle.draft_rnn(U, W1, W2, np.zeros((r, r)), np.zeros((1, 2, r)), [x0], 1.0, seed)
        np.testing.assert_allclose(flat["scores"][0, 1], U[0, 1])
    # the backbone input enters the same way: Q_2 = (0, 3) alone also forces token 6
    Q = np.zeros((1, 2, r))
    Q[0, 1, 1] = 3.0
    out = oracle.draft_rnn(rng.normal(0, 1, size=(1, 2, V)), np.zeros((V, r)), W2, np.zeros((r, r)), Q,
                           [x0], 1.0, 99)
    assert out["x"][0, 1] == 6


def test_state_output_is_the_recurrence():
    # want_state returns h_k; with W2 = 0 the tokens are the plain Gumbel argmax of
    # U, so the states can be checked step by step against tanh of the recurrence
    rng = np.random.default_rng(3)
    n, g, V, r = 3, 4, 50, 6
    U = rng.normal(0, 1, size=(n, g, V))
    W1 = rng.normal(0, 0.7, size=(V, r))
    Wh = rng.normal(0, 0.4, size=(r, r))
    Q = rng.normal(0, 0.5, size=(n, g, r))
    x0 = rng.integers(0, V, size=n)
    out = oracle.draft_rnn(U, W1, np.zeros((r, V)), Wh, Q, x0, 1.0, 11, want_state=True)
    for i in range(n):
        h, prev = np.zeros(r), x0[i]
        for k in range(g):
            h = np.tanh(W1[prev] + h @ Wh + Q[i, k])
            np.testing.assert_allclose(out["h"][i, k], h, rtol=0, atol=1e-12)
            prev = out["x"][i, k]
