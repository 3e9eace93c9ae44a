"""Helpers for GPU-vs-oracle parity tests.

Integer outputs must match exactly, except at a documented near tie: a Gumbel
argmax whose top-two perturbed scores differ by less than TIE (1e-5), or an
accept test whose |ln u - (ln p^t - ln p^d)| is below TIE.  Once a request
has an exempt decision, its later values are not compared (they depend on the
choice); the test checks that such exemptions stay rare.
"""
import numpy as np
import torch

import oracle
from speculative_decoding_draft_05_gb300 import workload

TIE = 1e-5
# Floating-point tolerances: 1e-5 absolute on fp32 paths, 2e-3 relative on bf16-input paths.
F32_ATOL = 1e-5
BF16_RTOL = 2e-3
BF16_ATOL = 1e-6


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def close(gpu, ref, dtype, what, extra=None):
    """extra: an optional per-element absolute allowance (same shape), added to the tolerance."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, what
    nan_g, nan_r = np.isnan(gpu), np.isnan(ref)
    assert (nan_g == nan_r).all(), f"{what}: NaN pattern differs"
    g, r = gpu[~nan_g], ref[~nan_r]
    if g.size == 0:
        return
    ex = 0.0 if extra is None else np.broadcast_to(np.asarray(extra, np.float64), gpu.shape)[~nan_g]
    if dtype == "f32":
        err = (np.abs(g - r) - ex).max()
        assert err <= F32_ATOL, f"{what}: max abs error beyond the allowance {err:.3g} > {F32_ATOL}"
    else:
        bad = np.abs(g - r) > BF16_RTOL * np.abs(r) + BF16_ATOL + ex
        assert not bad.any(), (f"{what}: {bad.sum()} values outside rtol {BF16_RTOL}; "
                               f"worst {np.abs(g - r)[bad].max():.3g}")


def compare_draft(gd, od, dtype, scores_ref=None, scores_gpu=None, tie=TIE, score_extra=None):
    """Compare draft outputs request by request.

    At a request's first token mismatch (allowed only at a near tie) the rest of
    that request is not compared: lse is still compared at that position (same
    distribution), logp and later positions are not.  tie is a scalar or an
    [n, gamma] array of per-position ties.  score_extra [n, gamma, V]
    is an optional absolute allowance on the scores (and, through its row
    maximum, on lse, logp and ln p^d).  Returns the exempt set.
    """
    gx = gd["x"]
    n, g = gx.shape
    m_lse = np.ones((n, g), bool)
    m_logp = np.ones((n, g), bool)
    exempt = set()
    for i in range(n):
        for k in range(g):
            if gx[i, k] != od["x"][i, k]:
                t = tie[i, k] if np.ndim(tie) else tie
                assert od["margin"][i, k] < t, (
                    f"draft token differs at request {i} position {k + 1}: gpu {gx[i, k]} oracle "
                    f"{od['x'][i, k]} with margin {od['margin'][i, k]:.3g}")
                exempt.add(i)
                m_lse[i, k + 1:] = False
                m_logp[i, k:] = False
                break
    row_ex = None if score_extra is None else np.asarray(score_extra).max(axis=-1)
    close(gd["lse"][m_lse], od["lse"][m_lse], dtype, "lse", None if row_ex is None else row_ex[m_lse])
    close(gd["logp"][m_logp], od["logp"][m_logp], dtype, "logp",
          None if row_ex is None else 2 * row_ex[m_logp])
    if scores_ref is not None:
        ex = None if score_extra is None else score_extra[m_lse]
        close(scores_gpu[m_lse], scores_ref[m_lse], dtype, "scores", ex)
        pd_g = np.exp(scores_gpu[m_lse] - gd["lse"][m_lse][:, None])
        pd_o = np.exp(scores_ref[m_lse] - od["lse"][m_lse][:, None])
        # |d ln p^d| <= |ds| + |d lse|: a relative allowance on p^d
        close(pd_g, pd_o, dtype, "p^d", None if ex is None else pd_o * (np.expm1(ex + row_ex[m_lse][:, None])))
    return exempt


def compare_verify(gv, ov, ell, dtype, skip=()):
    n = ell.shape[0]
    exempt = set(skip)
    for i in range(n):
        if i in exempt:
            continue
        if gv["n_acc"][i] != ov["n_acc"][i]:
            j = min(gv["n_acc"][i], ov["n_acc"][i])  # first row where the decisions differ
            assert ov["acc_margin"][i, j] < TIE, (
                f"accept decision differs at request {i} row {j + 1}, margin {ov['acc_margin'][i, j]:.3g}")
            exempt.add(i)
            continue
        if (gv["tokens"][i] != ov["tokens"][i]).any():
            assert ov["res_margin"][i] < TIE, (
                f"drawn token differs at request {i}: gpu {gv['tokens'][i].tolist()} oracle "
                f"{ov['tokens'][i].tolist()} margin {ov['res_margin'][i]:.3g}")
            exempt.add(i)
    keep = np.array([i not in exempt for i in range(n)])
    assert (gv["n_emit"] == gv["n_acc"] + 1).all()
    close(gv["cstar"][keep], ov["cstar"][keep], dtype, "c*")
    lt = gv["lse_t"][keep][:, : ov["lse_t"].shape[1]]
    close(lt, ov["lse_t"][keep], dtype, "LSE^t")
    return exempt


def gen_on(w, seed, device):
    return workload.generate(w, seed=seed, device=device)


def oracle_target_bias(W1_64, W2_64, x0, x):
    """Rows of the Markov bias along (x0, x_1..x_gamma), from the oracle: [n, gamma+1, V]."""
    prev = np.concatenate([np.asarray(x0)[:, None], np.asarray(x)], axis=1)
    n, g1 = prev.shape
    return oracle.markov_bias(W1_64, W2_64, prev.reshape(-1)).reshape(n, g1, -1)


def torch_bias_rows(W1, W2, x0, x):
    """Markov bias along (x0, x_1..x_gamma) by torch on the tensors' device: [n, gamma+1, V] fp32."""
    prev = torch.cat([x0.view(-1, 1).long(), x.long()], dim=1)
    n, g1 = prev.shape
    A = W1.float()[prev.view(-1)]
    return (A @ W2.float()).view(n, g1, -1)
