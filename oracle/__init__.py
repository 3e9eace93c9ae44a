"""CPU oracle for the DSpark per-round sampling path (draft -> schedule -> verify).

TEST INFRASTRUCTURE ONLY.  The product library (speculative_decoding_draft_05_gb300)
never imports this package.  Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference leg of ``bench.py`` use it.

The arithmetic lives in ``dspark_oracle.c`` (plain loops, fp64).  This module
builds it with gcc on first use and marshals numpy arrays through ctypes.
Function-level citations are in the C file; the summary:

* ``draft``     -- DSpark summary §3.1 and DSpark notes "DSpark 핵심 기술 1":
                   s_k = (U_k + W1[x_{k-1}] W2) / T, lse_k, x_k drawn from
                   softmax(s_k) by two-level Gumbel-max (a group of 32 ids by
                   its log-mass, then an id inside it), logp_k.
* ``draft_rnn`` -- DSpark summary §3.1 (the RNN head: a state across the block
                   and the backbone hidden state; an Elman recurrence in the
                   Markov head's rank-r space).
* ``schedule``  -- DSpark summary §3.2.2 (Algorithm 1).
* ``sts_calibrate`` / ``sts_ece`` / ``schedule_threshold`` -- DSpark summary
                   §3.2.1 (sequential temperature scaling) and §4.3.3 (static
                   threshold).
* ``schedule_capacity`` / ``schedule_topk`` -- DSpark summary §5.2 (zero-overhead
                   scheduling: capacity from old confidences without the early
                   stop, then the top K of the current order).
* ``verify``    -- standard rejection sampling (DSpark summary, opening bullets
                   and §3), soft label c* (DSpark summary §3.2.1).

Each function's pins (closed forms, brute force, golden values, planted mistakes)
are the tests/test_oracle_*.py files.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdspark_oracle.so")
_lock = threading.Lock()
_lib = None

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESAMPLE = 2
PURPOSE_DRAFT_GROUP = 3
PURPOSE_RESAMPLE_GROUP = 4
GROUP = 32  # ids per group of the two-level Gumbel-max


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C, no target-specific flags)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, u32, u64, dbl = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_philox4x32_10.restype = None
            L.oracle_rng_word.argtypes = [u64, u32, u32, u32, u32]
            L.oracle_rng_word.restype = u32
            L.oracle_uniform.argtypes = [u32]
            L.oracle_uniform.restype = dbl
            L.oracle_gumbel.argtypes = [u32]
            L.oracle_gumbel.restype = dbl
            L.oracle_markov_bias_rows.argtypes = [P, P, i32, i32, P, i32, P]
            L.oracle_markov_bias_rows.restype = None
            L.oracle_draft.argtypes = [i32, P, i32, i32, i32, dbl, u64, P, P, P, P, P, P, P, P, P, i32]
            L.oracle_draft.restype = i32
            L.oracle_draft_rnn.argtypes = [i32, P, i32, i32, i32, dbl, u64, P, P, P, P, P, P, P, P, P,
                                           P, P, P, i32]
            L.oracle_draft_rnn.restype = i32
            L.oracle_round_bf16.argtypes = [dbl]
            L.oracle_round_bf16.restype = dbl
            L.oracle_schedule.argtypes = [i32, i32, P, P, i32, P, P, P]
            L.oracle_schedule.restype = i32
            L.oracle_schedule_capacity.argtypes = [i32, i32, P, P, i32, P, P]
            L.oracle_schedule_capacity.restype = i32
            L.oracle_schedule_topk.argtypes = [i32, i32, P, i32, P]
            L.oracle_schedule_topk.restype = i32
            L.oracle_temper.argtypes = [dbl, dbl]
            L.oracle_temper.restype = dbl
            L.oracle_sts_calibrate.argtypes = [i32, i32, P, P, P, i32, i32, P, P]
            L.oracle_sts_calibrate.restype = i32
            L.oracle_sts_ece.argtypes = [i32, i32, P, P, P, i32, P]
            L.oracle_sts_ece.restype = i32
            L.oracle_schedule_threshold.argtypes = [i32, i32, P, P, dbl, P]
            L.oracle_schedule_threshold.restype = i32
            L.oracle_verify.argtypes = [i32, P, i32, i32, dbl, u64, P, P, P, P, P, P, P, P, P, P, P,
                                        P, P, P, i32]
            L.oracle_verify.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------- RNG
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rng_word(seed: int, request: int, position: int, purpose: int, v: int) -> int:
    return int(lib().oracle_rng_word(seed, request, position, purpose, v))


def uniform(word: int) -> float:
    return float(lib().oracle_uniform(word))


def gumbel(word: int) -> float:
    return float(lib().oracle_gumbel(word))


# --------------------------------------------------------------------------- draft
def markov_bias(W1, W2, prev) -> np.ndarray:
    """B rows W1[prev] @ W2 by plain loops, fp64.  prev: int array [n]."""
    W1 = _f64(W1)
    W2 = _f64(W2)
    prev = _i32(prev).reshape(-1)
    V, r = W1.shape
    assert W2.shape == (r, V)
    out = np.empty((prev.size, V), dtype=np.float64)
    lib().oracle_markov_bias_rows(_ptr(W1), _ptr(W2), V, r, _ptr(prev), prev.size, _ptr(out))
    return out


def draft(U, W1, W2, x0, T: float, seed: int, req_ids=None, want_scores=True, nthreads=None):
    """Semi-autoregressive draft for the requests in ``req_ids`` (default: all).

    U: [n, gamma, V] rows of the requests listed in req_ids; W1 [V, r]; W2 [r, V];
    x0: [n] anchors.  Returns dict(x, logp, lse, scores, margin).
    """
    U = _f64(U)
    W1 = _f64(W1)
    W2 = _f64(W2)
    x0 = _i32(x0).reshape(-1)
    n, g, V = U.shape
    r = W1.shape[1]
    req = _i32(np.arange(n) if req_ids is None else req_ids).reshape(-1)
    assert req.size == n and x0.size == n
    x = np.zeros((n, g), dtype=np.int32)
    logp = np.zeros((n, g))
    lse = np.zeros((n, g))
    margin = np.zeros((n, g))
    scores = np.zeros((n, g, V)) if want_scores else None
    rc = lib().oracle_draft(n, _ptr(req), g, V, r, float(T), int(seed), _ptr(U), _ptr(W1), _ptr(W2),
                            _ptr(x0), _ptr(x), _ptr(logp), _ptr(lse), _ptr(scores), _ptr(margin),
                            nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_draft rejected its arguments (code {rc})")
    return dict(x=x, logp=logp, lse=lse, scores=scores, margin=margin)


def round_bf16(v: float) -> float:
    return float(lib().oracle_round_bf16(float(v)))


def draft_rnn(U, W1, W2, Wh, Q, x0, T: float, seed: int, req_ids=None, want_scores=True, want_state=False,
              nthreads=None):
    """Draft with the RNN head: h_k = tanh(W1[x_{k-1}] + h_{k-1} Wh + Q_k), B_k = bf16(h_k) W2.

    U [n, gamma, V]; W1 [V, r]; W2 [r, V]; Wh [r, r]; Q [n, gamma, r]; x0 [n].
    want_state adds "h" [n, gamma, r], the fp64 state h_k of every step."""
    U = _f64(U)
    W1 = _f64(W1)
    W2 = _f64(W2)
    Wh = _f64(Wh)
    Q = _f64(Q)
    x0 = _i32(x0).reshape(-1)
    n, g, V = U.shape
    r = W1.shape[1]
    assert Wh.shape == (r, r) and Q.shape == (n, g, r)
    req = _i32(np.arange(n) if req_ids is None else req_ids).reshape(-1)
    x = np.zeros((n, g), dtype=np.int32)
    logp = np.zeros((n, g))
    lse = np.zeros((n, g))
    margin = np.zeros((n, g))
    scores = np.zeros((n, g, V)) if want_scores else None
    h = np.zeros((n, g, r)) if want_state else None
    rc = lib().oracle_draft_rnn(n, _ptr(req), g, V, r, float(T), int(seed), _ptr(U), _ptr(W1), _ptr(W2),
                                _ptr(Wh), _ptr(Q), _ptr(x0), _ptr(x), _ptr(logp), _ptr(lse),
                                _ptr(scores), _ptr(margin), _ptr(h), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_draft_rnn rejected its arguments (code {rc})")
    out = dict(x=x, logp=logp, lse=lse, scores=scores, margin=margin)
    if want_state:
        out["h"] = h
    return out


# --------------------------------------------------------------------------- schedule
def schedule(conf, sps):
    """Algorithm 1.  conf: [R, gamma] float32; sps: fp64 table indexed by B."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    R, g = c.shape
    s = _f64(sps).reshape(-1)
    ell = np.zeros(R, dtype=np.int32)
    diag = np.zeros(4)
    a = np.zeros((R, g), dtype=np.float32)
    rc = lib().oracle_schedule(R, g, _ptr(c), _ptr(s), s.size, _ptr(ell), _ptr(diag), _ptr(a))
    if rc != 0:
        raise ValueError(f"oracle_schedule rejected its arguments (code {rc}; 3 = a step rate that is not positive and finite)")
    return dict(ell=ell, B=int(diag[0]), tau=float(diag[1]), theta=float(diag[2]),
                n_taken=int(diag[3]), a=a)


def schedule_capacity(conf_old, sps):
    """ZOS capacity K: the first global maximum of Theta along Algorithm 1's order."""
    c = np.ascontiguousarray(conf_old, dtype=np.float32)
    R, g = c.shape
    s = _f64(sps).reshape(-1)
    K = np.zeros(1, dtype=np.int32)
    diag = np.zeros(4)
    rc = lib().oracle_schedule_capacity(R, g, _ptr(c), _ptr(s), s.size, _ptr(K), _ptr(diag))
    if rc != 0:
        raise ValueError(f"oracle_schedule_capacity rejected its arguments (code {rc})")
    return dict(K=int(K[0]), B=int(diag[0]), tau=float(diag[1]), theta=float(diag[2]))


def schedule_topk(conf_now, K: int):
    """ZOS selection: l_r = candidates of r among the top K of the current order."""
    c = np.ascontiguousarray(conf_now, dtype=np.float32)
    R, g = c.shape
    ell = np.zeros(R, dtype=np.int32)
    rc = lib().oracle_schedule_topk(R, g, _ptr(c), int(K), _ptr(ell))
    if rc != 0:
        raise ValueError(f"oracle_schedule_topk rejected its arguments (code {rc})")
    return ell


def sts_grid(n=121):
    """A temperature grid: n log-spaced values from 0.1 to 10, T = 1 exactly in the middle."""
    h = (n - 1) / 2
    return 10.0 ** ((np.arange(n) - h) / h)


def temper(c: float, T: float) -> float:
    return float(lib().oracle_temper(float(c), float(T)))


def sts_calibrate(conf, accept, grid=None, bins=15):
    """Left-to-right grid search of per-position temperatures (minimum ECE each)."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    y = np.ascontiguousarray(accept, dtype=np.uint8)
    N, g = c.shape
    gr = _f64(sts_grid() if grid is None else grid).reshape(-1)
    temps = np.zeros(g)
    ece = np.zeros(g)
    rc = lib().oracle_sts_calibrate(N, g, _ptr(c), _ptr(y), _ptr(gr), gr.size, int(bins), _ptr(temps),
                                    _ptr(ece))
    if rc != 0:
        raise ValueError(f"oracle_sts_calibrate rejected its arguments (code {rc})")
    return dict(temps=temps, ece=ece)


def sts_ece(conf, accept, temps, bins=15):
    c = np.ascontiguousarray(conf, dtype=np.float32)
    y = np.ascontiguousarray(accept, dtype=np.uint8)
    N, g = c.shape
    t = _f64(temps).reshape(-1)
    out = np.zeros(g)
    rc = lib().oracle_sts_ece(N, g, _ptr(c), _ptr(y), _ptr(t), int(bins), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_sts_ece rejected its arguments (code {rc})")
    return out


def schedule_threshold(conf, theta: float, temps=None):
    """Static threshold: l_r = leading positions with calibrated survival >= theta."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    R, g = c.shape
    t = None if temps is None else _f64(temps).reshape(-1)
    ell = np.zeros(R, dtype=np.int32)
    rc = lib().oracle_schedule_threshold(R, g, _ptr(c), _ptr(t), float(theta), _ptr(ell))
    if rc != 0:
        raise ValueError(f"oracle_schedule_threshold rejected its arguments (code {rc})")
    return ell


# --------------------------------------------------------------------------- verify
def verify(x, logp, lse, scores, Z, ell, T: float, seed: int, req_ids=None, nthreads=None):
    """Rejection-sampling verify of the scheduled prefixes.

    x/logp/lse: [n, gamma]; scores: [n, gamma, V]; Z: [n, gamma+1, V]; ell: [n].
    Returns dict(n_acc, tokens, n_emit, cstar, lse_t, acc_margin, res_margin, stop_kind).
    """
    x = _i32(x)
    logp = _f64(logp)
    lse = _f64(lse)
    scores = _f64(scores)
    Z = _f64(Z)
    ell = _i32(ell).reshape(-1)
    n, g = x.shape
    V = scores.shape[2]
    assert Z.shape == (n, g + 1, V)
    req = _i32(np.arange(n) if req_ids is None else req_ids).reshape(-1)
    n_acc = np.zeros(n, dtype=np.int32)
    tokens = np.zeros((n, g + 1), dtype=np.int32)
    n_emit = np.zeros(n, dtype=np.int32)
    cstar = np.zeros((n, g))
    lse_t = np.zeros((n, g + 1))
    acc_margin = np.zeros((n, g))
    res_margin = np.zeros(n)
    stop_kind = np.zeros(n, dtype=np.int32)
    rc = lib().oracle_verify(n, _ptr(req), g, V, float(T), int(seed), _ptr(x), _ptr(logp), _ptr(lse),
                             _ptr(scores), _ptr(Z), _ptr(ell), _ptr(n_acc), _ptr(tokens), _ptr(n_emit),
                             _ptr(cstar), _ptr(lse_t), _ptr(acc_margin), _ptr(res_margin),
                             _ptr(stop_kind), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_verify rejected its arguments (code {rc})")
    return dict(n_acc=n_acc, tokens=tokens, n_emit=n_emit, cstar=cstar, lse_t=lse_t,
                acc_margin=acc_margin, res_margin=res_margin, stop_kind=stop_kind)


def round_(U, W1, W2, x0, conf, sps, Z, T: float, seed: int, nthreads=None):
    """One full round (draft -> schedule -> verify) on all requests."""
    d = draft(U, W1, W2, x0, T, seed, nthreads=nthreads)
    s = schedule(conf, sps)
    v = verify(d["x"], d["logp"], d["lse"], d["scores"], Z, s["ell"], T, seed, nthreads=nthreads)
    return d, s, v
