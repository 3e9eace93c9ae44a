"""The C-ABI library loads, exports every function include/dspark.h declares,
and rejects bad host-side arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_05_gb300 import build, binding

    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dspark_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ["dspark_draft_sample", "dspark_schedule", "dspark_verify"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.dspark_status_string(code)
    assert lib.dspark_version() >= 10000


def test_workspace_queries_are_host_only(lib):
    assert lib.dspark_draft_workspace_bytes(512, 16, 151936, 256, 1) > 512 * 1187 * 16
    assert lib.dspark_draft_workspace_bytes(0, 16, 151936, 256, 1) == 0
    assert lib.dspark_schedule_workspace_bytes(1024, 16) >= 4
    assert lib.dspark_verify_workspace_bytes(512, 16, 151936) >= 512 * 17 * 4


def _draft(lib, **kw):
    a = dict(U=16, W1=16, W2=16, x0=16, dtype=1, R=4, gamma=4, V=1024, r=64, T=1.0, seed=0, x=16,
             logp=16, lse=16, scores=16, ws=256, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.dspark_draft_sample(a["U"], a["W1"], a["W2"], a["x0"], a["dtype"], a["R"], a["gamma"],
                                   a["V"], a["r"], a["T"], a["seed"], a["x"], a["logp"], a["lse"],
                                   a["scores"], a["ws"], a["wsb"], a["stream"])


def test_draft_rejects_bad_arguments_on_the_host(lib):
    # Every case fails validation before any CUDA call (pointers are never dereferenced).
    assert _draft(lib, U=None) == 1
    assert _draft(lib, R=0) == 1
    assert _draft(lib, T=0.0) == 1
    assert _draft(lib, T=float("nan")) == 1
    assert _draft(lib, dtype=7) == 1
    assert _draft(lib, V=1001) == 2
    assert _draft(lib, r=48) == 2  # bf16 needs r % 64 == 0
    assert _draft(lib, r=512) == 2
    assert _draft(lib, gamma=65) == 2
    assert _draft(lib, U=8) == 1  # not 16-byte aligned
    assert _draft(lib, ws=None) == 3
    assert _draft(lib, wsb=16) == 3


def test_schedule_and_verify_reject_bad_arguments_on_the_host(lib):
    # schedule(conf, sps, sps_len, R, gamma, ell, diag, ws, wsb, stream)
    assert lib.dspark_schedule(None, 16, 100, 4, 4, 16, None, 256, 256, None) == 1
    assert lib.dspark_schedule(16, 16, 10, 4, 4, 16, None, 256, 256, None) == 1  # sps too short
    assert lib.dspark_schedule(16, 16, 10**6, 2048, 16, 16, None, 256, 256, None) == 2
    assert lib.dspark_schedule(16, 16, 100, 4, 4, 16, None, None, 256, None) == 3
    V = 1024
    base = [16, 16, 16, 16, 16, 1, 16, 4, 4, V, ctypes.c_float(1.0), 0, 16, 16, 16, 16, None, 256,
            1 << 20, None]
    bad = list(base)
    bad[4] = None
    assert lib.dspark_verify(*bad[:10], 1.0, *bad[11:]) == 1
    bad = list(base)
    bad[9] = 1020
    assert lib.dspark_verify(*bad[:10], 1.0, *bad[11:]) == 2
    bad = list(base)
    assert lib.dspark_verify(*bad[:10], -1.0, *bad[11:]) == 1
    bad = list(base)
    bad[18] = 8
    assert lib.dspark_verify(*bad[:10], 1.0, *bad[11:]) == 3


def test_zero_overhead_schedule_calls_reject_bad_arguments_on_the_host(lib):
    # capacity(conf_old, sps, sps_len, R, gamma, K, diag, ws, wsb, stream)
    assert lib.dspark_schedule_capacity(None, 16, 100, 4, 4, 16, None, 256, 256, None) == 1
    assert lib.dspark_schedule_capacity(16, 16, 10, 4, 4, 16, None, 256, 256, None) == 1
    assert lib.dspark_schedule_capacity(16, 16, 100, 4, 4, None, None, 256, 256, None) == 1
    assert lib.dspark_schedule_capacity(16, 16, 10**6, 2048, 16, 16, None, 256, 256, None) == 2
    assert lib.dspark_schedule_capacity(16, 16, 100, 4, 4, 16, None, None, 256, None) == 3
    # topk(conf, K, R, gamma, ell, ws, wsb, stream)
    assert lib.dspark_schedule_topk(16, None, 4, 4, 16, 256, 256, None) == 1
    assert lib.dspark_schedule_topk(16, 16, 0, 4, 16, 256, 256, None) == 1
    assert lib.dspark_schedule_topk(16, 16, 4, 65, 16, 256, 1 << 20, None) == 2
    assert lib.dspark_schedule_topk(16, 16, 4, 4, 16, 256, 8, None) == 3


def _draft_rnn(lib, **kw):
    a = dict(U=16, W1=16, W2=16, Wh=16, Q=16, x0=16, dtype=1, R=4, gamma=4, V=1024, r=64, T=1.0, seed=0,
             x=16, logp=16, lse=16, scores=16, ws=256, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.dspark_draft_sample_rnn(a["U"], a["W1"], a["W2"], a["Wh"], a["Q"], a["x0"], a["dtype"],
                                       a["R"], a["gamma"], a["V"], a["r"], a["T"], a["seed"], a["x"],
                                       a["logp"], a["lse"], a["scores"], a["ws"], a["wsb"], a["stream"])


def test_rnn_draft_rejects_bad_arguments_on_the_host(lib):
    # Every case fails validation before any CUDA call (pointers are never dereferenced).
    assert lib.dspark_draft_rnn_workspace_bytes(4, 4, 1024, 64) > lib.dspark_draft_workspace_bytes(4, 4, 1024, 64, 1)
    assert lib.dspark_draft_rnn_workspace_bytes(0, 4, 1024, 64) == 0
    assert _draft_rnn(lib, Wh=None) == 1
    assert _draft_rnn(lib, Q=None) == 1
    assert _draft_rnn(lib, T=0.0) == 1
    assert _draft_rnn(lib, dtype=0) == 2  # fp32: the RNN head is bf16 only
    assert _draft_rnn(lib, r=96) == 2
    assert _draft_rnn(lib, r=320) == 2
    assert _draft_rnn(lib, Wh=24) == 1  # not 16-byte aligned
    assert _draft_rnn(lib, Q=8) == 1
    assert _draft_rnn(lib, ws=None) == 3
    assert _draft_rnn(lib, wsb=16) == 3


def test_transposed_w2_calls_reject_bad_arguments_on_the_host(lib):
    # transpose_w2(W2, r, V, W2T, stream)
    assert lib.dspark_transpose_w2(None, 64, 1024, 16, None) == 1
    assert lib.dspark_transpose_w2(16, 64, 1024, None, None) == 1
    assert lib.dspark_transpose_w2(16, 48, 1024, 16, None) == 2
    assert lib.dspark_transpose_w2(16, 320, 1024, 16, None) == 2
    assert lib.dspark_transpose_w2(16, 64, 1001, 16, None) == 2
    assert lib.dspark_transpose_w2(8, 64, 1024, 16, None) == 1  # not 16-byte aligned

    def draft_w2t(**kw):
        a = dict(U=16, W1=16, W2T=16, x0=16, R=4, gamma=4, V=1024, r=64, T=1.0, seed=0, x=16,
                 logp=16, lse=16, scores=16, ws=256, wsb=1 << 30, stream=None)
        a.update(kw)
        return lib.dspark_draft_sample_w2t(a["U"], a["W1"], a["W2T"], a["x0"], a["R"], a["gamma"],
                                           a["V"], a["r"], a["T"], a["seed"], a["x"], a["logp"],
                                           a["lse"], a["scores"], a["ws"], a["wsb"], a["stream"])

    assert draft_w2t(W2T=None) == 1
    assert draft_w2t(R=0) == 1
    assert draft_w2t(T=-1.0) == 1
    assert draft_w2t(r=48) == 2
    assert draft_w2t(V=1001) == 2
    assert draft_w2t(W2T=8) == 1
    assert draft_w2t(ws=None) == 3

    def rnn_w2t(**kw):
        a = dict(U=16, W1=16, W2T=16, Wh=16, Q=16, x0=16, R=4, gamma=4, V=1024, r=64, T=1.0,
                 seed=0, x=16, logp=16, lse=16, scores=16, ws=256, wsb=1 << 30, stream=None)
        a.update(kw)
        return lib.dspark_draft_sample_rnn_w2t(a["U"], a["W1"], a["W2T"], a["Wh"], a["Q"], a["x0"],
                                               a["R"], a["gamma"], a["V"], a["r"], a["T"],
                                               a["seed"], a["x"], a["logp"], a["lse"], a["scores"],
                                               a["ws"], a["wsb"], a["stream"])

    assert rnn_w2t(W2T=None) == 1
    assert rnn_w2t(Wh=None) == 1
    assert rnn_w2t(r=96) == 2
    assert rnn_w2t(wsb=16) == 3
