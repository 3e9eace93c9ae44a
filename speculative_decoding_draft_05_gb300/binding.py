"""Thin ctypes binding of libdspark.so (include/dspark.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, then their device pointers go to the C-ABI together with the
current CUDA stream.  Every step of the path runs in the library's kernels.
There is no fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdspark.so")

DSPARK_F32 = 0
DSPARK_BF16 = 1
PURPOSE_DRAFT, PURPOSE_ACCEPT, PURPOSE_RESAMPLE = 0, 1, 2
DEV_BAD_INPUT, DEV_TIMEOUT = 1, 2

_lib = None


class DSparkError(RuntimeError):
    def __init__(self, call: str, status: int):
        lib = load()
        msg = lib.dspark_status_string(status).decode()
        detail = lib.dspark_last_error().decode()
        super().__init__(f"{call} failed: {msg} ({status})" + (f": {detail}" if detail else ""))
        self.status = status


def load() -> ctypes.CDLL:
    """Load libdspark.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, U64, F, D, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float,
                           ctypes.c_double, ctypes.c_size_t)
    L.dspark_status_string.argtypes = [I]
    L.dspark_status_string.restype = ctypes.c_char_p
    L.dspark_last_error.argtypes = []
    L.dspark_last_error.restype = ctypes.c_char_p
    L.dspark_version.restype = I
    L.dspark_draft_workspace_bytes.argtypes = [I, I, I, I, I]
    L.dspark_draft_workspace_bytes.restype = SZ
    L.dspark_draft_sample.argtypes = [P, P, P, P, I, I, I, I, I, F, U64, P, P, P, P, P, SZ, P]
    L.dspark_draft_sample.restype = I
    L.dspark_draft_rnn_workspace_bytes.argtypes = [I, I, I, I]
    L.dspark_draft_rnn_workspace_bytes.restype = SZ
    L.dspark_draft_sample_rnn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, U64, P, P, P, P, P, SZ, P]
    L.dspark_draft_sample_rnn.restype = I
    L.dspark_transpose_w2.argtypes = [P, I, I, P, P]
    L.dspark_transpose_w2.restype = I
    L.dspark_draft_sample_w2t.argtypes = [P, P, P, P, I, I, I, I, F, U64, P, P, P, P, P, SZ, P]
    L.dspark_draft_sample_w2t.restype = I
    L.dspark_draft_sample_rnn_w2t.argtypes = [P, P, P, P, P, P, I, I, I, I, F, U64, P, P, P, P, P,
                                              SZ, P]
    L.dspark_draft_sample_rnn_w2t.restype = I
    L.dspark_schedule_workspace_bytes.argtypes = [I, I]
    L.dspark_schedule_workspace_bytes.restype = SZ
    L.dspark_sts_workspace_bytes.argtypes = [I, I, I]
    L.dspark_sts_workspace_bytes.restype = SZ
    L.dspark_sts_calibrate.argtypes = [P, P, I, I, P, I, I, P, P, P, SZ, P]
    L.dspark_sts_calibrate.restype = I
    L.dspark_schedule_threshold.argtypes = [P, P, D, I, I, P, P]
    L.dspark_schedule_threshold.restype = I
    L.dspark_schedule.argtypes = [P, P, I, I, I, P, P, P, SZ, P]
    L.dspark_schedule.restype = I
    L.dspark_schedule_capacity.argtypes = [P, P, I, I, I, P, P, P, SZ, P]
    L.dspark_schedule_capacity.restype = I
    L.dspark_schedule_topk.argtypes = [P, P, I, I, P, P, SZ, P]
    L.dspark_schedule_topk.restype = I
    L.dspark_verify_workspace_bytes.argtypes = [I, I, I]
    L.dspark_verify_workspace_bytes.restype = SZ
    L.dspark_verify.argtypes = [P, P, P, P, P, I, P, I, I, I, F, U64, P, P, P, P, P, P, SZ, P]
    L.dspark_verify.restype = I
    L.dspark_verify_packed.argtypes = [P, P, P, P, P, I, P, I, P, I, I, I, F, U64, P, P, P, P, P, P,
                                       SZ, P]
    L.dspark_verify_packed.restype = I
    L.dspark_read_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    L.dspark_read_device_status.restype = I
    L.dspark_profile_start.argtypes = []
    L.dspark_profile_start.restype = I
    L.dspark_profile_stop.argtypes = [P, P, P]
    L.dspark_profile_stop.restype = I
    L.dspark_stream_probe.argtypes = [P, P, SZ, P]
    L.dspark_stream_probe.restype = I
    L.dspark_selftest_draft_timeout.argtypes = [P, P, P, P, I, I, I, I, ctypes.c_longlong, P, P, P, P,
                                                P, SZ, P]
    L.dspark_selftest_draft_timeout.restype = I
    _lib = L
    return L


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DSPARK_F32
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(call: str, status: int):
    if status != 0:
        raise DSparkError(call, status)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    return workspace


def draft_workspace_bytes(R: int, gamma: int, V: int, r: int, dtype: torch.dtype) -> int:
    code = DSPARK_BF16 if dtype == torch.bfloat16 else DSPARK_F32
    return int(load().dspark_draft_workspace_bytes(R, gamma, V, r, code))


def schedule_workspace_bytes(R: int, gamma: int) -> int:
    return int(load().dspark_schedule_workspace_bytes(R, gamma))


def sts_workspace_bytes(N: int, G: int, M: int) -> int:
    return int(load().dspark_sts_workspace_bytes(N, G, M))


def dspark_sts_calibrate(conf, accept, grid, bins: int = 15, *, temps=None, ece=None,
                         workspace=None, stream=None) -> dict:
    """Sequential temperature scaling: conf [N, gamma] float32, accept [N, gamma] uint8,
    grid [G] float64 (all on the device).  Returns temps, ece [gamma] float64."""
    L = load()
    N, g = conf.shape
    G = grid.numel()
    dev = conf.device
    temps = torch.empty(g, dtype=torch.float64, device=dev) if temps is None else temps
    ece = torch.empty(g, dtype=torch.float64, device=dev) if ece is None else ece
    ws = _workspace(sts_workspace_bytes(N, G, bins), dev, workspace)
    st = L.dspark_sts_calibrate(_dev(conf, "conf", torch.float32), _dev(accept, "accept", torch.uint8, (N, g)),
                                N, g, _dev(grid, "grid", torch.float64, (G,)), G, int(bins),
                                _dev(temps, "temps", torch.float64, (g,)),
                                _dev(ece, "ece", torch.float64, (g,)), ws.data_ptr(), ws.numel(),
                                _stream(stream))
    _check("dspark_sts_calibrate", st)
    return dict(temps=temps, ece=ece, workspace=ws)


def dspark_schedule_threshold(conf, theta: float, temps=None, *, ell=None, stream=None) -> dict:
    """Static threshold: l_r = leading positions whose (calibrated) survival >= theta."""
    L = load()
    R, g = conf.shape
    dev = conf.device
    ell = torch.empty(R, dtype=torch.int32, device=dev) if ell is None else ell
    st = L.dspark_schedule_threshold(_dev(conf, "conf", torch.float32),
                                     None if temps is None else _dev(temps, "temps", torch.float64, (g,)),
                                     float(theta), R, g, _dev(ell, "ell", torch.int32, (R,)),
                                     _stream(stream))
    _check("dspark_schedule_threshold", st)
    return dict(ell=ell)


def verify_workspace_bytes(R: int, gamma: int, V: int) -> int:
    return int(load().dspark_verify_workspace_bytes(R, gamma, V))


def dspark_draft_sample(U, W1, W2, x0, temperature: float, seed: int, *, x=None, logp=None,
                        lse=None, scores=None, workspace=None, stream=None) -> dict:
    """Semi-autoregressive draft.  U [R, gamma, V], W1 [V, r], W2 [r, V] (fp32 or bf16), x0 [R] int32."""
    L = load()
    R, g, V = U.shape
    r = W1.shape[1]
    dt = U.dtype
    dev = U.device
    x = torch.empty(R, g, dtype=torch.int32, device=dev) if x is None else x
    logp = torch.empty(R, g, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(R, g, dtype=torch.float32, device=dev) if lse is None else lse
    scores = torch.empty(R, g, V, dtype=torch.float32, device=dev) if scores is None else scores
    ws = _workspace(draft_workspace_bytes(R, g, V, r, dt), dev, workspace)
    st = L.dspark_draft_sample(
        _dev(U, "U", dt), _dev(W1, "W1", dt, (V, r)), _dev(W2, "W2", dt, (r, V)),
        _dev(x0, "x0", torch.int32, (R,)), _dtype_code(U), R, g, V, r, float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(x, "x", torch.int32, (R, g)),
        _dev(logp, "logp", torch.float32, (R, g)), _dev(lse, "lse", torch.float32, (R, g)),
        _dev(scores, "scores", torch.float32, (R, g, V)), ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_draft_sample", st)
    return dict(x=x, logp=logp, lse=lse, scores=scores, workspace=ws)


def dspark_transpose_w2(W2, W2T=None, *, stream=None):
    """W2 [r, V] bf16 -> W2T [V, r] bf16, the layout dspark_draft_sample_w2t reads."""
    L = load()
    r, V = W2.shape
    W2T = torch.empty(V, r, dtype=torch.bfloat16, device=W2.device) if W2T is None else W2T
    st = L.dspark_transpose_w2(_dev(W2, "W2", torch.bfloat16, (r, V)), r, V,
                               _dev(W2T, "W2T", torch.bfloat16, (V, r)), _stream(stream))
    _check("dspark_transpose_w2", st)
    return W2T


def dspark_draft_sample_w2t(U, W1, W2T, x0, temperature: float, seed: int, *, x=None, logp=None,
                            lse=None, scores=None, workspace=None, stream=None) -> dict:
    """dspark_draft_sample (bf16) with W2 given as W2T [V, r] from dspark_transpose_w2."""
    L = load()
    R, g, V = U.shape
    r = W1.shape[1]
    dt = torch.bfloat16
    dev = U.device
    x = torch.empty(R, g, dtype=torch.int32, device=dev) if x is None else x
    logp = torch.empty(R, g, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(R, g, dtype=torch.float32, device=dev) if lse is None else lse
    scores = torch.empty(R, g, V, dtype=torch.float32, device=dev) if scores is None else scores
    ws = _workspace(draft_workspace_bytes(R, g, V, r, dt), dev, workspace)
    st = L.dspark_draft_sample_w2t(
        _dev(U, "U", dt), _dev(W1, "W1", dt, (V, r)), _dev(W2T, "W2T", dt, (V, r)),
        _dev(x0, "x0", torch.int32, (R,)), R, g, V, r, float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(x, "x", torch.int32, (R, g)),
        _dev(logp, "logp", torch.float32, (R, g)), _dev(lse, "lse", torch.float32, (R, g)),
        _dev(scores, "scores", torch.float32, (R, g, V)), ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_draft_sample_w2t", st)
    return dict(x=x, logp=logp, lse=lse, scores=scores, workspace=ws)


def draft_rnn_workspace_bytes(R: int, gamma: int, V: int, r: int) -> int:
    return int(load().dspark_draft_rnn_workspace_bytes(R, gamma, V, r))


def dspark_draft_sample_rnn(U, W1, W2, Wh, Q, x0, temperature: float, seed: int, *, x=None,
                            logp=None, lse=None, scores=None, workspace=None, stream=None) -> dict:
    """Draft with the RNN head.  U [R, gamma, V], W1 [V, r], W2 [r, V], Wh [r, r] (bf16),
    Q [R, gamma, r] float32, x0 [R] int32."""
    L = load()
    R, g, V = U.shape
    r = W1.shape[1]
    dt = U.dtype
    dev = U.device
    x = torch.empty(R, g, dtype=torch.int32, device=dev) if x is None else x
    logp = torch.empty(R, g, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(R, g, dtype=torch.float32, device=dev) if lse is None else lse
    scores = torch.empty(R, g, V, dtype=torch.float32, device=dev) if scores is None else scores
    ws = _workspace(draft_rnn_workspace_bytes(R, g, V, r), dev, workspace)
    st = L.dspark_draft_sample_rnn(
        _dev(U, "U", dt), _dev(W1, "W1", dt, (V, r)), _dev(W2, "W2", dt, (r, V)),
        _dev(Wh, "Wh", dt, (r, r)), _dev(Q, "Q", torch.float32, (R, g, r)),
        _dev(x0, "x0", torch.int32, (R,)), _dtype_code(U), R, g, V, r, float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(x, "x", torch.int32, (R, g)),
        _dev(logp, "logp", torch.float32, (R, g)), _dev(lse, "lse", torch.float32, (R, g)),
        _dev(scores, "scores", torch.float32, (R, g, V)), ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_draft_sample_rnn", st)
    return dict(x=x, logp=logp, lse=lse, scores=scores, workspace=ws)


def dspark_draft_sample_rnn_w2t(U, W1, W2T, Wh, Q, x0, temperature: float, seed: int, *, x=None,
                                logp=None, lse=None, scores=None, workspace=None,
                                stream=None) -> dict:
    """dspark_draft_sample_rnn with W2 given as W2T [V, r] from dspark_transpose_w2."""
    L = load()
    R, g, V = U.shape
    r = W1.shape[1]
    dt = torch.bfloat16
    dev = U.device
    x = torch.empty(R, g, dtype=torch.int32, device=dev) if x is None else x
    logp = torch.empty(R, g, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(R, g, dtype=torch.float32, device=dev) if lse is None else lse
    scores = torch.empty(R, g, V, dtype=torch.float32, device=dev) if scores is None else scores
    ws = _workspace(draft_rnn_workspace_bytes(R, g, V, r), dev, workspace)
    st = L.dspark_draft_sample_rnn_w2t(
        _dev(U, "U", dt), _dev(W1, "W1", dt, (V, r)), _dev(W2T, "W2T", dt, (V, r)),
        _dev(Wh, "Wh", dt, (r, r)), _dev(Q, "Q", torch.float32, (R, g, r)),
        _dev(x0, "x0", torch.int32, (R,)), R, g, V, r, float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(x, "x", torch.int32, (R, g)),
        _dev(logp, "logp", torch.float32, (R, g)), _dev(lse, "lse", torch.float32, (R, g)),
        _dev(scores, "scores", torch.float32, (R, g, V)), ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_draft_sample_rnn_w2t", st)
    return dict(x=x, logp=logp, lse=lse, scores=scores, workspace=ws)


def dspark_schedule(conf, sps, *, ell=None, diag=None, workspace=None, stream=None) -> dict:
    """Algorithm 1.  conf [R, gamma] float32, sps float64 indexed by B."""
    L = load()
    R, g = conf.shape
    dev = conf.device
    ell = torch.empty(R, dtype=torch.int32, device=dev) if ell is None else ell
    diag = torch.empty(4, dtype=torch.float64, device=dev) if diag is None else diag
    ws = _workspace(schedule_workspace_bytes(R, g), dev, workspace)
    st = L.dspark_schedule(_dev(conf, "conf", torch.float32), _dev(sps, "sps", torch.float64),
                           sps.numel(), R, g, _dev(ell, "ell", torch.int32, (R,)),
                           _dev(diag, "diag", torch.float64, (4,)), ws.data_ptr(), ws.numel(),
                           _stream(stream))
    _check("dspark_schedule", st)
    return dict(ell=ell, diag=diag, workspace=ws)


def dspark_schedule_capacity(conf_old, sps, *, K=None, diag=None, workspace=None,
                             stream=None) -> dict:
    """Zero-overhead scheduling, capacity: K from old confidences (no early stop)."""
    L = load()
    R, g = conf_old.shape
    dev = conf_old.device
    K = torch.empty(1, dtype=torch.int32, device=dev) if K is None else K
    diag = torch.empty(4, dtype=torch.float64, device=dev) if diag is None else diag
    ws = _workspace(schedule_workspace_bytes(R, g), dev, workspace)
    st = L.dspark_schedule_capacity(_dev(conf_old, "conf_old", torch.float32),
                                    _dev(sps, "sps", torch.float64), sps.numel(), R, g,
                                    _dev(K, "K", torch.int32, (1,)),
                                    _dev(diag, "diag", torch.float64, (4,)), ws.data_ptr(),
                                    ws.numel(), _stream(stream))
    _check("dspark_schedule_capacity", st)
    return dict(K=K, diag=diag, workspace=ws)


def dspark_schedule_topk(conf, K, *, ell=None, workspace=None, stream=None) -> dict:
    """Zero-overhead scheduling, selection: the top K (device int32 [1]) of conf's order."""
    L = load()
    R, g = conf.shape
    dev = conf.device
    ell = torch.empty(R, dtype=torch.int32, device=dev) if ell is None else ell
    ws = _workspace(schedule_workspace_bytes(R, g), dev, workspace)
    st = L.dspark_schedule_topk(_dev(conf, "conf", torch.float32), _dev(K, "K", torch.int32, (1,)),
                                R, g, _dev(ell, "ell", torch.int32, (R,)), ws.data_ptr(),
                                ws.numel(), _stream(stream))
    _check("dspark_schedule_topk", st)
    return dict(ell=ell, workspace=ws)


def dspark_verify(x, logp, lse, scores, Z, ell, temperature: float, seed: int, *, n_acc=None,
                  tokens=None, n_emit=None, cstar=None, lse_t=None, want_lse_t=True,
                  workspace=None, stream=None) -> dict:
    """Rejection-sampling verify.  Z [R, gamma+1, V] (fp32 or bf16)."""
    L = load()
    R, g = x.shape
    V = scores.shape[2]
    dev = x.device
    n_acc = torch.empty(R, dtype=torch.int32, device=dev) if n_acc is None else n_acc
    tokens = torch.empty(R, g + 1, dtype=torch.int32, device=dev) if tokens is None else tokens
    n_emit = torch.empty(R, dtype=torch.int32, device=dev) if n_emit is None else n_emit
    cstar = torch.empty(R, g, dtype=torch.float32, device=dev) if cstar is None else cstar
    if lse_t is None and want_lse_t:
        lse_t = torch.empty(R, g + 1, dtype=torch.float32, device=dev)
    ws = _workspace(verify_workspace_bytes(R, g, V), dev, workspace)
    st = L.dspark_verify(
        _dev(x, "x", torch.int32, (R, g)), _dev(logp, "logp", torch.float32, (R, g)),
        _dev(lse, "lse", torch.float32, (R, g)), _dev(scores, "scores", torch.float32, (R, g, V)),
        _dev(Z, "Z", None, (R, g + 1, V)), _dtype_code(Z), _dev(ell, "ell", torch.int32, (R,)), R, g, V,
        float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(n_acc, "n_acc", torch.int32, (R,)),
        _dev(tokens, "tokens", torch.int32, (R, g + 1)), _dev(n_emit, "n_emit", torch.int32, (R,)),
        _dev(cstar, "cstar", torch.float32, (R, g)),
        None if lse_t is None else _dev(lse_t, "lse_t", torch.float32, (R, g + 1)),
        ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_verify", st)
    return dict(n_acc=n_acc, tokens=tokens, n_emit=n_emit, cstar=cstar, lse_t=lse_t, workspace=ws)


def dspark_verify_packed(x, logp, lse, scores, Zp, row_offsets, ell, temperature: float,
                         seed: int, *, n_acc=None, tokens=None, n_emit=None, cstar=None,
                         lse_t=None, want_lse_t=True, workspace=None, stream=None) -> dict:
    """dspark_verify with packed target logits: Zp [n_rows, V]; request r's rows
    for positions 1..l_r+1 start at row_offsets[r] (int32 [R + 1], on the device)."""
    L = load()
    R, g = x.shape
    V = scores.shape[2]
    dev = x.device
    n_rows = Zp.shape[0]
    n_acc = torch.empty(R, dtype=torch.int32, device=dev) if n_acc is None else n_acc
    tokens = torch.empty(R, g + 1, dtype=torch.int32, device=dev) if tokens is None else tokens
    n_emit = torch.empty(R, dtype=torch.int32, device=dev) if n_emit is None else n_emit
    cstar = torch.empty(R, g, dtype=torch.float32, device=dev) if cstar is None else cstar
    if lse_t is None and want_lse_t:
        lse_t = torch.empty(R, g + 1, dtype=torch.float32, device=dev)
    ws = _workspace(verify_workspace_bytes(R, g, V), dev, workspace)
    st = L.dspark_verify_packed(
        _dev(x, "x", torch.int32, (R, g)), _dev(logp, "logp", torch.float32, (R, g)),
        _dev(lse, "lse", torch.float32, (R, g)), _dev(scores, "scores", torch.float32, (R, g, V)),
        _dev(Zp, "Zp", None, (n_rows, V)), _dtype_code(Zp),
        _dev(row_offsets, "row_offsets", torch.int32, (R + 1,)), n_rows,
        _dev(ell, "ell", torch.int32, (R,)), R, g, V, float(temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev(n_acc, "n_acc", torch.int32, (R,)),
        _dev(tokens, "tokens", torch.int32, (R, g + 1)), _dev(n_emit, "n_emit", torch.int32, (R,)),
        _dev(cstar, "cstar", torch.float32, (R, g)),
        None if lse_t is None else _dev(lse_t, "lse_t", torch.float32, (R, g + 1)),
        ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_verify_packed", st)
    return dict(n_acc=n_acc, tokens=tokens, n_emit=n_emit, cstar=cstar, lse_t=lse_t, workspace=ws)


def dspark_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Device status word of the last call that used ``workspace`` (synchronises)."""
    out = ctypes.c_int32(0)
    _check("dspark_read_device_status",
           load().dspark_read_device_status(workspace.data_ptr(), _stream(stream), ctypes.byref(out)))
    return int(out.value)


KERNEL_KINDS = ["prepare", "draft_tile", "draft_combine", "schedule", "verify_rows", "verify_draw",
                "rnn_state", "verify_emit"]


def dspark_stream_probe(inp, out, stream=None) -> None:
    """Bandwidth probe: out[i] = float(inp[i]) for contiguous bf16 inp and float32 out
    (a measurement aid for the draft step's 2-byte-in / 4-byte-out traffic mix)."""
    if inp.dtype != torch.bfloat16 or out.dtype != torch.float32 or inp.numel() != out.numel():
        raise ValueError("stream probe: bf16 input and float32 output of the same size")
    if not (inp.is_cuda and out.is_cuda and inp.is_contiguous() and out.is_contiguous()):
        raise ValueError("stream probe: contiguous device tensors")
    _check("dspark_stream_probe", load().dspark_stream_probe(inp.data_ptr(), out.data_ptr(), inp.numel(),
                                                             _stream(stream)))


def dspark_profile_start() -> None:
    """Start event-timing every kernel launch of the library (on its own stream)."""
    _check("dspark_profile_start", load().dspark_profile_start())


def dspark_profile_stop() -> dict:
    """Stop timing; returns {kind: (summed ms, launches)} and the number of timed launches."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    timed = ctypes.c_int(0)
    _check("dspark_profile_stop", load().dspark_profile_stop(ms, cnt, ctypes.byref(timed)))
    out = {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}
    out["_timed_launches"] = int(timed.value)
    return out


def dspark_selftest_draft_timeout(U, W1, W2, x0, wait_cycles: int, *, workspace=None,
                                  stream=None) -> torch.Tensor:
    """Diagnostic: the tensor-core draft's step 1 with its W2 loads withheld and
    every device wait limited to ``wait_cycles`` SM clocks, so that the bounded
    waits run out.  Returns the workspace (its status word then carries
    DEV_TIMEOUT; read it with dspark_read_device_status)."""
    L = load()
    R, g, V = U.shape
    r = W1.shape[1]
    dev = U.device
    x = torch.empty(R, g, dtype=torch.int32, device=dev)
    logp = torch.empty(R, g, dtype=torch.float32, device=dev)
    lse = torch.empty(R, g, dtype=torch.float32, device=dev)
    scores = torch.empty(R, g, V, dtype=torch.float32, device=dev)
    ws = _workspace(draft_workspace_bytes(R, g, V, r, torch.bfloat16), dev, workspace)
    st = L.dspark_selftest_draft_timeout(
        _dev(U, "U", torch.bfloat16, (R, g, V)), _dev(W1, "W1", torch.bfloat16, (V, r)),
        _dev(W2, "W2", torch.bfloat16, (r, V)), _dev(x0, "x0", torch.int32, (R,)), R, g, V, r,
        int(wait_cycles), x.data_ptr(), logp.data_ptr(), lse.data_ptr(), scores.data_ptr(),
        ws.data_ptr(), ws.numel(), _stream(stream))
    _check("dspark_selftest_draft_timeout", st)
    return ws
