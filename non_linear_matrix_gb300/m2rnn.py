"""Thin ctypes binding of libm2rnn.so (include/m2rnn.h).

Argument marshalling only: it checks tensor placement and dtypes, allocates
output tensors with torch, passes raw device pointers and the current CUDA
stream to the C ABI and turns non-zero status codes into exceptions.  Every
step of the recurrence runs in the library's CUDA kernels; if the library is
not built this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libm2rnn.so")
# The checked build (index checks in every kernel, M2RNN_ERR_BOUNDS), loaded
# instead of LIB_PATH when M2RNN_LIBRARY=checked or after use_library("checked").
LIB_CHECKED_PATH = os.path.join(_HERE, "_build", "check", "libm2rnn_check.so")

M2RNN_F32, M2RNN_BF16 = 0, 1
STATUS = {
    0: "M2RNN_OK", -1: "M2RNN_ERR_INVALID_ARG", -2: "M2RNN_ERR_UNSUPPORTED_SHAPE",
    -3: "M2RNN_ERR_MISALIGNED", -4: "M2RNN_ERR_POINTER", -5: "M2RNN_ERR_WORKSPACE",
    -6: "M2RNN_ERR_CUDA", -7: "M2RNN_ERR_TIMEOUT", -8: "M2RNN_ERR_BOUNDS",
}

_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_EXPORTS = {
    "m2rnn_version": (ctypes.c_int, []),
    "m2rnn_checked": (ctypes.c_int, []),
    "m2rnn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "m2rnn_num_checkpoints": (ctypes.c_size_t, [_VP]),
    "m2rnn_fwd": (ctypes.c_int, [_VP] * 12),
    "m2rnn_bwd_workspace_size": (ctypes.c_size_t, [_VP, ctypes.c_int]),
    "m2rnn_bwd": (ctypes.c_int, [_VP] * 20 + [ctypes.c_size_t, _VP]),
    "m2rnn_device_status": (ctypes.c_int, [_VP, _VP, ctypes.c_int, _VP]),
    "m2rnn_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_longlong]),
    "m2rnn_set_fault_injection": (ctypes.c_int, [ctypes.c_int]),
    "m2rnn_bwd_noalloc": (ctypes.c_int, [_VP] * 18),
    "m2rnn_decode": (ctypes.c_int, [_VP] * 11),
    "m2rnn_decode_gated": (ctypes.c_int, [_VP] * 13),
    "m2rnn_fwd_gated": (ctypes.c_int, [_VP] * 14),
    "m2rnn_bwd_gated": (ctypes.c_int, [_VP] * 24 + [ctypes.c_size_t, _VP]),
    "m2rnn_fwd_norm": (ctypes.c_int, [_VP] * 13 + [ctypes.c_float] + [_VP] * 6),
    "m2rnn_bwd_norm_workspace_size": (ctypes.c_size_t, [_VP, ctypes.c_int]),
    "m2rnn_bwd_norm": (ctypes.c_int, [_VP] * 31 + [ctypes.c_size_t, _VP]),
}


class M2RNNError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("in_dtype", ctypes.c_int),
                ("ckpt_every", ctypes.c_int), ("Nq", ctypes.c_int)]


def _load(path: str, how: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           f"`python -m non_linear_matrix_gb300.build{how}` (there is no fallback)")
    L = ctypes.CDLL(path)
    for name, (res, args) in _EXPORTS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """The loaded native library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if os.environ.get("M2RNN_LIBRARY") == "checked":
                _lib = _load(LIB_CHECKED_PATH, " checked")
            else:
                _lib = _load(LIB_PATH, "")
    return _lib


def use_library(which: str):
    """Switch every later call to the normal ("normal") or the checked
    ("checked") build; both must have been built.  Each build keeps its own
    device status word."""
    global _lib
    if which not in ("normal", "checked"):
        raise ValueError(which)
    with _lock:
        _lib = _load(LIB_CHECKED_PATH, " checked") if which == "checked" else _load(LIB_PATH, "")


def status_string(code: int) -> str:
    return lib().m2rnn_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise M2RNNError(rc, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return M2RNN_BF16
    if t.dtype == torch.float32:
        return M2RNN_F32
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libm2rnn must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libm2rnn must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(q, v, ckpt_every: int = 0) -> Shape:
    """Shape of a call; q is [B,T,K] (shared by all heads) or [B,T,Nq,K]
    (Nq query/key groups)."""
    if q.dim() == 4:
        B, T, Nq, K = q.shape
    else:
        (B, T, K), Nq = q.shape, 1
    N, V = v.shape[2], v.shape[3]
    return Shape(B, T, N, K, V, _dtype_code(q), int(ckpt_every), Nq)


def num_checkpoints(shape: Shape) -> int:
    return int(lib().m2rnn_num_checkpoints(ctypes.byref(shape)))


def fwd(q, k, v, f, W, w_r, H0=None, *, ckpt_every: int = 0, want_HT: bool = True,
        out=None, stream=None):
    """Forward pass.  Returns (y, H_T or None, ckpt or None).

    q, k [B,T,K]; v [B,T,N,V]; f [B,T,N]; W [N,V,V]; w_r [N,V], all of one
    dtype (bf16 or f32); H0 [B,N,K,V] fp32 or None.  ``out`` may supply a
    dict of preallocated outputs (y, HT, ckpt)."""
    s = make_shape(q, v, ckpt_every)
    for t in (k, v, f, W, w_r):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, f, W, w_r must share one dtype")
    out = dict(out or {})
    y = out.get("y")
    if y is None:
        y = torch.empty_like(v)
    HT = out.get("HT")
    if HT is None and want_HT:
        HT = torch.empty(s.B, s.N, s.K, s.V, device=q.device, dtype=torch.float32)
    ck = out.get("ckpt")
    nck = num_checkpoints(s)
    if ck is None and nck > 0:
        ck = torch.empty(s.B, s.N, nck, s.K, s.V, device=q.device, dtype=torch.float32)
    rc = lib().m2rnn_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W), _ptr(w_r),
                         _ptr(H0), _ptr(y), _ptr(HT), _ptr(ck), _stream(stream))
    _check(rc, "m2rnn_fwd")
    return y, HT, ck


def fwd_gated(q, k, v, a, alpha, beta, W, w_r, H0=None, *, ckpt_every: int = 0,
              want_HT: bool = True, out=None, stream=None):
    """Forward pass with the fused input gate f = exp(-alpha softplus(a + beta)),
    computed inside the kernel.  a [B,T,N]; alpha, beta [N]; the rest as for
    ``fwd``.  Returns (y, H_T or None, ckpt or None)."""
    s = make_shape(q, v, ckpt_every)
    for t in (k, v, a, alpha, beta, W, w_r):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, a, alpha, beta, W, w_r must share one dtype")
    out = dict(out or {})
    y = out.get("y")
    if y is None:
        y = torch.empty_like(v)
    HT = out.get("HT")
    if HT is None and want_HT:
        HT = torch.empty(s.B, s.N, s.K, s.V, device=q.device, dtype=torch.float32)
    ck = out.get("ckpt")
    nck = num_checkpoints(s)
    if ck is None and nck > 0:
        ck = torch.empty(s.B, s.N, nck, s.K, s.V, device=q.device, dtype=torch.float32)
    rc = lib().m2rnn_fwd_gated(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(alpha),
                               _ptr(beta), _ptr(W), _ptr(w_r), _ptr(H0), _ptr(y), _ptr(HT),
                               _ptr(ck), _stream(stream))
    _check(rc, "m2rnn_fwd_gated")
    return y, HT, ck


def decode(q, k, v, f, W, w_r, H, *, H_out=None, y=None, stream=None):
    """One decode step for B sequences.  Returns (y, H_out).

    q, k [B,K] (or [B,Nq,K] with Nq query/key groups); v [B,N,V]; f [B,N];
    W [N,V,V]; w_r [N,V], one dtype (bf16 or f32); H [B,N,K,V] fp32 is the
    state before the step.  H_out defaults to a new tensor; pass ``H_out=H``
    to update the state in place."""
    if q.dim() == 3:
        B, Nq, K = q.shape
    else:
        (B, K), Nq = q.shape, 1
    N, V = v.shape[1], v.shape[2]
    for t in (k, v, f, W, w_r):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, f, W, w_r must share one dtype")
    s = Shape(B, 1, N, K, V, _dtype_code(q), 0, Nq)
    if H_out is None:
        H_out = torch.empty_like(H)
    if y is None:
        y = torch.empty_like(v)
    rc = lib().m2rnn_decode(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W),
                            _ptr(w_r), _ptr(H), _ptr(H_out), _ptr(y), _stream(stream))
    _check(rc, "m2rnn_decode")
    return y, H_out


def decode_gated(q, k, v, a, alpha, beta, W, w_r, H, *, H_out=None, y=None, stream=None):
    """One decode step with the fused input gate: a [B,N], alpha and beta
    [N] replace f; otherwise as ``decode``.  Returns (y, H_out)."""
    if q.dim() == 3:
        B, Nq, K = q.shape
    else:
        (B, K), Nq = q.shape, 1
    N, V = v.shape[1], v.shape[2]
    for t in (k, v, a, alpha, beta, W, w_r):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, a, alpha, beta, W, w_r must share one dtype")
    s = Shape(B, 1, N, K, V, _dtype_code(q), 0, Nq)
    if H_out is None:
        H_out = torch.empty_like(H)
    if y is None:
        y = torch.empty_like(v)
    rc = lib().m2rnn_decode_gated(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(alpha),
                                  _ptr(beta), _ptr(W), _ptr(w_r), _ptr(H), _ptr(H_out), _ptr(y),
                                  _stream(stream))
    _check(rc, "m2rnn_decode_gated")
    return y, H_out


def bwd_workspace_size(shape: Shape, ckpt_given: bool) -> int:
    return int(lib().m2rnn_bwd_workspace_size(ctypes.byref(shape), int(bool(ckpt_given))))


def bwd(q, k, v, f, W, w_r, dy, H0=None, ckpt=None, dHT=None, *, ckpt_every: int = 64,
        want_dH0: bool = False, want_dckpt: bool = False, workspace=None, out=None,
        stream=None):
    """BPTT backward.  Returns dict(dq, dk, dv, df, dW, dw_r[, dH0][, dckpt]) (fp32).

    ``dckpt`` is dL/dH at every checkpoint ([B,N,nck,K,V])."""
    s = make_shape(q, v, ckpt_every)
    dev = q.device
    f32 = dict(device=dev, dtype=torch.float32)
    out = dict(out or {})
    g = {
        "dq": out.get("dq"), "dk": out.get("dk"), "dv": out.get("dv"), "df": out.get("df"),
        "dW": out.get("dW"), "dw_r": out.get("dw_r"),
    }
    shapes = {"dq": tuple(q.shape), "dk": tuple(q.shape), "dv": (s.B, s.T, s.N, s.V),
              "df": (s.B, s.T, s.N), "dW": (s.N, s.V, s.V), "dw_r": (s.N, s.V)}
    for name, shp in shapes.items():
        if g[name] is None:
            g[name] = torch.empty(shp, **f32)
    dH0 = out.get("dH0")
    if dH0 is None and want_dH0:
        dH0 = torch.empty(s.B, s.N, s.K, s.V, **f32)
    dck = out.get("dckpt")
    if dck is None and want_dckpt:
        dck = torch.empty(s.B, s.N, num_checkpoints(s), s.K, s.V, **f32)
    need = bwd_workspace_size(s, ckpt is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    rc = lib().m2rnn_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W), _ptr(w_r),
                         _ptr(H0), _ptr(ckpt), _ptr(dy), _ptr(dHT),
                         _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["df"]),
                         _ptr(g["dW"]), _ptr(g["dw_r"]), _ptr(dH0), _ptr(dck), _ptr(workspace),
                         ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(rc, "m2rnn_bwd")
    if dH0 is not None:
        g["dH0"] = dH0
    if dck is not None:
        g["dckpt"] = dck
    return g


def bwd_noalloc(q, k, v, f, W, w_r, dy, H0=None, dHT=None, *, ckpt_every: int = 64,
                want_dH0: bool = False, out=None, stream=None):
    """Backward pass that allocates nothing inside the library (checkpoints
    are recomputed into a buffer built into it).  Same outputs as
    ``bwd(..., ckpt=None)``; output tensors come from ``out`` or are created
    here by the caller side."""
    s = make_shape(q, v, ckpt_every)
    f32 = dict(device=q.device, dtype=torch.float32)
    out = dict(out or {})
    shapes = {"dq": tuple(q.shape), "dk": tuple(q.shape), "dv": (s.B, s.T, s.N, s.V),
              "df": (s.B, s.T, s.N), "dW": (s.N, s.V, s.V), "dw_r": (s.N, s.V)}
    g = {n: out.get(n) if out.get(n) is not None else torch.empty(shp, **f32)
         for n, shp in shapes.items()}
    dH0 = out.get("dH0")
    if dH0 is None and want_dH0:
        dH0 = torch.empty(s.B, s.N, s.K, s.V, **f32)
    rc = lib().m2rnn_bwd_noalloc(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W),
                                 _ptr(w_r), _ptr(H0), _ptr(dy), _ptr(dHT), _ptr(g["dq"]),
                                 _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["df"]), _ptr(g["dW"]),
                                 _ptr(g["dw_r"]), _ptr(dH0), _stream(stream))
    _check(rc, "m2rnn_bwd_noalloc")
    if dH0 is not None:
        g["dH0"] = dH0
    return g


def bwd_gated(q, k, v, a, alpha, beta, W, w_r, dy, H0=None, ckpt=None, dHT=None, *,
              ckpt_every: int = 64, want_dH0: bool = False, want_dckpt: bool = False,
              workspace=None, out=None, stream=None):
    """BPTT backward through the fused input gate.  Returns dict(dq, dk, dv,
    da, dalpha, dbeta, dW, dw_r[, dH0][, dckpt]) (fp32); ``ckpt`` must come
    from ``fwd_gated`` with the same inputs."""
    s = make_shape(q, v, ckpt_every)
    f32 = dict(device=q.device, dtype=torch.float32)
    out = dict(out or {})
    shapes = {"dq": tuple(q.shape), "dk": tuple(q.shape), "dv": (s.B, s.T, s.N, s.V),
              "da": (s.B, s.T, s.N), "dalpha": (s.N,), "dbeta": (s.N,),
              "dW": (s.N, s.V, s.V), "dw_r": (s.N, s.V)}
    g = {n: out.get(n) if out.get(n) is not None else torch.empty(shp, **f32)
         for n, shp in shapes.items()}
    dH0 = out.get("dH0")
    if dH0 is None and want_dH0:
        dH0 = torch.empty(s.B, s.N, s.K, s.V, **f32)
    dck = out.get("dckpt")
    if dck is None and want_dckpt:
        dck = torch.empty(s.B, s.N, num_checkpoints(s), s.K, s.V, **f32)
    need = bwd_workspace_size(s, ckpt is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    rc = lib().m2rnn_bwd_gated(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(alpha),
                               _ptr(beta), _ptr(W), _ptr(w_r), _ptr(H0), _ptr(ckpt), _ptr(dy),
                               _ptr(dHT), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                               _ptr(g["da"]), _ptr(g["dalpha"]), _ptr(g["dbeta"]), _ptr(g["dW"]),
                               _ptr(g["dw_r"]), _ptr(dH0), _ptr(dck), _ptr(workspace),
                               ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(rc, "m2rnn_bwd_gated")
    if dH0 is not None:
        g["dH0"] = dH0
    if dck is not None:
        g["dckpt"] = dck
    return g


def fwd_norm(q, k, v, f, W, w_r, g, w_norm, eps: float = 0.0, H0=None, *, gate=None,
             ckpt_every: int = 0, want_HT: bool = True, out=None, stream=None):
    """Forward pass with the readout epilogue out = w_norm (.) (y (.) g) rstd,
    rstd = (mean over the token's N*V features of (y (.) g)^2 + eps)^(-1/2).
    ``gate=(a, alpha, beta)`` replaces f (pass f=None).  Returns dict(y, out,
    rstd, HT, ckpt)."""
    s = make_shape(q, v, ckpt_every)
    a, alpha, beta = gate if gate is not None else (None, None, None)
    out = dict(out or {})
    r = {"y": out.get("y"), "out": out.get("out"), "rstd": out.get("rstd"),
         "HT": out.get("HT"), "ckpt": out.get("ckpt")}
    if r["y"] is None:
        r["y"] = torch.empty_like(v)
    if r["out"] is None:
        r["out"] = torch.empty_like(v)
    if r["rstd"] is None:
        r["rstd"] = torch.empty(s.B, s.T, device=q.device, dtype=torch.float32)
    if r["HT"] is None and want_HT:
        r["HT"] = torch.empty(s.B, s.N, s.K, s.V, device=q.device, dtype=torch.float32)
    nck = num_checkpoints(s)
    if r["ckpt"] is None and nck > 0:
        r["ckpt"] = torch.empty(s.B, s.N, nck, s.K, s.V, device=q.device, dtype=torch.float32)
    rc = lib().m2rnn_fwd_norm(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(a),
                              _ptr(alpha), _ptr(beta), _ptr(W), _ptr(w_r), _ptr(H0), _ptr(g),
                              _ptr(w_norm), ctypes.c_float(eps), _ptr(r["y"]), _ptr(r["out"]),
                              _ptr(r["rstd"]), _ptr(r["HT"]), _ptr(r["ckpt"]), _stream(stream))
    _check(rc, "m2rnn_fwd_norm")
    return r


def bwd_norm(q, k, v, f, W, w_r, g, w_norm, y, rstd, dout, H0=None, ckpt=None, dHT=None, *,
             gate=None, ckpt_every: int = 64, want_dH0: bool = False, want_dckpt: bool = False,
             workspace=None, out=None, stream=None):
    """Backward pass through the readout epilogue and the recurrence.
    Returns dict(dq, dk, dv, df | da+dalpha+dbeta, dW, dw_r, dg, dw_norm
    [, dH0][, dckpt]) (fp32)."""
    s = make_shape(q, v, ckpt_every)
    a, alpha, beta = gate if gate is not None else (None, None, None)
    f32 = dict(device=q.device, dtype=torch.float32)
    out = dict(out or {})
    shapes = {"dq": tuple(q.shape), "dk": tuple(q.shape), "dv": (s.B, s.T, s.N, s.V),
              "dW": (s.N, s.V, s.V), "dw_r": (s.N, s.V), "dg": (s.B, s.T, s.N, s.V),
              "dw_norm": (s.N, s.V)}
    if gate is None:
        shapes["df"] = (s.B, s.T, s.N)
    else:
        shapes.update(da=(s.B, s.T, s.N), dalpha=(s.N,), dbeta=(s.N,))
    gr = {n: out.get(n) if out.get(n) is not None else torch.empty(shp, **f32)
          for n, shp in shapes.items()}
    dH0 = out.get("dH0")
    if dH0 is None and want_dH0:
        dH0 = torch.empty(s.B, s.N, s.K, s.V, **f32)
    dck = out.get("dckpt")
    if dck is None and want_dckpt:
        dck = torch.empty(s.B, s.N, num_checkpoints(s), s.K, s.V, **f32)
    need = int(lib().m2rnn_bwd_norm_workspace_size(ctypes.byref(s), int(ckpt is not None)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    dfa = gr["df"] if gate is None else gr["da"]
    rc = lib().m2rnn_bwd_norm(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(a),
                              _ptr(alpha), _ptr(beta), _ptr(W), _ptr(w_r), _ptr(H0), _ptr(ckpt),
                              _ptr(g), _ptr(w_norm), _ptr(y), _ptr(rstd), _ptr(dout), _ptr(dHT),
                              _ptr(gr["dq"]), _ptr(gr["dk"]), _ptr(gr["dv"]), _ptr(dfa),
                              _ptr(gr.get("dalpha")), _ptr(gr.get("dbeta")), _ptr(gr["dW"]),
                              _ptr(gr["dw_r"]), _ptr(gr["dg"]), _ptr(gr["dw_norm"]), _ptr(dH0),
                              _ptr(dck), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                              _stream(stream))
    _check(rc, "m2rnn_bwd_norm")
    if dH0 is not None:
        gr["dH0"] = dH0
    if dck is not None:
        gr["dckpt"] = dck
    return gr


def device_status(clear: bool = True, stream=None):
    """(status, detail) of the device status word; synchronises the stream."""
    st, de = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().m2rnn_device_status(ctypes.byref(st), ctypes.byref(de), int(clear),
                                     _stream(stream)), "m2rnn_device_status")
    return st.value, de.value


def set_wait_limit_ns(limit_ns: int):
    _check(lib().m2rnn_set_wait_limit_ns(int(limit_ns)), "m2rnn_set_wait_limit_ns")


def set_fault_injection(mode: int):
    """Test hook: 1 makes kernels start no input transfers (time-out path)."""
    _check(lib().m2rnn_set_fault_injection(int(mode)), "m2rnn_set_fault_injection")
