"""fp64 CPU oracle for the M2RNN recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``m2rnn_oracle.c`` (plain C, fp64, OpenMP over
independent (batch, head) pairs).  It follows Eqs. (10)-(12) of "M2RNN:
Non-Linear RNNs with Matrix-Valued States" (frame "Write, transform, retain,
and read a matrix state" of the paper-discussion deck) for the forward pass,
and the chain rule of the backup frame "the recurrent gradient needs both
paths" for the backward pass.  This module only compiles that file, converts
arrays to contiguous float64 and marshals pointers.

Layouts: q, k [B,T,K]; v [B,T,N,V]; f [B,T,N]; W [N,V,V] with
(H W)_{ij} = sum_l H_{il} W_{lj}; w_r [N,V]; H0/H_T [B,N,K,V]; y [B,T,N,V].

Grouped queries and keys (frame "Tensor parallelism trades topology
dependence for sync": one query/key group per group of value heads, N_q =
N_k = G): q and k may be given as [B,T,G,K] with G dividing N.  Value head n
then reads group n // (N / G) (contiguous blocks of N / G heads, one block
per tensor-parallel rank in the deck's topology-aware form), and dq, dk are
[B,T,G,K], summed over the heads of each group.  Each group is an
independent problem with N_q = 1, so fwd / bwd run the C routines once per
group on that group's slices.

The readout epilogue follows the frames "Most of the block can be computed
before recurrence" (after readout: multiply by the output gate g_t, apply
RMSNorm) and "Backup: RMSNormTP synchronizes per-token statistics" (the norm
and its gradient): o = y (.) g over a token's d = N*V features, s =
(mean_d o^2 + eps)^(-1/2), out = w (.) o s; backward p = w (.) dout,
r = sum_d p o, do = s p - r s^3 o / d.  eps = 0 is the pages' form (they omit
it); the functions take it as an argument.

The gated functions follow the frame "The gate preserves a direct path
through time": f_{t,n} = exp(-alpha_n softplus(a_{t,n} + beta_n)), with a
[B,T,N] and alpha, beta [N].  They compute f (and the gate's derivatives) in
numpy fp64 and call the same C routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m2rnn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libm2rnn_oracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.m2rnn_oracle_threads.restype = ctypes.c_int
            lib.m2rnn_oracle_fwd.restype = ctypes.c_int
            lib.m2rnn_oracle_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses (honours OMP_NUM_THREADS)."""
    return int(_load().m2rnn_oracle_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def _dims(q, v):
    B, T, K = q.shape
    N, V = v.shape[2], v.shape[3]
    return B, T, N, K, V


def _groups(q, v):
    """Head blocks [(group, first head, last head + 1)] of grouped q/k."""
    G, N = q.shape[2], v.shape[2]
    if N % G != 0:
        raise ValueError(f"{G} q/k groups do not divide {N} value heads")
    hpg = N // G
    return [(g, g * hpg, (g + 1) * hpg) for g in range(G)]


def fwd(q, k, v, f, W, w_r, H0=None, want_states: bool = False):
    """Forward pass.  Returns dict(y, HT[, states]) as float64 arrays.

    ``states`` (if requested) holds H_0..H_T as [B,N,T+1,K,V].  q, k are
    [B,T,K] (shared by all heads) or [B,T,G,K] (grouped)."""
    q, k, v, f, W, w_r, H0 = map(_f64, (q, k, v, f, W, w_r, H0))
    if q.ndim == 4:  # grouped: one N_q = 1 problem per group of heads
        parts = [(h0, h1, fwd(q[:, :, g], k[:, :, g], v[:, :, h0:h1], f[:, :, h0:h1],
                              W[h0:h1], w_r[h0:h1], None if H0 is None else H0[:, h0:h1],
                              want_states))
                 for g, h0, h1 in _groups(q, v)]
        out = {"y": np.concatenate([r["y"] for *_, r in parts], axis=2),
               "HT": np.concatenate([r["HT"] for *_, r in parts], axis=1)}
        if want_states:
            out["states"] = np.concatenate([r["states"] for *_, r in parts], axis=1)
        return out
    B, T, N, K, V = _dims(q, v)
    y = np.zeros((B, T, N, V))
    HT = np.zeros((B, N, K, V))
    states = np.zeros((B, N, T + 1, K, V)) if want_states else None
    rc = _load().m2rnn_oracle_fwd(B, T, N, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(f),
                                  _ptr(W), _ptr(w_r), _ptr(H0), _ptr(y), _ptr(HT),
                                  _ptr(states))
    if rc != 0:
        raise RuntimeError(f"m2rnn_oracle_fwd failed: {rc}")
    out = {"y": y, "HT": HT}
    if want_states:
        out["states"] = states
    return out


def bwd(q, k, v, f, W, w_r, dy, H0=None, dHT=None):
    """BPTT backward.  Returns dict(dq, dk, dv, df, dW, dw_r, dH0) (float64);
    with grouped q, k ([B,T,G,K]) dq and dk are [B,T,G,K]."""
    q, k, v, f, W, w_r, dy, H0, dHT = map(_f64, (q, k, v, f, W, w_r, dy, H0, dHT))
    if q.ndim == 4:  # grouped: one N_q = 1 problem per group of heads
        sl = lambda a, h0, h1: None if a is None else a[:, h0:h1]  # noqa: E731
        parts = [bwd(q[:, :, g], k[:, :, g], v[:, :, h0:h1], f[:, :, h0:h1], W[h0:h1],
                     w_r[h0:h1], dy[:, :, h0:h1], sl(H0, h0, h1), sl(dHT, h0, h1))
                 for g, h0, h1 in _groups(q, v)]
        out = {n: np.stack([r[n] for r in parts], axis=2) for n in ("dq", "dk")}
        for n, ax in (("dv", 2), ("df", 2), ("dW", 0), ("dw_r", 0), ("dH0", 1)):
            out[n] = np.concatenate([r[n] for r in parts], axis=ax)
        return out
    B, T, N, K, V = _dims(q, v)
    out = {
        "dq": np.zeros((B, T, K)), "dk": np.zeros((B, T, K)),
        "dv": np.zeros((B, T, N, V)), "df": np.zeros((B, T, N)),
        "dW": np.zeros((N, V, V)), "dw_r": np.zeros((N, V)),
        "dH0": np.zeros((B, N, K, V)),
    }
    rc = _load().m2rnn_oracle_bwd(B, T, N, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(f),
                                  _ptr(W), _ptr(w_r), _ptr(H0), _ptr(dy), _ptr(dHT),
                                  *(_ptr(out[n]) for n in
                                    ("dq", "dk", "dv", "df", "dW", "dw_r", "dH0")))
    if rc != 0:
        raise RuntimeError(f"m2rnn_oracle_bwd failed: {rc}")
    return out


def _gate_parts(a, alpha, beta):
    """x = a + beta, softplus(x), f = exp(-alpha softplus(x)), sigmoid(x) (fp64)."""
    a, alpha, beta = map(_f64, (a, alpha, beta))
    x = a + beta                                   # beta broadcasts over [..., N]
    sp = np.logaddexp(0.0, x)                      # softplus(x) = log(1 + e^x)
    f = np.exp(-alpha * sp)
    sig = 0.5 * (1.0 + np.tanh(0.5 * x))           # sigmoid(x) = softplus'(x)
    return x, sp, f, sig


def gate(a, alpha, beta):
    """f_{t,n} = exp(-alpha_n softplus(a_{t,n} + beta_n)) (float64)."""
    return _gate_parts(a, alpha, beta)[2]


def fwd_gated(q, k, v, a, alpha, beta, W, w_r, H0=None, want_states: bool = False):
    """Forward pass with the input gate computed from a."""
    return fwd(q, k, v, gate(a, alpha, beta), W, w_r, H0, want_states)


def bwd_gated(q, k, v, a, alpha, beta, W, w_r, dy, H0=None, dHT=None):
    """Backward pass with the input gate: the chain rule through
    f = exp(-alpha s), s = softplus(a + beta):
        df/da = df/dbeta = -alpha f sigmoid(a + beta),   df/dalpha = -s f.
    Returns dict(dq, dk, dv, da, dalpha, dbeta, dW, dw_r, dH0) (float64)."""
    _, sp, f, sig = _gate_parts(a, alpha, beta)
    r = bwd(q, k, v, f, W, w_r, dy, H0, dHT)
    alpha64 = _f64(alpha)
    df = r.pop("df")
    da = df * (-alpha64 * f * sig)
    r["da"] = da
    r["dalpha"] = (df * (-sp * f)).reshape(-1, df.shape[-1]).sum(axis=0)
    r["dbeta"] = da.reshape(-1, da.shape[-1]).sum(axis=0)
    return r


def readout_norm(y, g, w, eps: float = 0.0):
    """out = w (.) o s with o = y (.) g and s = (mean over the token's N*V
    features of o^2 + eps)^(-1/2).  y, g [B,T,N,V]; w [N,V].  Returns
    dict(out [B,T,N,V], rstd s [B,T]) (float64)."""
    y, g, w = map(_f64, (y, g, w))
    o = y * g
    d = o.shape[2] * o.shape[3]
    s = 1.0 / np.sqrt((o * o).sum(axis=(2, 3)) / d + eps)
    return {"out": w[None, None] * o * s[:, :, None, None], "rstd": s}


def readout_norm_bwd(y, g, w, dout, eps: float = 0.0):
    """Gradients of readout_norm for dL/dout = dout: p = w (.) dout,
    r = sum_d p o, do = s p - r s^3 o / d, then dy = do (.) g, dg = do (.) y
    and dw = sum over (b, t) of dout (.) o s.  Returns dict(dy, dg, dw)."""
    y, g, w, dout = map(_f64, (y, g, w, dout))
    o = y * g
    d = o.shape[2] * o.shape[3]
    s = 1.0 / np.sqrt((o * o).sum(axis=(2, 3)) / d + eps)[:, :, None, None]
    p = w[None, None] * dout
    r = (p * o).sum(axis=(2, 3))[:, :, None, None]
    do = s * p - r * s ** 3 * o / d
    return {"dy": do * g, "dg": do * y, "dw": (dout * o * s).sum(axis=(0, 1))}


def fwd_norm(q, k, v, f, W, w_r, g, w_norm, eps: float = 0.0, H0=None):
    """Forward pass followed by the readout epilogue: dict(y, out, rstd, HT)."""
    r = fwd(q, k, v, f, W, w_r, H0)
    r.update(readout_norm(r["y"], g, w_norm, eps))
    return r


def bwd_norm(q, k, v, f, W, w_r, g, w_norm, dout, eps: float = 0.0, H0=None, dHT=None):
    """Backward pass through the readout epilogue and the recurrence:
    dict(dq, dk, dv, df, dW, dw_r, dH0, dg, dw_norm) (float64)."""
    y = fwd(q, k, v, f, W, w_r, H0)["y"]
    n = readout_norm_bwd(y, g, w_norm, dout, eps)
    r = bwd(q, k, v, f, W, w_r, n["dy"], H0, dHT)
    r["dg"], r["dw_norm"] = n["dg"], n["dw"]
    return r
