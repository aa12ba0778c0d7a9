"""Readout epilogue (frames "Most of the block can be computed before
recurrence" and "Backup: RMSNormTP synchronizes per-token statistics"):
out = w_norm (.) (y (.) g) rstd over a token's N*V features, fused into the
forward kernel's epilogue (sum of squares) plus a scaling kernel, and its
backward (dg, dw_norm and dL/dy feeding the recurrence's backward).  GPU
results through the C ABI against the oracle's readout_norm / fwd_norm /
bwd_norm on the same seeded inputs.

Tolerances: y and H_T as the forward's (max |.| 2e-3 fp32 operands, 2e-2
bf16).  The epilogue is checked on the GPU's own y, since it divides by the
token's RMS and so multiplies y's absolute error by w g rstd (about 5 at
these distributions): out elementwise within 2^-7 (bf16) or 1e-5 (fp32)
of |out|, rstd within 2^-8 / 1e-5 relative.  The bf16 bounds: the kernel
forms rstd from the fp32 y before y is rounded to bf16 (half an ulp, 2^-8
relative), which moves each o^2 by at most 2^-7 and rstd by at most 2^-8;
out adds its own rounding (2^-8).  Gradients relative L2 <= 1e-2.  Long sequences: the recurrence
per checkpoint interval as in the other parity tests.
"""
import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-2}
OUT_RTOL = {"f32": 1e-5, "bf16": 2.0 ** -7}
RSTD_RTOL = {"f32": 1e-5, "bf16": 2.0 ** -8}
GTOL = 1e-2


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn as m
    return m


def _dev(x):
    return {n: t.cuda() for n, t in x.items()}


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _rel(a, r):
    a = _np(a) if hasattr(a, "detach") else a
    den = np.linalg.norm(r)
    return np.linalg.norm(a - r) / den if den > 0 else np.linalg.norm(a)


def _status_ok(m2rnn):
    st, de = m2rnn.device_status(clear=True)
    assert st == 0, (st, de)


def _fwd(m2rnn, g, eps, C=0, H0=None, gated=False):
    gate = (g["a"], g["alpha"], g["beta"]) if gated else None
    return m2rnn.fwd_norm(g["q"], g["k"], g["v"], None if gated else g["f"], g["W"], g["w_r"],
                          g["g"], g["w_norm"], eps, H0, gate=gate, ckpt_every=C)


def _check_epilogue(oracle_mod, x, r, eps, dtype, label):
    """out and rstd against the oracle's epilogue applied to the GPU's y."""
    ref = oracle_mod.readout_norm(_np(r["y"]), x["g"], x["w_norm"], eps)
    eo = (np.abs(_np(r["out"]) - ref["out"]) / (np.abs(ref["out"]) + 1e-6)).max()
    es = np.abs(_np(r["rstd"]) / ref["rstd"] - 1).max()
    assert eo <= OUT_RTOL[dtype] and es <= RSTD_RTOL[dtype], (label, eo, es)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,V", [(4, 16), (32, 16), (8, 32)])
@pytest.mark.parametrize("eps", [0.0, 1e-5])
def test_forward_norm_whole(m2rnn, oracle_mod, dtype, N, V, eps):
    """y and H_T against fwd_norm of the oracle (whole trajectory, T = 40),
    rstd within the y tolerance (relative), out and rstd on the GPU's y."""
    x = make_inputs(2, 40, N, 64, V, dtype, 1100 + N + V, norm=True)
    r = _fwd(m2rnn, _dev(x), eps)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    ref = oracle_mod.fwd_norm(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["g"],
                              x["w_norm"], eps)
    tol = TOL[dtype]
    for n in ("y", "HT"):
        assert np.abs(_np(r[n]) - ref[n]).max() <= tol, n
    assert np.abs(_np(r["rstd"]) / ref["rstd"] - 1).max() <= tol
    _check_epilogue(oracle_mod, x, r, eps, dtype, "whole")


def test_forward_norm_large(m2rnn, oracle_mod):
    """B=64, T=512, N=32: whole-wave plus tail launches (both add their
    heads' sums of squares); the epilogue on the GPU's own y for every
    token."""
    x = make_inputs(64, 512, 32, 64, 16, "bf16", 1177, norm=True)
    r = _fwd(m2rnn, _dev(x), 1e-6)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    _check_epilogue(oracle_mod, x, r, 1e-6, "bf16", "B64 T512")


def _bwd_restart(m2rnn, oracle_mod, x, C, dtype, gated=False, give_ckpt=True, label=""):
    """GPU fwd_norm + bwd_norm; the epilogue's gradients against the
    oracle's readout_norm_bwd on the GPU's y, the recurrence's against the
    oracle restarted per checkpoint interval with that dL/dy."""
    g = _dev(x)
    r = _fwd(m2rnn, g, 1e-6, C, gated=gated)
    gate = (g["a"], g["alpha"], g["beta"]) if gated else None
    gr = m2rnn.bwd_norm(g["q"], g["k"], g["v"], None if gated else g["f"], g["W"], g["w_r"],
                        g["g"], g["w_norm"], r["y"], r["rstd"], g["dy"],
                        ckpt=r["ckpt"] if give_ckpt else None, gate=gate, ckpt_every=C,
                        want_dH0=True, want_dckpt=True)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    yg = _np(r["y"])
    nb = oracle_mod.readout_norm_bwd(yg, x["g"], x["w_norm"], x["dy"], 1e-6)
    errs = {"dg": _rel(gr["dg"], nb["dg"]), "dw_norm": _rel(gr["dw_norm"], nb["dw"])}
    q, k, v = x["q"], x["k"], x["v"]
    B, T, K = q.shape[0], q.shape[1], q.shape[-1]
    N, V = v.shape[2], v.shape[3]
    fsrc = x["a"] if gated else x["f"]
    nck = -(-T // C)
    ckn, dckn = _np(r["ckpt"]), _np(gr["dckpt"])
    nxt = np.concatenate([dckn[:, :, 1:], np.zeros((B, N, 1, K, V))], axis=2)
    names = ("dq", "dk", "dv", "da" if gated else "df", "dW", "dw_r")
    ref = {n: np.zeros(tuple(gr[n].shape)) for n in names}
    for c0, c1, L in ((0, T // C, C), (T // C, nck, T - (T // C) * C)):
        if c1 <= c0:
            continue
        t0, t1, nbk = c0 * C, c0 * C + (c1 - c0) * L, c1 - c0

        def split(z):
            z = np.asarray(z if not hasattr(z, "detach") else _np(z))[:, t0:t1]
            return z.reshape(B * nbk, L, *z.shape[2:])

        def per(z):
            return np.ascontiguousarray(np.moveaxis(z[:, :, c0:c1], 2, 1)).reshape(B * nbk, N, K, V)
        if gated:
            o = oracle_mod.bwd_gated(split(q), split(k), split(v), split(fsrc), x["alpha"],
                                     x["beta"], x["W"], x["w_r"], split(nb["dy"]), H0=per(ckn),
                                     dHT=per(nxt))
        else:
            o = oracle_mod.bwd(split(q), split(k), split(v), split(fsrc), x["W"], x["w_r"],
                               split(nb["dy"]), H0=per(ckn), dHT=per(nxt))
        for n in names:
            if n in ("dW", "dw_r"):
                ref[n] += o[n]
            else:
                ref[n][:, t0:t1] = o[n].reshape(B, nbk * L, *o[n].shape[2:])
    errs.update({n: _rel(gr[n], ref[n]) for n in names})
    assert max(errs.values()) <= GTOL, (label, errs)
    return errs


@pytest.mark.parametrize("kernel", ["0", "1"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_norm(m2rnn, oracle_mod, monkeypatch, kernel, dtype):
    """Both backward kernels, both dtypes, ragged last interval."""
    monkeypatch.setenv("M2RNN_BWD_KERNEL", kernel)
    x = make_inputs(2, 100, 4, 64, 16, dtype, 1200, with_dy=True, norm=True)
    _bwd_restart(m2rnn, oracle_mod, x, 24, dtype, label=f"k{kernel} {dtype}")


@pytest.mark.parametrize("N", [32, 40])
def test_backward_norm_row_widths(m2rnn, oracle_mod, N):
    """A token's d = N V features on either side of the normalisation
    backward's switch: d = 512 (the register kernel, two full 8-column
    groups per lane) and d = 640 (the kernel with dw in shared memory)."""
    x = make_inputs(2, 40, N, 64, 16, "bf16", 1250 + N, with_dy=True, norm=True)
    _bwd_restart(m2rnn, oracle_mod, x, 16, "bf16", label=f"d={16 * N}")


def test_backward_norm_gated_grouped_recomputed(m2rnn, oracle_mod):
    """The epilogue with the fused gate, 2 query/key groups and checkpoints
    recomputed into the workspace (after the epilogue's dL/dy)."""
    x = make_inputs(2, 90, 8, 64, 16, "bf16", 1210, with_dy=True, norm=True, gated=True,
                    groups=2)
    _bwd_restart(m2rnn, oracle_mod, x, 32, "bf16", gated=True, give_ckpt=False, label="gated")


@pytest.mark.parametrize("K,V,dtype,Nq", [(16, 16, "f32", 1), (32, 16, "bf16", 2),
                                          (128, 16, "bf16", 1), (64, 32, "f32", 2),
                                          (128, 32, "bf16", 1)])
def test_norm_gated_shape_matrix(m2rnn, oracle_mod, K, V, dtype, Nq):
    """The epilogue with the fused gate at the other K, V and dtype
    combinations, which run other kernel instances (1-, 2- and 8-slice
    heads; the serial backward at V = 32; fp32 operands), with and without
    query/key groups: out and rstd on the GPU's y, every gradient per
    16-step checkpoint interval, ragged last interval."""
    x = make_inputs(2, 50, 4, K, V, dtype, 1300 + K + V, with_dy=True, norm=True, gated=True,
                    groups=Nq)
    r = _fwd(m2rnn, _dev(x), 1e-6, 16, gated=True)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    _check_epilogue(oracle_mod, x, r, 1e-6, dtype, f"K{K} V{V} {dtype}")
    _bwd_restart(m2rnn, oracle_mod, x, 16, dtype, gated=True, label=f"K{K} V{V} {dtype} Nq{Nq}")


def test_backward_norm_whole_short(m2rnn, oracle_mod):
    """Whole-sequence gradients of the block against bwd_norm of the oracle."""
    for dtype in ("bf16", "f32"):
        x = make_inputs(2, 24, 4, 64, 16, dtype, 1220, with_dy=True, norm=True)
        g = _dev(x)
        r = _fwd(m2rnn, g, 0.0, 8)
        gr = m2rnn.bwd_norm(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["g"],
                            g["w_norm"], r["y"], r["rstd"], g["dy"], ckpt=r["ckpt"], ckpt_every=8)
        torch.cuda.synchronize()
        _status_ok(m2rnn)
        ref = oracle_mod.bwd_norm(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["g"],
                                  x["w_norm"], x["dy"])
        errs = {n: _rel(gr[n], ref[n]) for n in
                ("dq", "dk", "dv", "df", "dW", "dw_r", "dg", "dw_norm")}
        assert max(errs.values()) <= GTOL, (dtype, errs)


def test_norm_workload_interval_parity(m2rnn, oracle_mod):
    """The readout-epilogue fwd+bwd workload bench.py times (B=8, T=4096,
    N=32, C=64), on its own inputs and in its launch configuration: the
    epilogue on every token and every gradient per 64-step interval."""
    x = workload_inputs(WORKLOADS["fwdbwd_norm_bf16_b8_t4096_n32"])
    _bwd_restart(m2rnn, oracle_mod, x, 64, "bf16", label="norm b8 t4096")
