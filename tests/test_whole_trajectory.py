"""Whole-trajectory parity: the GPU forward and backward on the benchmarked
workloads against the fp64 oracle run over the whole sequence, with no
restarts, up to each head's divergence horizon.

The horizons come from tests/golden/conditioning.json (written from the
oracle alone by tests/golden/make_conditioning.py and pinned by
tests/test_conditioning.py).  They mark where the oracle departs from its own
trajectory when the product H W is perturbed by the bf16 unit roundoff, the
size of the rounding the bf16-operand path applies to it at every step:
  * y of head (b, n) is compared at every step t < h_y[b][n] = min(h_w5e3,
    h_amp10)[b][n]: the oracle itself moves by at most 5e-3 there (a quarter
    of the 2e-2 bound) under that perturbation, and its amplification of a
    1e-7 input perturbation stays below 10 (one random perturbation of W can
    miss a window that the input perturbation shows); H_T of every head with
    no window (h_y = T) is compared too;
  * the gradients of the loss restricted to t < h_w2e3[b][n] (dy zeroed from
    the horizon on, so no head's backward crosses its window) are compared
    whole at the fwd+bwd workloads' full size and launch (checkpoints every
    64 steps), relative L2 <= max(1e-2, 2 sens_w) per tensor, sens_w being
    the record's relative change of that gradient under the unit-roundoff
    perturbation of W (twice it: the change under one bf16 ulp, the
    per-draw bound of the other backward tests, to first order);
  * the readout epilogue (x g_t, RMSNorm over a token's N V features): its
    recurrence has the ungated fwd+bwd workload's inputs and horizons; y is
    compared as above and out at every token all of whose heads are inside
    their horizon (the norm couples a token's heads).
On these workloads most heads have no window, so most comparisons span the
whole sequence.  Steps past a horizon are covered by the per-interval tests
in test_fwd_parity.py and test_bwd_parity.py.
"""
import json
import os
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_conditioning as mc  # noqa: E402

from non_linear_matrix_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

REC = json.load(open(os.path.join(HERE, "golden", "conditioning.json")))
YTOL = {"f32": 2e-3, "bf16": 2e-2}
GTOL = 1e-2


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn as m
    return m


def _status_ok(m2rnn):
    st, de = m2rnn.device_status(clear=True)
    assert st == 0, (st, de)


@pytest.mark.parametrize("name", sorted(mc.FORWARD))
def test_forward_whole_trajectory(m2rnn, oracle_mod, name):
    w = WORKLOADS[name]
    r = REC["forward"][name]
    x = workload_inputs(w, with_dy=False)
    g = {n: t.cuda() for n, t in x.items()}
    if w.gated:
        y, HT, _ = m2rnn.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                                   g["w_r"])
    else:
        y, HT, _ = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    bs = r["batch_items"]
    xs = {n: (t[bs] if n in ("q", "k", "v", "f", "a") else t) for n, t in x.items()}
    if w.gated:
        ref = oracle_mod.fwd_gated(xs["q"], xs["k"], xs["v"], xs["a"], xs["alpha"], xs["beta"],
                                   xs["W"], xs["w_r"])
    else:
        ref = oracle_mod.fwd(xs["q"], xs["k"], xs["v"], xs["f"], xs["W"], xs["w_r"])
    yg = y[bs].float().cpu().double().numpy()
    e = np.abs(yg - ref["y"]).max(axis=3)                 # [B', T, N]
    h = np.minimum(np.asarray(r["h_w5e3"]), np.asarray(r["h_amp10"]))
    inside = np.arange(w.T)[None, :, None] < h[:, None, :]
    worst_y = float(np.where(inside, e, 0.0).max())
    whole = h == w.T
    eh = np.abs(HT[bs].cpu().double().numpy() - ref["HT"]).max(axis=(2, 3))
    worst_h = float(eh[whole].max()) if whole.any() else 0.0
    print(name, f"steps compared {inside.mean():.3f}, heads whole {whole.mean():.3f}, "
          f"max |y - y_ref| {worst_y:.2e}, max |H_T - H_T_ref| {worst_h:.2e}")
    assert worst_y <= YTOL[w.dtype], (name, worst_y)
    assert worst_h <= YTOL[w.dtype], (name, worst_h)
    assert whole.mean() >= 0.5, name


@pytest.mark.parametrize("name,key", [(mc.GRADIENT, "gradient"),
                                      (mc.GRADIENT_GATED, "gradient_gated")])
def test_backward_whole_trajectory(m2rnn, oracle_mod, name, key):
    """B=8, T=4096, N=32, checkpoints every 64 steps, f given or from the
    fused gate: every gradient of the horizon-restricted loss, whole
    sequence, against the oracle."""
    w = WORKLOADS[name]
    h = REC["forward"][name]["h_w2e3"]
    sens_w = REC[key]["sens_w"]
    x = workload_inputs(w)
    mask = torch.from_numpy(mc.horizon_mask(h, w.T))[..., None]
    x["dy"] = (x["dy"].double() * mask).to(x["dy"].dtype)  # exact: kept values or zeros
    g = {n: t.cuda() for n, t in x.items()}
    C = w.ckpt_every
    if w.gated:
        gate = (g["a"], g["alpha"], g["beta"])
        _, _, ck = m2rnn.fwd_gated(g["q"], g["k"], g["v"], *gate, g["W"], g["w_r"], ckpt_every=C)
        gr = m2rnn.bwd_gated(g["q"], g["k"], g["v"], *gate, g["W"], g["w_r"], g["dy"], ckpt=ck,
                             ckpt_every=C, want_dH0=True)
        ref = oracle_mod.bwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"],
                                   x["w_r"], x["dy"])
        names = ("dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r", "dH0")
    else:
        _, _, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=C)
        gr = m2rnn.bwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"], ckpt=ck,
                       ckpt_every=C, want_dH0=True)
        ref = oracle_mod.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"])
        names = ("dq", "dk", "dv", "df", "dW", "dw_r", "dH0")
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    errs, bad = {}, {}
    for n in names:
        a, rr = gr[n].cpu().double().numpy(), ref[n]
        errs[n] = float(np.linalg.norm(a - rr) / max(np.linalg.norm(rr), 1e-30))
        bound = max(GTOL, 2.0 * sens_w[n])
        if errs[n] > bound:
            bad[n] = (errs[n], bound)
    print(name, "restricted-loss gradients, steps kept", float(mask.mean()), errs)
    assert not bad, (bad, errs)


def test_readout_epilogue_whole_trajectory(m2rnn, oracle_mod):
    """The readout epilogue's workload (B=8, T=4096, N=32): y per head up to
    its horizon, the token statistic rstd (relative, y's bound) at every
    token whose heads are all inside theirs, and out at every token against
    the oracle's epilogue applied to the GPU's own y (elementwise within
    2^-7 of |out|: out divides by the token's RMS, which multiplies y's
    absolute error by w g rstd, so the epilogue is checked on its own)."""
    w = WORKLOADS["fwdbwd_norm_bf16_b8_t4096_n32"]
    r = REC["forward"][mc.GRADIENT]
    x = workload_inputs(w, with_dy=False)
    plain = workload_inputs(WORKLOADS[mc.GRADIENT], with_dy=False)
    for n in ("q", "k", "v", "f", "W", "w_r"):  # the same recurrence as the ungated workload
        assert torch.equal(x[n], plain[n]), n
    g = {n: t.cuda() for n, t in x.items()}
    eps = 1e-6
    res = m2rnn.fwd_norm(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["g"], g["w_norm"],
                         eps)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    ref = oracle_mod.fwd_norm(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["g"],
                              x["w_norm"], eps)
    yg = res["y"].float().cpu().double().numpy()
    h = np.minimum(np.asarray(r["h_w5e3"]), np.asarray(r["h_amp10"]))  # [B, N]
    inside = np.arange(w.T)[None, :, None] < h[:, None, :]
    worst_y = float(np.where(inside, np.abs(yg - ref["y"]).max(axis=3), 0.0).max())
    tok = inside.all(axis=2)                                           # [B, T]
    er = np.abs(res["rstd"].cpu().double().numpy() / ref["rstd"] - 1)
    worst_r = float(np.where(tok, er, 0.0).max())
    epi = oracle_mod.readout_norm(yg, x["g"], x["w_norm"], eps)
    og = res["out"].float().cpu().double().numpy()
    worst_o = float((np.abs(og - epi["out"]) / (np.abs(epi["out"]) + 1e-6)).max())
    print("norm: tokens inside", tok.mean(), "max |y - y_ref|", worst_y, "rstd rel", worst_r,
          "out rel (epilogue on the GPU's y)", worst_o)
    assert worst_y <= YTOL[w.dtype], worst_y
    assert worst_r <= YTOL[w.dtype], worst_r
    assert worst_o <= 2.0 ** -7, worst_o
    assert tok.any()  # (few tokens have all 32 heads before their windows: 2.5 % here)
