"""Fused input gate (frame "The gate preserves a direct path through time",
Eq. 13): f = exp(-alpha softplus(a + beta)) evaluated inside the forward and
backward kernels, with the chain rule to a, alpha and beta applied in the
backward kernel.  GPU results through the C ABI against the oracle's gated
functions on the same seeded inputs.

Tolerances are those of the ungated path: max |.| <= 2e-3 (fp32 operands)
or 2e-2 (bf16 operands) on y, H_T and checkpoints; relative L2 <= 1e-2 per
gradient tensor, dalpha and dbeta included.  dalpha and dbeta are each a sum
over all B*T steps of a signed per-step term that cancels to a small part of
its terms' absolute mass (tests/golden/conditioning.json, "gate_cancel"),
which magnifies bf16-level step errors; where a draw's own sensitivity to a
one-ulp perturbation of W exceeds 1e-2, that sensitivity is the bound
(tests/test_conditioning.py pins the measurement), and the error relative to
the terms' mass, max_n |g_n - r_n| / sum_{b,t} |term_{b,t,n}| <= 1e-2, is
required as well.  Sequences longer than a few intervals are compared per
checkpoint interval (the oracle restarts from the GPU's checkpoint and takes
the GPU's dckpt of the next interval as incoming gradient), for the reason
the ungated parity tests give: the recurrence is ill-conditioned over long
spans at these input distributions.
"""
import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

FTOL = {"f32": 2e-3, "bf16": 2e-2}
GTOL = 1e-2
GATE = ("a", "alpha", "beta")


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
    a = _np(a)
    den = np.linalg.norm(r)
    return np.linalg.norm(a - r) / den if den > 0 else np.linalg.norm(a)


def _status_ok(m2rnn):
    st, de = m2rnn.device_status(clear=True)
    assert st == 0, (st, de)


def _fwd(m2rnn, g, H0=None, C=0):
    return m2rnn.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                           g["w_r"], H0, ckpt_every=C)


def _fwd_restart(oracle_mod, x, y, HT, ck, C, tol, H0=None, label=""):
    """Oracle's gated forward restarted from the GPU checkpoint of every
    interval of C steps: y over the interval and the state at its end."""
    q, k, v, a = (x[n] for n in ("q", "k", "v", "a"))
    B, T, K = q.shape
    N, V = v.shape[2], v.shape[3]
    ckn, yn, HTn = _np(ck), _np(y), _np(HT)
    nck = ckn.shape[2]
    h0 = np.zeros((B, N, K, V)) if H0 is None else H0.double().numpy()
    assert np.abs(ckn[:, :, 0] - h0).max() <= 1e-6, label
    nxt_all = np.concatenate([ckn[:, :, 1:], HTn[:, :, None]], axis=2)
    worst = 0.0
    for c0, c1, L in ((0, T // C, C), (T // C, nck, T - (T // C) * C)):
        if c1 <= c0:
            continue
        t0, t1, nb = c0 * C, c0 * C + (c1 - c0) * L, c1 - c0

        def split(z):
            z = z[:, t0:t1]
            return z.reshape(B * nb, L, *z.shape[2:])

        def per(z):
            return np.ascontiguousarray(np.moveaxis(z[:, :, c0:c1], 2, 1)).reshape(B * nb, N, K, V)
        r = oracle_mod.fwd_gated(split(q), split(k), split(v), split(a), x["alpha"], x["beta"],
                                 x["W"], x["w_r"], H0=per(ckn))
        worst = max(worst, np.abs(split(yn) - r["y"]).max(), np.abs(per(nxt_all) - r["HT"]).max())
    assert worst <= tol, (label, worst)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,V", [(64, 16), (32, 16), (64, 32), (128, 16)])
@pytest.mark.parametrize("T", [1, 37, 130])
def test_forward_gated(m2rnn, oracle_mod, dtype, K, V, T):
    """y, H_T and checkpoints against the oracle's gated forward with an
    initial state: the whole trajectory for T <= 37, per 16-step interval
    for T = 130.  (At T = 130 the oracle's own H_T moves by up to 0.07 when
    W is perturbed at bf16 resolution, e.g. K = 32, so whole-trajectory
    values are beyond the conditioning limit there.)"""
    B, N = 2, 4
    x = make_inputs(B, T, N, K, V, dtype, 5000 + K + V + T, gated=True)
    H0 = torch.rand(B, N, K, V, generator=torch.Generator().manual_seed(T)) - 0.5
    g = _dev(x)
    y, HT, ck = _fwd(m2rnn, g, H0.cuda(), 16)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    tol = FTOL[dtype]
    if T > 40:
        _fwd_restart(oracle_mod, x, y, HT, ck, 16, tol, H0=H0, label=f"{dtype} K{K} V{V}")
        return
    ref = oracle_mod.fwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"],
                               x["w_r"], H0=H0, want_states=True)
    assert np.abs(_np(y) - ref["y"]).max() <= tol
    assert np.abs(_np(HT) - ref["HT"]).max() <= tol
    idx = list(range(0, T, 16))
    assert np.abs(_np(ck) - ref["states"][:, :, idx]).max() <= tol


def test_forward_gated_wave_split(m2rnn, oracle_mod):
    """Enough batch items for the forward's whole-wave launch plus a tail
    launch with fewer heads per CTA: the gate input is offset per launch."""
    B, T, N = 41, 40, 32
    x = make_inputs(B, T, N, 64, 16, "bf16", 811, gated=True)
    y, HT, _ = _fwd(m2rnn, _dev(x))
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    ref = oracle_mod.fwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"],
                               x["w_r"])
    assert np.abs(_np(y) - ref["y"]).max() <= FTOL["bf16"]
    assert np.abs(_np(HT) - ref["HT"]).max() <= FTOL["bf16"]


def _gate_mass(oracle_mod, a, alpha, beta, da):
    """Per head, the absolute mass sum_{b,t} |term| of the per-step terms
    that dbeta (da itself) and dalpha (df * (-softplus f) = da * softplus /
    (alpha sigmoid)) sum, from the oracle's gate values."""
    _, sp, _, sig = oracle_mod._gate_parts(a, alpha, beta)
    return {"dbeta": np.abs(da).sum(axis=(0, 1)),
            "dalpha": np.abs(da * sp / (_np(alpha) * sig)).sum(axis=(0, 1))}


def _mass_err(g, r, mass):
    return float(np.max(np.abs(_np(g) - r) / np.maximum(mass, 1e-30)))


def _gated_ref(oracle_mod, x, ckn, dckn, C, dHT=None, W=None):
    """The oracle's gated backward restarted every interval of C steps from
    the GPU's checkpoint, with the GPU's gradient of the next checkpoint as
    incoming state gradient (W replaces x["W"] in sensitivity runs).
    Returns (reference gradients, per-head absolute mass of the dalpha and
    dbeta terms)."""
    q, k, v, a, dy = (x[n] for n in ("q", "k", "v", "a", "dy"))
    W = x["W"] if W is None else W
    B, T = q.shape[0], q.shape[1]  # q: [B,T,K] or grouped [B,T,Nq,K]
    N, V, K = v.shape[2], v.shape[3], ckn.shape[3]
    nck = -(-T // C)
    last = np.zeros((B, N, 1, K, V)) if dHT is None else dHT.double().numpy()[:, :, None]
    nxt = np.concatenate([dckn[:, :, 1:], last], axis=2)
    ref = {"dq": np.zeros(q.shape), "dk": np.zeros(q.shape), "dv": np.zeros((B, T, N, V)),
           "da": np.zeros((B, T, N)), "dalpha": np.zeros(N), "dbeta": np.zeros(N),
           "dW": np.zeros((N, V, V)), "dw_r": np.zeros((N, V)),
           "dckpt": np.zeros((B, N, nck, K, V))}
    mass = {"dalpha": np.zeros(N), "dbeta": np.zeros(N)}
    for c0, c1, L in ((0, T // C, C), (T // C, nck, T - (T // C) * C)):
        if c1 <= c0:
            continue
        t0, t1, nb = c0 * C, c0 * C + (c1 - c0) * L, c1 - c0

        def split(z):
            z = z[:, t0:t1]
            return z.reshape(B * nb, L, *z.shape[2:])

        def per(z):
            return np.ascontiguousarray(np.moveaxis(z[:, :, c0:c1], 2, 1)).reshape(B * nb, N, K, V)
        r = oracle_mod.bwd_gated(split(q), split(k), split(v), split(a), x["alpha"], x["beta"],
                                 W, x["w_r"], split(dy), H0=per(ckn), dHT=per(nxt))
        ref["dq"][:, t0:t1] = r["dq"].reshape(B, nb * L, *q.shape[2:])
        ref["dk"][:, t0:t1] = r["dk"].reshape(B, nb * L, *q.shape[2:])
        ref["dv"][:, t0:t1] = r["dv"].reshape(B, nb * L, N, V)
        ref["da"][:, t0:t1] = r["da"].reshape(B, nb * L, N)
        for n in ("dalpha", "dbeta", "dW", "dw_r"):
            ref[n] += r[n]
        for n, m in _gate_mass(oracle_mod, split(a), x["alpha"], x["beta"], r["da"]).items():
            mass[n] += m
        ref["dckpt"][:, :, c0:c1] = np.moveaxis(r["dH0"].reshape(B, nb, N, K, V), 1, 2)
    ref["dH0"] = ref["dckpt"][:, :, 0]
    return ref, mass


# Relative size of the random perturbation of W that stands in for the GPU
# path's own rounding when a draw's conditioning is measured: one bf16 ulp
# (2^-8; the bf16-operand path rounds H in H W at every step by up to 2^-9
# and approximates tanh beside it); for fp32 operands, carried as bf16
# hi + lo pairs, one ulp of that pair (2^-16).
SENS_U = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -16}


def _gated_restart(m2rnn, oracle_mod, x, C, H0=None, dHT=None, give_ckpt=True, label=""):
    """GPU gated backward against the oracle restarted per checkpoint
    interval.  Every gradient, dalpha and dbeta included, must meet relative
    L2 <= max(1e-2, kappa), kappa being the oracle's own relative change of
    that gradient (same restarts) when W is perturbed elementwise by a random
    relative SENS_U; dalpha and dbeta must also meet the mass-relative bound
    max_n |g_n - r_n| / sum |terms| <= 1e-2."""
    g = _dev(x)
    H0g = None if H0 is None else H0.cuda()
    dHTg = None if dHT is None else dHT.cuda()
    _, _, ck = _fwd(m2rnn, g, H0g, C)
    gr = m2rnn.bwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"], g["w_r"],
                         g["dy"], H0=H0g, ckpt=ck if give_ckpt else None, dHT=dHTg, ckpt_every=C,
                         want_dH0=True, want_dckpt=True)
    torch.cuda.synchronize()
    _status_ok(m2rnn)
    ckn, dckn = _np(ck), _np(gr["dckpt"])
    ref, mass = _gated_ref(oracle_mod, x, ckn, dckn, C, dHT)
    W = x["W"].double().numpy()
    z = np.random.default_rng(2024).standard_normal(W.shape)
    alt, _ = _gated_ref(oracle_mod, x, ckn, dckn, C, dHT,
                        W=W * (1.0 + SENS_U[x["q"].dtype] * z))
    errs = {n: _rel(gr[n], ref[n]) for n in ref}
    kappa = {n: float(np.linalg.norm(alt[n] - ref[n]) / max(np.linalg.norm(ref[n]), 1e-30))
             for n in ref}
    bad = {n: (errs[n], kappa[n]) for n in errs if errs[n] > max(GTOL, kappa[n])}
    mass_errs = {n: _mass_err(gr[n], ref[n], mass[n]) for n in mass}
    print(label, {n: (round(errs[n], 5), round(kappa[n], 5)) for n in errs}, mass_errs)
    assert not bad and max(mass_errs.values()) <= GTOL, (label, bad, errs, kappa, mass_errs)
    return errs, kappa, mass_errs


@pytest.mark.parametrize("kernel", ["0", "1"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,C", [(1, 4), (61, 7), (130, 64)])
def test_backward_gated(m2rnn, oracle_mod, monkeypatch, kernel, dtype, T, C):
    """Both backward kernels (serial 0, pipelined 1), ragged intervals,
    H0 and dH_T given."""
    monkeypatch.setenv("M2RNN_BWD_KERNEL", kernel)
    x = make_inputs(2, T, 3, 64, 16, dtype, 7000 + T + C, with_dy=True, gated=True)
    gen = torch.Generator().manual_seed(C)
    H0 = torch.rand(2, 3, 64, 16, generator=gen) - 0.5
    dHT = torch.randn(2, 3, 64, 16, generator=gen)
    _gated_restart(m2rnn, oracle_mod, x, C, H0=H0, dHT=dHT, label=f"k{kernel} {dtype} T{T} C{C}")


@pytest.mark.parametrize("wpc", ["1", "4"])
def test_backward_gated_row_slices(m2rnn, oracle_mod, monkeypatch, wpc):
    """The pipelined kernel with K = 64 split into 4 row slices (1 warp per
    CTA): da, dalpha and dbeta are summed over slices with reductions."""
    monkeypatch.setenv("M2RNN_BWD_KERNEL", "1")
    monkeypatch.setenv("M2RNN_BWD_WPC", wpc)
    x = make_inputs(2, 150, 3, 64, 16, "bf16", 600, with_dy=True, gated=True)
    _gated_restart(m2rnn, oracle_mod, x, 32, label=f"wpc{wpc}")


def test_backward_gated_v32_recomputed(m2rnn, oracle_mod):
    """V = 32 (serial kernel) with checkpoints recomputed into the workspace."""
    x = make_inputs(2, 100, 3, 64, 32, "bf16", 901, with_dy=True, gated=True)
    _gated_restart(m2rnn, oracle_mod, x, 16, give_ckpt=False, label="v32")


def test_backward_gated_whole_short(m2rnn, oracle_mod):
    """Whole-sequence gated gradients on a short, well-conditioned sequence."""
    for dtype in ("bf16", "f32"):
        x = make_inputs(2, 24, 3, 64, 16, dtype, 4243, with_dy=True, gated=True)
        g = _dev(x)
        gr = m2rnn.bwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                             g["w_r"], g["dy"], ckpt_every=8)
        torch.cuda.synchronize()
        _status_ok(m2rnn)
        ref = oracle_mod.bwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"],
                                   x["w_r"], x["dy"])
        errs = {n: _rel(gr[n], ref[n]) for n in ("dq", "dk", "dv", "da", "dW", "dw_r")}
        mass = _gate_mass(oracle_mod, x["a"], x["alpha"], x["beta"], ref["da"])
        for n in mass:
            errs[n] = _mass_err(gr[n], ref[n], mass[n])
        assert max(errs.values()) <= GTOL, (dtype, errs)


def test_gate_alpha_zero(m2rnn):
    """alpha = 0 gives f = 1 exactly: H stays 0, y = w_r (.) v, and a and
    beta receive no gradient."""
    x = make_inputs(2, 40, 3, 64, 16, "bf16", 17, with_dy=True, gated=True)
    x["alpha"] = torch.zeros_like(x["alpha"])
    g = _dev(x)
    y, HT, _ = _fwd(m2rnn, g)
    gr = m2rnn.bwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"], g["w_r"],
                         g["dy"], ckpt_every=16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(HT) == 0
    expect = (x["w_r"].float()[None, None] * x["v"].float()).to(torch.bfloat16)
    assert torch.equal(y.cpu(), expect)
    assert torch.count_nonzero(gr["da"]) == 0 and torch.count_nonzero(gr["dbeta"]) == 0
    assert torch.count_nonzero(gr["dW"]) == 0


def test_gated_workload_interval_parity(m2rnn, oracle_mod):
    """The gated fwd+bwd workload bench.py times (B=8, T=4096, N=32, C=64),
    on its own inputs and in its launch configuration: every gradient,
    including the dalpha / dbeta sums, per 64-step interval."""
    x = workload_inputs(WORKLOADS["fwdbwd_gated_bf16_b8_t4096_n32"])
    _gated_restart(m2rnn, oracle_mod, x, 64, label="gated b8 t4096 n32")


def test_gated_zero_steps(m2rnn):
    x = _dev(make_inputs(2, 0, 3, 64, 16, "bf16", 0, with_dy=True, gated=True))
    gr = m2rnn.bwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"], x["w_r"],
                         x["dy"], ckpt_every=8)
    torch.cuda.synchronize()
    assert torch.count_nonzero(gr["dalpha"]) == 0 and torch.count_nonzero(gr["dbeta"]) == 0


def test_gated_grouped_qk(m2rnn, oracle_mod):
    """The gate together with 4 query/key groups of 2 heads."""
    x = make_inputs(2, 90, 8, 64, 16, "bf16", 990, with_dy=True, gated=True, groups=4)
    _gated_restart(m2rnn, oracle_mod, x, 32, label="gated Nq4")
