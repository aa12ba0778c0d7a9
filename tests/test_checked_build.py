"""The checked build (libm2rnn_check.so, -DM2RNN_CHECK=1): every global
index a kernel computes is tested against the extent the call's shape gives
its array, and a violation is recorded in the device status word
(M2RNN_ERR_BOUNDS) instead of being performed.  Every entry point runs here
on ragged shapes (T not a multiple of the ring chunk, the checkpoint interval
or the sub-interval; odd head counts; K = 16 and 128; V = 32; grouped q/k;
the whole-wave plus tail forward; both backward kernels at 1, 2 and 4 warps
per CTA; recomputed checkpoints) and must leave the status clean.  Its
results must equal the normal build's: bit for bit where outputs are stored,
within the rounding of a different summation order where they are
accumulated with atomics (dq, dk, dW, dw_r and cross-slice dv, df)."""

import pytest
import torch

from non_linear_matrix_gb300.inputs import decode_state, make_inputs

pytestmark = pytest.mark.gpu

ATOMIC_REL = 1e-5


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import build as b
    b.build(checked=True)
    from non_linear_matrix_gb300 import m2rnn as m
    m.use_library("normal")
    yield m
    m.use_library("normal")


def _both(m2rnn, run):
    """run() under the normal and the checked build; the checked build's
    status word must stay clean."""
    m2rnn.use_library("normal")
    ref = run()
    torch.cuda.synchronize()
    m2rnn.use_library("checked")
    try:
        assert m2rnn.lib().m2rnn_checked() == 1
        m2rnn.device_status(clear=True)
        got = run()
        torch.cuda.synchronize()
        st, de = m2rnn.device_status(clear=True)
    finally:
        m2rnn.use_library("normal")
    assert (st, de) == (0, 0), (st, de)
    return ref, got


def _same(ref, got, atomic=()):
    for n, r in ref.items():
        if r is None:
            continue
        g = got[n]
        if n in atomic:
            err = (g.double() - r.double()).norm() / r.double().norm().clamp_min(1e-30)
            assert err <= ATOMIC_REL, (n, float(err))
        else:
            assert torch.equal(g, r), n


def _dev(x):
    return {n: t.cuda() for n, t in x.items()}


FWD_BWD = [
    (3, 77, 5, 64, 16, "bf16", 24, 1),
    (2, 41, 3, 16, 16, "f32", 16, 1),
    (2, 53, 4, 128, 16, "bf16", 64, 2),
    (2, 35, 3, 64, 32, "bf16", 8, 1),
    (41, 40, 32, 64, 16, "bf16", 16, 4),  # whole-wave + tail forward, serial backward
]


@pytest.mark.parametrize("B,T,N,K,V,dtype,C,Nq", FWD_BWD)
def test_fwd_bwd_checked(m2rnn, B, T, N, K, V, dtype, C, Nq):
    g = _dev(make_inputs(B, T, N, K, V, dtype, 300 + T, with_dy=True, groups=Nq))
    gen = torch.Generator().manual_seed(T)
    H0 = (torch.rand(B, N, K, V, generator=gen) - 0.5).cuda()
    dHT = torch.randn(B, N, K, V, generator=gen).cuda()
    args = (g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])

    def fwd():
        y, HT, ck = m2rnn.fwd(*args, H0, ckpt_every=C)
        return {"y": y, "HT": HT, "ckpt": ck}

    ref, got = _both(m2rnn, fwd)
    _same(ref, got)
    ck = ref["ckpt"]
    for given in (True, False):
        def bwd():
            return m2rnn.bwd(*args, g["dy"], H0=H0, ckpt=ck if given else None, dHT=dHT,
                             ckpt_every=C, want_dH0=True, want_dckpt=True)
        r, q = _both(m2rnn, bwd)
        _same(r, q, atomic=("dq", "dk", "dW", "dw_r", "dv", "df"))


@pytest.mark.parametrize("kernel,wpc", [("0", "1"), ("0", "2"), ("0", "4"), ("1", "1"),
                                        ("1", "2"), ("1", "4")])
def test_bwd_kernels_checked(m2rnn, monkeypatch, kernel, wpc):
    monkeypatch.setenv("M2RNN_BWD_KERNEL", kernel)
    monkeypatch.setenv("M2RNN_BWD_WPC", wpc)
    B, T, N, C = 2, 70, 3, 32
    g = _dev(make_inputs(B, T, N, 64, 16, "bf16", 71, with_dy=True, groups=1))
    args = (g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
    _, _, ck = m2rnn.fwd(*args, ckpt_every=C)

    def bwd():
        return m2rnn.bwd(*args, g["dy"], ckpt=ck, ckpt_every=C, want_dH0=True, want_dckpt=True)

    r, q = _both(m2rnn, bwd)
    _same(r, q, atomic=("dq", "dk", "dW", "dw_r", "dv", "df"))


@pytest.mark.parametrize("G,gated", [("4", False), ("5", True)])
def test_wave_kernel_checked(m2rnn, monkeypatch, G, gated):
    """The one-wave forward kernel (CTAs across two batch items), plain and
    with the fused gate, under both builds."""
    monkeypatch.setenv("M2RNN_FWD_WAVE", "1")
    monkeypatch.setenv("M2RNN_FWD_WAVE_G", G)
    g = _dev(make_inputs(5, 77, 6, 64, 16, "bf16", 77, gated=gated))
    H0 = (torch.rand(5, 6, 64, 16, generator=torch.Generator().manual_seed(2)) - 0.5).cuda()

    def fwd():
        if gated:
            y, HT, ck = m2rnn.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"],
                                        g["W"], g["w_r"], H0, ckpt_every=24)
        else:
            y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H0,
                                  ckpt_every=24)
        return {"y": y, "HT": HT, "ckpt": ck}

    ref, got = _both(m2rnn, fwd)
    _same(ref, got)


def test_gated_norm_noalloc_checked(m2rnn):
    B, T, N, K, V, C = 3, 45, 6, 64, 16, 16
    g = _dev(make_inputs(B, T, N, K, V, "bf16", 5, with_dy=True, gated=True, norm=True))
    gate = (g["a"], g["alpha"], g["beta"])

    def fwd_norm():
        return m2rnn.fwd_norm(g["q"], g["k"], g["v"], None, g["W"], g["w_r"], g["g"],
                              g["w_norm"], 1e-6, gate=gate, ckpt_every=C)

    r, q = _both(m2rnn, fwd_norm)
    _same(r, q, atomic=("rstd", "out"))  # rstd sums the heads' squares with atomics
    y, rstd, ck = r["y"], r["rstd"], r["ckpt"]

    def bwd_norm():
        return m2rnn.bwd_norm(g["q"], g["k"], g["v"], None, g["W"], g["w_r"], g["g"],
                              g["w_norm"], y, rstd, g["dy"], ckpt=ck, gate=gate, ckpt_every=C,
                              want_dH0=True)

    r2, q2 = _both(m2rnn, bwd_norm)
    _same(r2, q2, atomic=tuple(r2))

    def bwd_gated():
        return m2rnn.bwd_gated(g["q"], g["k"], g["v"], *gate, g["W"], g["w_r"], g["dy"], ckpt=ck,
                               ckpt_every=C)

    r3, q3 = _both(m2rnn, bwd_gated)
    _same(r3, q3, atomic=tuple(r3))

    def noalloc():
        return m2rnn.bwd_noalloc(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"],
                                 ckpt_every=C, want_dH0=True)

    r4, q4 = _both(m2rnn, noalloc)
    _same(r4, q4, atomic=tuple(r4))


@pytest.mark.parametrize("K,V,dtype,Nq,gated", [(64, 16, "bf16", 1, False), (128, 32, "f32", 1, False),
                                                (16, 16, "bf16", 5, False), (64, 16, "bf16", 1, True)])
def test_decode_checked(m2rnn, K, V, dtype, Nq, gated):
    B, N = 7, 5
    x = make_inputs(B, 1, N, K, V, dtype, 23, groups=Nq, gated=gated)
    g = {n: (t[:, 0].contiguous() if n in ("q", "k", "v", "f", "a") else t).cuda()
         for n, t in x.items()}
    H = decode_state(B, N, K, V, 3).cuda()

    def dec():
        if gated:
            y, Ho = m2rnn.decode_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"],
                                       g["W"], g["w_r"], H)
        else:
            y, Ho = m2rnn.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H)
        return {"y": y, "H": Ho}

    r, q = _both(m2rnn, dec)
    _same(r, q)
