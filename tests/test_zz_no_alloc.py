"""m2rnn_bwd_noalloc: the backward pass for callers that cannot allocate.

Callers that must not call cudaMalloc while they run the backward pass (a
frozen or exhausted memory pool, an allocator that must not be re-entered,
a runtime with only pre-registered buffers) use this entry point: it
recomputes the checkpoints into a buffer compiled into the library instead
of a caller workspace.  These tests call it through the C ABI twice in a row
and compare with m2rnn_bwd (ckpt = NULL, caller workspace): the two run the
same kernels on the same recomputed checkpoints, so they may differ only by
the order of the atomic head and batch sums (relative L2 <= 1e-5 per
gradient).  One more case checks it against the fp64 oracle within the
gradient tolerance of the other parity tests (relative L2 <= 1e-2).  The
file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL_SAME_PATH = 1e-5  # same kernels, same checkpoints: atomics' order only
TOL_ORACLE = 1e-2
NAMES = ("dq", "dk", "dv", "df", "dW", "dw_r", "dH0")


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn as m
    return m


def _rel(a, r):
    a, r = a.detach().cpu().double().numpy(), r.detach().cpu().double().numpy()
    den = np.linalg.norm(r)
    return np.linalg.norm(a - r) / den if den > 0 else np.linalg.norm(a)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_bwd_twice(m2rnn, dtype):
    B, T, N, K, V, C = 3, 300, 8, 64, 16, 64
    x = make_inputs(B, T, N, K, V, dtype, 123, with_dy=True)
    g = {n: t.cuda() for n, t in x.items()}
    gen = torch.Generator().manual_seed(5)
    H0 = (torch.rand(B, N, K, V, generator=gen) - 0.5).cuda()
    dHT = torch.randn(B, N, K, V, generator=gen).cuda()
    ref = m2rnn.bwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"], H0=H0, dHT=dHT,
                    ckpt=None, ckpt_every=C, want_dH0=True)
    torch.cuda.synchronize()
    for call in range(2):  # the shared buffer keeps the previous call's contents
        got = m2rnn.bwd_noalloc(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"], H0=H0,
                                dHT=dHT, ckpt_every=C, want_dH0=True)
        torch.cuda.synchronize()
        st, detail = m2rnn.device_status(clear=True)
        assert st == 0, (st, detail)
        errs = {n: _rel(got[n], ref[n]) for n in NAMES}
        assert max(errs.values()) <= TOL_SAME_PATH, (call, errs)


def test_noalloc_matches_oracle(m2rnn, oracle_mod):
    """Against the fp64 oracle, whole sequence (48 steps, checkpoints every
    16), with H0 and dH_T given."""
    B, T, N, K, V, C = 2, 48, 4, 64, 16, 16
    x = make_inputs(B, T, N, K, V, "bf16", 4343, with_dy=True)
    g = {n: t.cuda() for n, t in x.items()}
    gen = torch.Generator().manual_seed(9)
    H0 = torch.rand(B, N, K, V, generator=gen) - 0.5
    dHT = torch.randn(B, N, K, V, generator=gen)
    got = m2rnn.bwd_noalloc(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"],
                            H0=H0.cuda(), dHT=dHT.cuda(), ckpt_every=C, want_dH0=True)
    torch.cuda.synchronize()
    st, detail = m2rnn.device_status(clear=True)
    assert st == 0, (st, detail)
    ref = oracle_mod.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"], H0=H0,
                         dHT=dHT)
    errs = {}
    for n in NAMES:
        a, r = got[n].detach().cpu().double().numpy(), ref[n]
        errs[n] = np.linalg.norm(a - r) / max(np.linalg.norm(r), 1e-30)
    assert max(errs.values()) <= TOL_ORACLE, errs


def test_noalloc_refuses_oversized_problem(m2rnn):
    """Checkpoints needing more than the built-in buffer are refused with
    M2RNN_ERR_WORKSPACE before any device work; a bad shape or a missing
    checkpoint interval with M2RNN_ERR_INVALID_ARG or
    M2RNN_ERR_UNSUPPORTED_SHAPE, also before any device work."""
    s = m2rnn.Shape(64, 4096, 32, 64, 16, 1, 64)  # 512 MiB of checkpoints
    p = ctypes.c_void_p(16)
    rc = m2rnn.lib().m2rnn_bwd_noalloc(ctypes.byref(s), *([p] * 16), None)
    assert rc == -5
    for bad, want in ((m2rnn.Shape(2, 8, 3, 48, 16, 1, 4), -2),   # K = 48
                      (m2rnn.Shape(2, 8, 3, 64, 16, 1, 0), -1),   # no checkpoint interval
                      (m2rnn.Shape(0, 8, 3, 64, 16, 1, 4), -1)):  # B = 0
        assert m2rnn.lib().m2rnn_bwd_noalloc(ctypes.byref(bad), *([p] * 16), None) == want
