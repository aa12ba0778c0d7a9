"""m2rnn_bwd_noalloc: the backward pass for callers that cannot allocate.

Callers that must not call cudaMalloc while they run the backward pass (a
frozen or exhausted memory pool, an allocator that must not be re-entered,
a runtime with only pre-registered buffers) use this entry point: it
recomputes the checkpoints into a buffer compiled into the library instead
of a caller workspace.  These tests call it through the C ABI twice in a row
and compare with m2rnn_bwd (ckpt = NULL, caller workspace) within the
gradient tolerance the other tests use (relative L2 <= 1e-2).  The file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2
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
        assert max(errs.values()) <= TOL, (call, errs)


def test_noalloc_refuses_oversized_problem(m2rnn):
    """Checkpoints needing more than the built-in buffer are refused with
    M2RNN_ERR_WORKSPACE before any device work."""
    s = m2rnn.Shape(64, 4096, 32, 64, 16, 1, 64)  # 512 MiB of checkpoints
    p = ctypes.c_void_p(16)
    rc = m2rnn.lib().m2rnn_bwd_noalloc(ctypes.byref(s), *([p] * 16), None)
    assert rc == -5
