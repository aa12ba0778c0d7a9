"""Forward parity: libm2rnn (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Tolerances (max |.| elementwise on y and H_T): 2e-3 for fp32 operands, 2e-2
for bf16 operands.  Sizes the oracle finishes in seconds are compared in
full; the largest workloads are compared on sampled (batch, head) pairs,
which the oracle computes independently from sliced inputs.
"""
import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-2}


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


def _check_status(m2rnn):
    st, de = m2rnn.device_status(clear=True)
    assert st == 0, (st, de)


def _compare(m2rnn, oracle_mod, x, dtype, H0=None, ckpt_every=0, label=""):
    g = _dev(x)
    H0g = None if H0 is None else H0.cuda()
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H0g,
                          ckpt_every=ckpt_every)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    ref = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], H0=H0,
                         want_states=ckpt_every > 0)
    ey = np.abs(_np(y) - ref["y"]).max() if ref["y"].size else 0.0
    eh = np.abs(_np(HT) - ref["HT"]).max()
    assert ey <= TOL[dtype], (label, "y", ey)
    assert eh <= TOL[dtype], (label, "H_T", eh)
    if ckpt_every > 0:
        T = x["q"].shape[1]
        idx = list(range(0, T, ckpt_every))
        ec = np.abs(_np(ck) - ref["states"][:, :, idx]).max()
        assert ec <= TOL[dtype], (label, "ckpt", ec)
    return ey, eh


@pytest.mark.parametrize("name", ["fwd_f32_b1_t64_n4", "fwd_bf16_b8_t2048_n32"])
def test_small_workloads_full(m2rnn, oracle_mod, name):
    w = WORKLOADS[name]
    x = workload_inputs(w, with_dy=False)
    _compare(m2rnn, oracle_mod, x, w.dtype, ckpt_every=64, label=name)


def test_long_sequence_full(m2rnn, oracle_mod):
    """B=1, T=65536, N=64: the serial chain; compared on every output."""
    w = WORKLOADS["fwd_bf16_b1_t65536_n64"]
    x = workload_inputs(w, with_dy=False)
    _compare(m2rnn, oracle_mod, x, w.dtype, label=w.name)


def _sampled(m2rnn, oracle_mod, w, pairs):
    x = workload_inputs(w, with_dy=False)
    g = _dev(x)
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=64)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    for b, n in pairs:
        ref = oracle_mod.fwd(x["q"][b:b + 1], x["k"][b:b + 1], x["v"][b:b + 1, :, n:n + 1],
                             x["f"][b:b + 1, :, n:n + 1], x["W"][n:n + 1], x["w_r"][n:n + 1],
                             want_states=True)
        ey = np.abs(_np(y[b, :, n]) - ref["y"][0, :, 0]).max()
        eh = np.abs(_np(HT[b, n]) - ref["HT"][0, 0]).max()
        ec = np.abs(_np(ck[b, n]) - ref["states"][0, 0, ::64]).max()
        assert max(ey, eh, ec) <= TOL[w.dtype], (w.name, b, n, ey, eh, ec)


@pytest.mark.parametrize("name", ["fwd_bf16_b64_t4096_n32", "fwd_bf16_b64_t4096_n32_k128",
                                  "fwd_bf16_b64_t4096_n32_v32"])
def test_throughput_workloads_sampled(m2rnn, oracle_mod, name):
    w = WORKLOADS[name]
    pairs = [(0, 0), (0, w.N - 1), (w.B - 1, 0), (w.B - 1, w.N - 1), (17, 5), (33, 18),
             (48, 30), (5, 11)]
    _sampled(m2rnn, oracle_mod, w, pairs)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,V", [(16, 16), (32, 16), (64, 16), (128, 16), (64, 32), (128, 32)])
@pytest.mark.parametrize("T", [1, 33, 100])
def test_shapes_ragged(m2rnn, oracle_mod, dtype, K, V, T):
    """Ragged time (not a multiple of the 32-step ring chunk), heads not a
    multiple of the per-CTA group, every supported K and V, random H0."""
    B, N = 2, 5
    x = make_inputs(B, T, N, K, V, dtype, 1000 + K + V + T)
    H0 = torch.rand(B, N, K, V, generator=torch.Generator().manual_seed(T)) - 0.5
    _compare(m2rnn, oracle_mod, x, dtype, H0=H0, ckpt_every=16, label=f"{dtype} {K} {V} {T}")


def test_many_heads_per_cta_groups(m2rnn, oracle_mod):
    """Shapes whose dispatch uses several heads per CTA and 2-slice warps."""
    for (B, T, N) in [(40, 70, 64), (3, 40, 7)]:
        x = make_inputs(B, T, N, 64, 16, "bf16", B + T + N)
        _compare(m2rnn, oracle_mod, x, "bf16", label=f"{B} {T} {N}")


def test_zero_steps(m2rnn):
    x = _dev(make_inputs(2, 0, 3, 64, 16, "bf16", 0))
    H0 = torch.rand(2, 3, 64, 16, device="cuda")
    y, HT, ck = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], H0, ckpt_every=8)
    torch.cuda.synchronize()
    assert y.numel() == 0 and ck is None
    assert torch.equal(HT, H0)
    y, HT, _ = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    torch.cuda.synchronize()
    assert torch.count_nonzero(HT) == 0


def test_continuation_matches_single_pass(m2rnn):
    """fwd(T1) then fwd(T2, H0 = H_T1) gives the same result as fwd(T1+T2)."""
    x = _dev(make_inputs(4, 200, 8, 64, 16, "bf16", 77))
    y, HT, _ = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    a = {n: x[n][:, :75].contiguous() for n in ("q", "k", "v", "f")}
    c = {n: x[n][:, 75:].contiguous() for n in ("q", "k", "v", "f")}
    y1, H1, _ = m2rnn.fwd(a["q"], a["k"], a["v"], a["f"], x["W"], x["w_r"])
    y2, H2, _ = m2rnn.fwd(c["q"], c["k"], c["v"], c["f"], x["W"], x["w_r"], H1)
    torch.cuda.synchronize()
    assert torch.allclose(torch.cat([y1, y2], 1).float(), y.float(), atol=1e-2, rtol=0)
    assert torch.allclose(H2, HT, atol=1e-3, rtol=0)


def test_host_pointer_rejected(m2rnn):
    x = make_inputs(1, 8, 2, 64, 16, "bf16", 0)
    g = _dev(x)
    import ctypes
    s = m2rnn.make_shape(g["q"], g["v"])
    host = x["q"]  # CPU tensor: not device memory
    rc = m2rnn.lib().m2rnn_fwd(ctypes.byref(s), ctypes.c_void_p(host.data_ptr()),
                               *(ctypes.c_void_p(g[n].data_ptr()) for n in ("k", "v", "f", "W", "w_r")),
                               None, ctypes.c_void_p(torch.empty_like(g["v"]).data_ptr()), None, None,
                               None)
    assert rc == -4


def test_timeout_path_reports_and_recovers(m2rnn, oracle_mod):
    """A wait limit far below the time a chunk takes makes the kernel's
    waits give up: it must stop, report M2RNN_ERR_TIMEOUT through the device
    status word, and leave the context usable for the next, correct call."""
    x = make_inputs(4, 4096, 8, 64, 16, "bf16", 3)
    g = _dev(x)
    m2rnn.device_status(clear=True)
    m2rnn.set_wait_limit_ns(200)
    try:
        m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
        st, detail = m2rnn.device_status(clear=True)
    finally:
        m2rnn.set_wait_limit_ns(0)
    assert st == -7 and detail in (1, 2, 3, 4), (st, detail)
    _compare(m2rnn, oracle_mod, make_inputs(2, 50, 4, 64, 16, "bf16", 5), "bf16")
