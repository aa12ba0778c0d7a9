"""Forward parity: libm2rnn (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Tolerances (max |.| elementwise on y, H_T and checkpoints): 2e-3 for fp32
operands, 2e-2 for bf16 operands.

Short sequences are compared along the whole trajectory.  Long sequences are
compared per checkpoint interval: the oracle restarts from the GPU's own
checkpoint at the start of every interval of C steps, and y over the
interval plus the state at its end (the next checkpoint, or H_T) must match.
This checks every step of the GPU path while bounding the amplification of
rounding differences to C steps: at these input distributions the
recurrence has transient unstable windows (the oracle alone, fed inputs
perturbed by 1e-7, departs from itself by more than 1e-3 around step 540 of
the B=8, T=2048 workload), so no finite-precision implementation follows the
fp64 trajectory elementwise through them.
The largest workloads are compared on sampled (batch, head) pairs, which the
oracle computes from sliced inputs.
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


def _restart_parity(oracle_mod, x, y, HT, ck, C, tol, label, H0=None):
    """Oracle restarted from the GPU checkpoint of every interval of C steps
    (inputs given for all heads of the batch items in x)."""
    q, k, v, f = (x[n] for n in ("q", "k", "v", "f"))
    B, T, K = q.shape[0], q.shape[1], q.shape[-1]  # q: [B,T,K] or grouped [B,T,Nq,K]
    N, V = v.shape[2], v.shape[3]
    ckn = _np(ck)                      # [B,N,nck,K,V]
    yn, HTn = _np(y), _np(HT)
    nck = ckn.shape[2]
    assert nck == -(-T // C)
    h0 = np.zeros((B, N, K, V)) if H0 is None else H0.double().numpy()
    assert np.abs(ckn[:, :, 0] - h0).max() <= 1e-6, (label, "ckpt[0] != H0")
    worst = {"y": 0.0, "state": 0.0}
    groups = ((0, T // C, C), (T // C, nck, T - (T // C) * C))  # full intervals, ragged tail
    for c0, c1, L in groups:
        if c1 <= c0:
            continue
        t0, t1 = c0 * C, c0 * C + (c1 - c0) * L
        nb = c1 - c0

        def split(a):  # [B, t0:t1, ...] -> [B*nb, L, ...]
            a = a[:, t0:t1]
            return a.reshape(B * nb, L, *a.shape[2:])
        Hs = np.ascontiguousarray(np.moveaxis(ckn[:, :, c0:c1], 2, 1)).reshape(B * nb, N, K, V)
        r = oracle_mod.fwd(split(q), split(k), split(v), split(f), x["W"], x["w_r"], H0=Hs)
        ey = np.abs(split(yn) - r["y"]).max()
        nxt = np.concatenate([ckn[:, :, 1:], HTn[:, :, None]], axis=2)[:, :, c0:c1]
        nxt = np.ascontiguousarray(np.moveaxis(nxt, 2, 1)).reshape(B * nb, N, K, V)
        es = np.abs(nxt - r["HT"]).max()
        worst["y"] = max(worst["y"], ey)
        worst["state"] = max(worst["state"], es)
    assert worst["y"] <= tol and worst["state"] <= tol, (label, worst)
    return worst


@pytest.mark.parametrize("name", ["fwd_f32_b1_t64_n4", "fwd_bf16_b8_t2048_n32"])
def test_small_workloads(m2rnn, oracle_mod, name):
    w = WORKLOADS[name]
    x = workload_inputs(w, with_dy=False)
    if w.T <= 256:
        _compare(m2rnn, oracle_mod, x, w.dtype, ckpt_every=32, label=name)
    g = _dev(x)
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=64)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    _restart_parity(oracle_mod, x, y, HT, ck, 64, TOL[w.dtype], name)


def test_long_sequence(m2rnn, oracle_mod):
    """B=1, T=65536, N=64: the serial chain, every output checked per
    64-step interval."""
    w = WORKLOADS["fwd_bf16_b1_t65536_n64"]
    x = workload_inputs(w, with_dy=False)
    g = _dev(x)
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=64)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    _restart_parity(oracle_mod, x, y, HT, ck, 64, TOL[w.dtype], w.name)


def _sampled(m2rnn, oracle_mod, w, pairs):
    x = workload_inputs(w, with_dy=False)
    g = _dev(x)
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=64)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    for b, n in pairs:
        xs = {"q": x["q"][b:b + 1], "k": x["k"][b:b + 1], "v": x["v"][b:b + 1, :, n:n + 1],
              "f": x["f"][b:b + 1, :, n:n + 1], "W": x["W"][n:n + 1], "w_r": x["w_r"][n:n + 1]}
        _restart_parity(oracle_mod, xs, y[b:b + 1, :, n:n + 1].contiguous(),
                        HT[b:b + 1, n:n + 1].contiguous(), ck[b:b + 1, n:n + 1].contiguous(),
                        64, TOL[w.dtype], (w.name, b, n))


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
    """Ragged time (not a multiple of the ring chunk, 32 or 64 steps), heads
    not a multiple of the per-CTA group, every supported K and V, random H0."""
    B, N = 2, 5
    x = make_inputs(B, T, N, K, V, dtype, 1000 + K + V + T)
    H0 = torch.rand(B, N, K, V, generator=torch.Generator().manual_seed(T)) - 0.5
    _compare(m2rnn, oracle_mod, x, dtype, H0=H0, ckpt_every=16, label=f"{dtype} {K} {V} {T}")


def test_restart_parity_ragged_tail_and_H0(m2rnn, oracle_mod):
    """Checkpoint-interval parity with a ragged last interval and a given H0."""
    B, T, N = 3, 1000, 6
    x = make_inputs(B, T, N, 64, 16, "bf16", 31)
    H0 = torch.rand(B, N, 64, 16, generator=torch.Generator().manual_seed(3)) - 0.5
    g = _dev(x)
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H0.cuda(),
                          ckpt_every=48)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    _restart_parity(oracle_mod, x, y, HT, ck, 48, TOL["bf16"], "ragged", H0=H0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ring_chunk_lengths(m2rnn, oracle_mod, monkeypatch, dtype):
    """Ring chunks of 2, 5, 32 and 64 steps (forced through M2RNN_FWD_TC) on a
    ragged T with checkpoints that fall inside chunks and a given H0: the
    same y, H_T and checkpoints bit for bit (the chunk length changes when a
    step's inputs arrive, not its arithmetic), and those against the oracle
    restarted at every checkpoint."""
    B, T, N = 2, 147, 5
    x = make_inputs(B, T, N, 64, 16, dtype, 820)
    H0 = torch.rand(B, N, 64, 16, generator=torch.Generator().manual_seed(9)) - 0.5
    g = _dev(x)
    runs = {}
    for tc in ("2", "5", "32", "64"):
        monkeypatch.setenv("M2RNN_FWD_TC", tc)
        y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H0.cuda(),
                              ckpt_every=24)
        torch.cuda.synchronize()
        _check_status(m2rnn)
        runs[tc] = (y, HT, ck)
    for tc in ("2", "5", "32"):
        for a, b2, what in zip(runs[tc], runs["64"], ("y", "H_T", "ckpt")):
            assert torch.equal(a, b2), (tc, what)
    y, HT, ck = runs["64"]
    _restart_parity(oracle_mod, x, y, HT, ck, 24, TOL[dtype], f"chunks {dtype}", H0=H0)


@pytest.mark.parametrize("mt", ["0", "1", "2", "4"])
def test_rows_per_warp_variants(m2rnn, oracle_mod, monkeypatch, mt):
    """Every rows-per-warp variant (forced through M2RNN_FWD_MT; 0 = half
    slices of 8 rows) on a ragged shape with H0 and checkpoints."""
    monkeypatch.setenv("M2RNN_FWD_MT", mt)
    B, T, N = 3, 77, 6
    x = make_inputs(B, T, N, 64, 16, "bf16", 600 + int(mt))
    H0 = torch.rand(B, N, 64, 16, generator=torch.Generator().manual_seed(4)) - 0.5
    _compare(m2rnn, oracle_mod, x, "bf16", H0=H0, ckpt_every=16, label=f"MT={mt}")


@pytest.mark.parametrize("G", ["1", "4", "5", "14"])
@pytest.mark.parametrize("gated", [False, True])
def test_wave_kernel(m2rnn, oracle_mod, monkeypatch, G, gated):
    """The one-wave kernel (forced through M2RNN_FWD_WAVE; G heads per CTA
    over the flattened (b, n) order, so with G = 4 or 5 and N = 6 CTAs span
    two batch items), a ragged T (not a multiple of the 32-step chunk), H0
    and checkpoints, f given or from the fused gate: whole trajectory."""
    monkeypatch.setenv("M2RNN_FWD_WAVE", "1")
    monkeypatch.setenv("M2RNN_FWD_WAVE_G", G)
    B, T, N = 5, 77, 6 if G != "14" else 16  # (G = 14: a last CTA of 10 heads)
    x = make_inputs(B, T, N, 64, 16, "bf16", 640 + int(G), gated=gated)
    H0 = torch.rand(B, N, 64, 16, generator=torch.Generator().manual_seed(int(G))) - 0.5
    if not gated:
        _compare(m2rnn, oracle_mod, x, "bf16", H0=H0, ckpt_every=16, label=f"wave G={G}")
        return
    g = _dev(x)
    y, HT, ck = m2rnn.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                                g["w_r"], H0.cuda(), ckpt_every=16)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    ref = oracle_mod.fwd_gated(x["q"], x["k"], x["v"], x["a"], x["alpha"], x["beta"], x["W"],
                               x["w_r"], H0=H0, want_states=True)
    assert np.abs(_np(y) - ref["y"]).max() <= TOL["bf16"]
    assert np.abs(_np(HT) - ref["HT"]).max() <= TOL["bf16"]
    assert np.abs(_np(ck) - ref["states"][:, :, list(range(0, T, 16))]).max() <= TOL["bf16"]


def test_wave_kernel_checkpoint_only(m2rnn, monkeypatch):
    """With y = NULL (the backward's own checkpoint recompute) the one-wave
    kernel writes checkpoints only, bit for bit those of the full run."""
    monkeypatch.setenv("M2RNN_FWD_WAVE", "1")
    monkeypatch.setenv("M2RNN_FWD_WAVE_G", "5")
    x = _dev(make_inputs(4, 100, 6, 64, 16, "bf16", 5, with_dy=True))
    _, _, ck = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], ckpt_every=20)
    a = m2rnn.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"], ckpt=ck, ckpt_every=20)
    b = m2rnn.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"], ckpt=None,
                  ckpt_every=20)
    torch.cuda.synchronize()
    _check_status(m2rnn)
    for n in a:
        err = (a[n].double() - b[n].double()).norm() / a[n].double().norm().clamp_min(1e-30)
        assert err <= 1e-5, (n, float(err))


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
    """With fault injection the producer starts no transfers, so the other
    warps' waits can never complete: they must give up after the wait limit,
    record M2RNN_ERR_TIMEOUT in the device status word, and leave the context
    usable for the next, correct call."""
    x = make_inputs(2, 256, 8, 64, 16, "bf16", 3)
    g = _dev(x)
    m2rnn.device_status(clear=True)
    m2rnn.set_wait_limit_ns(20_000_000)  # 20 ms
    m2rnn.set_fault_injection(1)
    try:
        m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
        st, detail = m2rnn.device_status(clear=True)
    finally:
        m2rnn.set_fault_injection(0)
        m2rnn.set_wait_limit_ns(0)
    assert st == -7 and detail in (2, 3), (st, detail)
    _compare(m2rnn, oracle_mod, make_inputs(2, 50, 4, 64, 16, "bf16", 5), "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Nq", [2, 4, 32])
def test_grouped_qk(m2rnn, oracle_mod, dtype, Nq):
    """N_q = N_k = Nq query/key groups: head n reads q, k of group
    n // (N / Nq), so a CTA's heads stay inside one group and the producer
    copies the group's rows one step at a time.  Whole trajectory at T = 40
    and per 16-step interval at T = 300."""
    for T in (40, 300):
        x = make_inputs(3, T, 32, 64, 16, dtype, 700 + Nq + T, groups=Nq)
        if T <= 40:
            _compare(m2rnn, oracle_mod, x, dtype, ckpt_every=16, label=f"Nq{Nq} T{T}")
            continue
        g = _dev(x)
        y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=16)
        torch.cuda.synchronize()
        _check_status(m2rnn)
        _restart_parity(oracle_mod, x, y, HT, ck, 16, TOL[dtype], f"Nq{Nq} T{T}")


def test_grouped_qk_wave_split(m2rnn, oracle_mod):
    """A batch large enough for the whole-wave launch plus the tail launch,
    with 4 groups of 8 heads: both launches' q/k offsets."""
    x = make_inputs(41, 40, 32, 64, 16, "bf16", 733, groups=4)
    _compare(m2rnn, oracle_mod, x, "bf16", label="Nq4 wave split")


def test_state_bitwise_across_launch_variants(m2rnn, monkeypatch):
    """The state update is the same per element whatever the launch shape:
    the whole-wave and tail launches with compile-time K and heads per CTA
    (two slices per warp), the generic instance with one slice per warp
    (previous step's readout deferred), a single launch and the one-wave
    kernel (one warp per head, 9 heads per CTA across batch items) all give
    the same H_T bit for bit (y may differ in the last bits: its row sums
    are grouped by warp)."""
    x = _dev(make_inputs(41, 96, 32, 64, 16, "bf16", 733))
    runs = {}
    for name, env in (("planned", {"M2RNN_FWD_WAVE": "0"}),
                      ("one_slice", {"M2RNN_FWD_MT": "1", "M2RNN_FWD_WAVE": "0"}),
                      ("one_launch", {"M2RNN_FWD_ONE_LAUNCH": "1", "M2RNN_FWD_WAVE": "0"}),
                      ("wave", {"M2RNN_FWD_WAVE": "1", "M2RNN_FWD_WAVE_G": "9"})):
        for k in ("M2RNN_FWD_MT", "M2RNN_FWD_ONE_LAUNCH", "M2RNN_FWD_WAVE", "M2RNN_FWD_WAVE_G"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        y, HT, _ = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
        torch.cuda.synchronize()
        runs[name] = (y.float(), HT)
    _check_status(m2rnn)
    for name in ("one_slice", "one_launch", "wave"):
        assert torch.equal(runs[name][1], runs["planned"][1]), name
        assert (runs[name][0] - runs["planned"][0]).abs().max().item() <= 2e-2, name


SHAPES = [  # (B, T, N, env): one-head CTAs; 8-head + 2-head tail instances; one-wave kernel
    (2, 37, 8, {}),
    (41, 24, 32, {}),
    (5, 33, 32, {"M2RNN_FWD_WAVE": "1", "M2RNN_FWD_WAVE_G": "9"}),
]


@pytest.mark.parametrize("B,T,N,env", SHAPES)
def test_degenerate_f_one(m2rnn, monkeypatch, B, T, N, env):
    """f = 1 from H0 = 0 (Eq. 11 then never admits the candidate): the state
    stays exactly 0 and y = w_r (.) v, i.e. the bf16 rounding of the fp32
    product, bit for bit, in every launch shape."""
    for k in ("M2RNN_FWD_WAVE", "M2RNN_FWD_WAVE_G"):
        monkeypatch.delenv(k, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    x = make_inputs(B, T, N, 64, 16, "bf16", 900 + B)
    x["f"] = torch.ones_like(x["f"])
    g = _dev(x)
    y, HT, _ = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
    torch.cuda.synchronize()
    _check_status(m2rnn)
    assert torch.count_nonzero(HT) == 0
    expect = (x["w_r"].float()[None, None] * x["v"].float()).to(torch.bfloat16)
    assert torch.equal(y.cpu(), expect)


@pytest.mark.parametrize("B,T,N,env", SHAPES)
def test_degenerate_no_transition(m2rnn, oracle_mod, monkeypatch, B, T, N, env):
    """W = 0 and f = 0: every step forgets the past and H_t = tanh(k_t v_t^T)
    (Eqs. 10-11), so H_T depends on the last step only; y against the oracle."""
    for k in ("M2RNN_FWD_WAVE", "M2RNN_FWD_WAVE_G"):
        monkeypatch.delenv(k, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    x = make_inputs(B, T, N, 64, 16, "bf16", 950 + B)
    x["f"] = torch.zeros_like(x["f"])
    x["W"] = torch.zeros_like(x["W"])
    g = _dev(x)
    y, HT, _ = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
    torch.cuda.synchronize()
    _check_status(m2rnn)
    kT = x["k"][:, -1].double()                       # [B, K]
    vT = x["v"][:, -1].double()                       # [B, N, V]
    expect = torch.tanh(kT[:, None, :, None] * vT[:, :, None, :])
    assert (HT.cpu().double() - expect).abs().max().item() <= 1e-3  # tanh.approx, |.| <= 1
    ref = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    assert np.abs(_np(y) - ref["y"]).max() <= TOL["bf16"]


def test_state_bound_full_size(m2rnn):
    """|H_t| <= 1: H is a convex blend of tanh values starting from 0 (Eq. 11),
    which holds at any size; checked on H_T of the B=64, T=4096, N=32 forward
    in the launch plan the benchmark times (up to fp32 rounding of the blend)."""
    w = WORKLOADS["fwd_bf16_b64_t4096_n32"]
    g = _dev(workload_inputs(w, with_dy=False))
    _, HT, _ = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"])
    torch.cuda.synchronize()
    _check_status(m2rnn)
    assert torch.isfinite(HT).all()
    assert HT.abs().max().item() <= 1.0 + 1e-6
