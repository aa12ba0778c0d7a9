"""Single-step decode (m2rnn_decode) against the fp64 oracle at T = 1, and
against the GPU forward kernel: T decode calls must reproduce the forward's
H_T bitwise, because the state update performs the same operations in the
same order.  Tolerances are the forward's (max abs 2e-3 for fp32 inputs,
2e-2 for bf16)."""
import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import decode_state, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-2}


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn as m
    return m


def _state(B, N, K, V, seed):
    return decode_state(B, N, K, V, seed)


def _one_step(x):
    """Inputs of one decode step: the first time step of a drawn sequence."""
    return {n: (x[n][:, 0].contiguous() if n in ("q", "k", "v", "f") else x[n]) for n in
            ("q", "k", "v", "f", "W", "w_r")}


def _compare_oracle(m2rnn, oracle_mod, x1, H, dtype, in_place=False):
    g = {n: t.cuda() for n, t in x1.items()}
    Hg = H.cuda()
    if in_place:
        y, Ho = m2rnn.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], Hg, H_out=Hg)
        assert Ho.data_ptr() == Hg.data_ptr()
    else:
        y, Ho = m2rnn.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], Hg)
    torch.cuda.synchronize()
    ref = oracle_mod.fwd(x1["q"][:, None], x1["k"][:, None], x1["v"][:, None], x1["f"][:, None],
                         x1["W"], x1["w_r"], H0=H)
    ey = np.abs(y.float().cpu().numpy() - ref["y"][:, 0]).max()
    eh = np.abs(Ho.cpu().double().numpy() - ref["HT"]).max()
    assert max(ey, eh) <= TOL[dtype], (ey, eh)
    return y, Ho


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,V", [(16, 16), (32, 16), (64, 16), (128, 16), (64, 32), (128, 32)])
def test_decode_parity(m2rnn, oracle_mod, dtype, K, V):
    B, N = 5, 3
    x = make_inputs(B, 1, N, K, V, dtype, 900 + K + V)
    _compare_oracle(m2rnn, oracle_mod, _one_step(x), _state(B, N, K, V, K), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_in_place(m2rnn, oracle_mod, dtype):
    B, N, K, V = 4, 5, 64, 16
    x1 = _one_step(make_inputs(B, 1, N, K, V, dtype, 77))
    H = _state(B, N, K, V, 5)
    y0, H0 = _compare_oracle(m2rnn, oracle_mod, x1, H, dtype)
    y1, H1 = _compare_oracle(m2rnn, oracle_mod, x1, H, dtype, in_place=True)
    assert torch.equal(y0, y1) and torch.equal(H0, H1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,V", [(64, 16), (128, 32)])
def test_decode_chain_matches_forward(m2rnn, dtype, K, V):
    """T decode calls from H0 give the forward kernel's H_T exactly, and y
    per step within the tolerance (the forward reads y out through the
    tensor cores, decode in fp32)."""
    B, T, N = 3, 40, 4
    x = {n: t.cuda() for n, t in make_inputs(B, T, N, K, V, dtype, 31).items()}
    H0 = _state(B, N, K, V, 8).cuda()
    yf, HT, _ = m2rnn.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], H0)
    H = H0.clone()
    ys = []
    for t in range(T):
        y, _ = m2rnn.decode(x["q"][:, t].contiguous(), x["k"][:, t].contiguous(),
                            x["v"][:, t].contiguous(), x["f"][:, t].contiguous(), x["W"],
                            x["w_r"], H, H_out=H)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(H, HT)
    ey = (torch.stack(ys, 1).float() - yf.float()).abs().max().item()
    assert ey <= TOL[dtype], ey


def test_decode_many_sequences_sampled(m2rnn, oracle_mod):
    """B = 2048 sequences x 32 heads, the decode workload bench.py times;
    the oracle checks a sample of sequences in full."""
    B, N, K, V = 2048, 32, 64, 16
    x1 = _one_step(make_inputs(B, 1, N, K, V, "bf16", 5))
    H = _state(B, N, K, V, 9)
    g = {n: t.cuda() for n, t in x1.items()}
    y, Ho = m2rnn.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H.cuda())
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 311, 777, 1024, 1500, 2047])
    sub = {n: (t[rows] if n in ("q", "k", "v", "f") else t) for n, t in x1.items()}
    ref = oracle_mod.fwd(sub["q"][:, None], sub["k"][:, None], sub["v"][:, None], sub["f"][:, None],
                         sub["W"], sub["w_r"], H0=H[rows])
    ey = np.abs(y[rows.cuda()].float().cpu().numpy() - ref["y"][:, 0]).max()
    eh = np.abs(Ho[rows.cuda()].cpu().double().numpy() - ref["HT"]).max()
    assert max(ey, eh) <= TOL["bf16"], (ey, eh)


def test_decode_rejects_overlapping_states(m2rnn):
    B, N, K, V = 2, 2, 64, 16
    x1 = {n: t.cuda() for n, t in _one_step(make_inputs(B, 1, N, K, V, "bf16", 1)).items()}
    buf = torch.zeros(B * N * K * V + 64, device="cuda")
    H_in = buf[:B * N * K * V].view(B, N, K, V)
    H_out = buf[64:].view(B, N, K, V)
    with pytest.raises(m2rnn.M2RNNError) as e:
        m2rnn.decode(x1["q"], x1["k"], x1["v"], x1["f"], x1["W"], x1["w_r"], H_in, H_out=H_out)
    assert e.value.code == -1


@pytest.mark.parametrize("Nq", [2, 6])
def test_decode_grouped_qk(m2rnn, oracle_mod, Nq):
    """Nq query/key groups: q, k [B,Nq,K], head n reads group n // (N/Nq)."""
    B, N, K, V = 4, 6, 64, 16
    x = make_inputs(B, 1, N, K, V, "bf16", 950 + Nq, groups=Nq)
    _compare_oracle(m2rnn, oracle_mod, _one_step(x), _state(B, N, K, V, Nq), "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_gated(m2rnn, oracle_mod, dtype):
    """The fused gate in decode: one step against the oracle's gated forward
    at T = 1, and T steps against m2rnn_fwd_gated's H_T bit for bit."""
    B, T, N, K, V = 3, 12, 4, 64, 16
    x = make_inputs(B, T, N, K, V, dtype, 971, gated=True)
    H0 = _state(B, N, K, V, 19)
    g = {n: t.cuda() for n, t in x.items()}
    y1, H1 = m2rnn.decode_gated(g["q"][:, 0].contiguous(), g["k"][:, 0].contiguous(),
                                g["v"][:, 0].contiguous(), g["a"][:, 0].contiguous(), g["alpha"],
                                g["beta"], g["W"], g["w_r"], H0.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.fwd_gated(x["q"][:, :1], x["k"][:, :1], x["v"][:, :1], x["a"][:, :1],
                               x["alpha"], x["beta"], x["W"], x["w_r"], H0=H0)
    assert np.abs(y1.float().cpu().numpy() - ref["y"][:, 0]).max() <= TOL[dtype]
    assert np.abs(H1.cpu().double().numpy() - ref["HT"]).max() <= TOL[dtype]
    _, HT, _ = m2rnn.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                               g["w_r"], H0.cuda())
    H = H0.cuda()
    for t in range(T):
        _, H = m2rnn.decode_gated(g["q"][:, t].contiguous(), g["k"][:, t].contiguous(),
                                  g["v"][:, t].contiguous(), g["a"][:, t].contiguous(),
                                  g["alpha"], g["beta"], g["W"], g["w_r"], H, H_out=H)
    torch.cuda.synchronize()
    assert torch.equal(H, HT)
