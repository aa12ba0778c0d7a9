"""Pins for the fp64 oracle, against facts the pages and the mathematics fix.

Each test states the passage it follows.  None of them re-types the oracle's
own loop: they use invariants of Eqs. (10)-(12), closed forms, a library
routine (torch.nn.RNN), finite differences and torch.autograd.
"""
import numpy as np
import pytest
import torch

from non_linear_matrix_gb300.inputs import make_inputs


def _np(x):
    return x.detach().to(torch.float64).numpy()


def _small(B=2, T=7, N=3, K=8, V=4, seed=11, f_mean=2.0, with_dy=False, dtype="f32"):
    return make_inputs(B, T, N, K, V, dtype, seed, f_mean, with_dy=with_dy)


# --- forward ---------------------------------------------------------------

def test_f_one_keeps_zero_state(oracle_mod):
    """Gate frame: f_t = 1 retains the state; from H_0 = 0 the state stays 0
    and Eq. (12) leaves only the value residual y_t = w_r (.) v_t (exact)."""
    x = _small()
    f = torch.ones_like(x["f"])
    o = oracle_mod.fwd(x["q"], x["k"], x["v"], f, x["W"], x["w_r"], want_states=True)
    assert np.all(o["states"] == 0.0)
    assert np.all(o["HT"] == 0.0)
    expect = _np(x["w_r"])[None, None] * _np(x["v"])
    assert np.array_equal(o["y"], expect)


def test_w_zero_f_zero_is_elementwise_tanh_of_rank_one(oracle_mod):
    """Eqs. (10)-(11) with W = 0 and f = 0: H_t = tanh(k_t v_t^T), exact up
    to the last-ulp rounding of the two libm tanh implementations."""
    x = _small()
    W = torch.zeros_like(x["W"])
    f = torch.zeros_like(x["f"])
    o = oracle_mod.fwd(x["q"], x["k"], x["v"], f, W, x["w_r"], want_states=True)
    k, v = _np(x["k"]), _np(x["v"])
    for b in range(k.shape[0]):
        for n in range(v.shape[2]):
            for t in range(k.shape[1]):
                expect = np.tanh(np.multiply.outer(k[b, t], v[b, t, n]))
                np.testing.assert_allclose(o["states"][b, n, t + 1], expect, rtol=4e-16,
                                           atol=0)


@pytest.mark.parametrize("scale", [1.0, 50.0])
def test_state_bounded_by_one(oracle_mod, scale):
    """H_t is a convex blend (f in [0,1]) of H_{t-1} and tanh values,
    starting from 0, so |H_t| <= 1 elementwise for every t."""
    x = _small(T=40, seed=5)
    o = oracle_mod.fwd(x["q"], x["k"] * scale, x["v"] * scale, x["f"], x["W"] * scale,
                       x["w_r"], want_states=True)
    assert np.abs(o["states"]).max() <= 1.0
    assert np.abs(o["states"]).max() > 0.1 * min(scale, 5.0)  # non-trivial


def test_single_step_closed_form(oracle_mod):
    """T = 1 from H_0 = 0: Z_1 = tanh(k v^T) whatever W is, H_1 = (1-f) Z_1,
    y_1 = H_1^T q + w_r (.) v."""
    x = _small(T=1, seed=3)
    o = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    q, k, v, f, wr = map(_np, (x["q"], x["k"], x["v"], x["f"], x["w_r"]))
    B, _, N, V = v.shape
    for b in range(B):
        for n in range(N):
            H1 = (1 - f[b, 0, n]) * np.tanh(np.multiply.outer(k[b, 0], v[b, 0, n]))
            y1 = H1.T @ q[b, 0] + wr[n] * v[b, 0, n]
            np.testing.assert_allclose(o["y"][b, 0, n], y1, rtol=0, atol=1e-14)
            np.testing.assert_allclose(o["HT"][b, n], H1, rtol=0, atol=1e-15)


def test_vector_rnn_special_case_matches_torch_rnn(oracle_mod):
    """Backup frame "embedding a vector RNN in one matrix row" (Theorem 1 /
    App. B): f = 0, w_r = 0, q = k = e_1 give y_t = h_t with
    h_t = tanh(W^T h_{t-1} + v_t), i.e. an Elman RNN with W_ih = I,
    W_hh = W^T and no bias.  Checked against torch.nn.RNN in fp64; this pins
    the orientation of W (H W, not H W^T) and the use of H_t in the readout."""
    B, T, N, K, V = 2, 30, 3, 6, 5
    x = make_inputs(B, T, N, K, V, "f32", 21)
    e1 = torch.zeros(B, T, K)
    e1[..., 0] = 1.0
    f = torch.zeros(B, T, N)
    wr = torch.zeros(N, V)
    W = x["W"] * 2.0  # a stronger transition so the map is far from identity
    o = oracle_mod.fwd(e1, e1, x["v"], f, W, wr, want_states=True)
    for n in range(N):
        rnn = torch.nn.RNN(V, V, nonlinearity="tanh", bias=False, batch_first=True,
                           dtype=torch.float64)
        with torch.no_grad():
            rnn.weight_ih_l0.copy_(torch.eye(V, dtype=torch.float64))
            rnn.weight_hh_l0.copy_(W[n].to(torch.float64).T)
            h, _ = rnn(x["v"][:, :, n, :].to(torch.float64))
        np.testing.assert_allclose(o["y"][:, :, n, :], h.numpy(), rtol=0, atol=1e-13)
        # rows other than the first stay zero
        assert np.all(o["states"][:, n, :, 1:, :] == 0.0)


def test_key_permutation_invariance(oracle_mod):
    """Rows of H evolve independently (W acts within a row, q combines rows
    at readout): permuting the K coordinates of q and k permutes the rows of
    H and leaves y unchanged."""
    x = _small(K=10, seed=8)
    perm = torch.randperm(10, generator=torch.Generator().manual_seed(0))
    o1 = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    o2 = oracle_mod.fwd(x["q"][..., perm], x["k"][..., perm], x["v"], x["f"], x["W"], x["w_r"])
    np.testing.assert_allclose(o2["y"], o1["y"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(o2["HT"], o1["HT"][:, :, perm.numpy(), :], rtol=0, atol=1e-15)


def test_head_permutation_equivariance(oracle_mod):
    """Multi-value sharing: each value head has its own v, f, W, w_r and
    state; permuting heads together with those permutes the outputs."""
    x = _small(N=5, seed=9)
    perm = torch.tensor([3, 0, 4, 1, 2])
    o1 = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    o2 = oracle_mod.fwd(x["q"], x["k"], x["v"][:, :, perm], x["f"][:, :, perm],
                        x["W"][perm], x["w_r"][perm])
    p = perm.numpy()
    np.testing.assert_array_equal(o2["y"], o1["y"][:, :, p])
    np.testing.assert_array_equal(o2["HT"], o1["HT"][:, p])


def test_chunk_continuation(oracle_mod):
    """The recurrence is a scan: running T1 steps, then T2 steps from
    H0 = H_{T1}, equals running T1 + T2 steps."""
    x = _small(T=20, seed=10)
    o = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    a = {n: t[:, :7] for n, t in x.items() if n in ("q", "k", "v", "f")}
    c = {n: t[:, 7:] for n, t in x.items() if n in ("q", "k", "v", "f")}
    o1 = oracle_mod.fwd(a["q"], a["k"], a["v"], a["f"], x["W"], x["w_r"])
    o2 = oracle_mod.fwd(c["q"], c["k"], c["v"], c["f"], x["W"], x["w_r"], H0=o1["HT"])
    np.testing.assert_allclose(np.concatenate([o1["y"], o2["y"]], 1), o["y"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(o2["HT"], o["HT"], rtol=0, atol=1e-14)


# --- backward ---------------------------------------------------------------

def _loss(oracle_mod, inp, dy, dHT):
    o = oracle_mod.fwd(inp["q"], inp["k"], inp["v"], inp["f"], inp["W"], inp["w_r"], H0=inp["H0"])
    return float(np.sum(o["y"] * dy) + np.sum(o["HT"] * dHT))


@pytest.mark.parametrize("T", [1, 3, 8])
def test_backward_matches_central_differences(oracle_mod, T):
    """BPTT backward (backup frame "the recurrent gradient needs both
    paths", plus the value-residual and q/k/v terms it mentions) against
    brute-force central differences of L = sum y (.) dy + sum H_T (.) dH_T,
    in fp64, at T <= 8 and every input element."""
    B, N, K, V = 2, 2, 3, 3
    x = make_inputs(B, T, N, K, V, "f32", 100 + T, with_dy=True)
    rng = np.random.default_rng(T)
    inp = {n: _np(x[n]).copy() for n in ("q", "k", "v", "f", "W", "w_r")}
    inp["H0"] = rng.uniform(-0.5, 0.5, size=(B, N, K, V))
    dy = _np(x["dy"])
    dHT = rng.normal(size=(B, N, K, V))
    g = oracle_mod.bwd(inp["q"], inp["k"], inp["v"], inp["f"], inp["W"], inp["w_r"], dy,
                       H0=inp["H0"], dHT=dHT)
    names = {"q": "dq", "k": "dk", "v": "dv", "f": "df", "W": "dW", "w_r": "dw_r", "H0": "dH0"}
    h = 1e-6
    for name, gname in names.items():
        arr = inp[name]
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(oracle_mod, inp, dy, dHT)
            arr[idx] = old - h
            lm = _loss(oracle_mod, inp, dy, dHT)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(g[gname] - fd).max() / max(1.0, np.abs(fd).max())
        assert err <= 1e-6, (gname, err)


def test_backward_matches_autograd(oracle_mod):
    """Independent check of every gradient with torch.autograd in fp64 on a
    plain tensor restatement of Eqs. (10)-(12) at a small shape."""
    B, T, N, K, V = 2, 12, 3, 5, 4
    x = make_inputs(B, T, N, K, V, "f32", 55, with_dy=True)
    t = {n: x[n].to(torch.float64).clone().requires_grad_(True)
         for n in ("q", "k", "v", "f", "W", "w_r")}
    H0 = (torch.rand(B, N, K, V, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
          - 0.5).requires_grad_(True)
    dHT = torch.randn(B, N, K, V, dtype=torch.float64, generator=torch.Generator().manual_seed(2))
    H = H0
    ys = []
    for s in range(T):
        A = torch.matmul(H, t["W"].unsqueeze(0)) + \
            t["k"][:, s, None, :, None] * t["v"][:, s, :, None, :]
        Z = torch.tanh(A)
        fs = t["f"][:, s, :, None, None]
        H = fs * H + (1 - fs) * Z
        ys.append(torch.einsum("bnkv,bk->bnv", H, t["q"][:, s]) + t["w_r"][None] * t["v"][:, s])
    y = torch.stack(ys, 1)
    dy = x["dy"].to(torch.float64)
    (torch.sum(y * dy) + torch.sum(H * dHT)).backward()
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"],
                       H0=H0.detach(), dHT=dHT)
    pairs = {"dq": t["q"], "dk": t["k"], "dv": t["v"], "df": t["f"], "dW": t["W"],
             "dw_r": t["w_r"]}
    for gname, leaf in pairs.items():
        np.testing.assert_allclose(g[gname], leaf.grad.numpy(), rtol=1e-10, atol=1e-12,
                                   err_msg=gname)
    np.testing.assert_allclose(g["dH0"], H0.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_f_one(oracle_mod):
    """f = 1 keeps H = 0 and blocks the candidate path ((1 - f) = 0): then
    dW = 0, dk = 0, dq = 0 and dv = w_r (.) dy exactly (with dH_T = 0)."""
    x = _small(with_dy=True)
    f = torch.ones_like(x["f"])
    g = oracle_mod.bwd(x["q"], x["k"], x["v"], f, x["W"], x["w_r"], x["dy"])
    assert np.all(g["dW"] == 0) and np.all(g["dk"] == 0) and np.all(g["dq"] == 0)
    np.testing.assert_array_equal(g["dv"], _np(x["w_r"])[None, None] * _np(x["dy"]))


# --- fused input gate (frame "The gate preserves a direct path through time")

def test_gate_special_values(oracle_mod):
    """softplus(0) = ln 2, so a = -beta gives f = 2^(-alpha); alpha = 0 gives
    f = 1 for every a; for a + beta >> 1, softplus(x) -> x."""
    alpha = np.array([0.0, 0.5, 1.0, 2.0])
    beta = np.array([-2.0, 0.3, 1.5, -0.7])
    a = np.broadcast_to(-beta, (2, 3, 4)).copy()
    f = oracle_mod.gate(a, alpha, beta)
    assert np.allclose(f, np.broadcast_to(2.0 ** (-alpha), f.shape), rtol=1e-15, atol=0)
    f0 = oracle_mod.gate(np.random.default_rng(0).normal(size=(2, 3, 4)) * 5, np.zeros(4), beta)
    assert np.array_equal(f0, np.ones_like(f0))
    big = oracle_mod.gate(np.full((1, 1, 4), 40.0), alpha, beta)[0, 0]
    assert np.allclose(big, np.exp(-alpha * (40.0 + beta)), rtol=1e-12, atol=0)


def test_gate_alpha_zero_keeps_zero_state(oracle_mod):
    """alpha = 0 makes f = 1: H stays 0, y = w_r (.) v, and a, beta get no
    gradient."""
    x = make_inputs(2, 6, 3, 8, 4, "f32", 5, with_dy=True, gated=True)
    alpha = torch.zeros(3)
    o = oracle_mod.fwd_gated(x["q"], x["k"], x["v"], x["a"], alpha, x["beta"], x["W"], x["w_r"])
    assert np.array_equal(o["HT"], np.zeros_like(o["HT"]))
    assert np.allclose(o["y"], _np(x["w_r"])[None, None] * _np(x["v"]), rtol=1e-15, atol=0)
    g = oracle_mod.bwd_gated(x["q"], x["k"], x["v"], x["a"], alpha, x["beta"], x["W"], x["w_r"],
                             x["dy"])
    assert np.count_nonzero(g["da"]) == 0 and np.count_nonzero(g["dbeta"]) == 0


@pytest.mark.parametrize("T", [1, 4])
def test_gated_backward_matches_central_differences(oracle_mod, T):
    """da, dalpha, dbeta of the gated backward against brute-force central
    differences of L = sum y (.) dy + sum H_T (.) dH_T in fp64, every
    element of a, alpha and beta."""
    B, N, K, V = 2, 2, 3, 3
    x = make_inputs(B, T, N, K, V, "f32", 300 + T, with_dy=True, gated=True)
    rng = np.random.default_rng(T + 7)
    inp = {n: _np(x[n]).copy() for n in ("q", "k", "v", "a", "alpha", "beta", "W", "w_r")}
    H0 = rng.uniform(-0.5, 0.5, size=(B, N, K, V))
    dy = _np(x["dy"])
    dHT = rng.normal(size=(B, N, K, V))

    def loss():
        o = oracle_mod.fwd_gated(inp["q"], inp["k"], inp["v"], inp["a"], inp["alpha"],
                                 inp["beta"], inp["W"], inp["w_r"], H0=H0)
        return float(np.sum(o["y"] * dy) + np.sum(o["HT"] * dHT))

    g = oracle_mod.bwd_gated(inp["q"], inp["k"], inp["v"], inp["a"], inp["alpha"], inp["beta"],
                             inp["W"], inp["w_r"], dy, H0=H0, dHT=dHT)
    h = 1e-6
    for name, gname in (("a", "da"), ("alpha", "dalpha"), ("beta", "dbeta")):
        arr = inp[name]
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = loss()
            arr[idx] = old - h
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(g[gname] - fd).max() / max(1.0, np.abs(fd).max())
        assert err <= 1e-6, (gname, err)


# --- grouped queries and keys (frame "Tensor parallelism trades topology
# dependence for sync": one query/key group per block of value heads) -------

def test_grouped_identical_groups_equal_shared(oracle_mod):
    """Every group given the same q, k is the shared form N_q = 1: y, H_T
    and all parameter gradients agree, and the shared dq, dk are the sums of
    the per-group ones (the heads of a group sum into its dq, dk)."""
    x = make_inputs(2, 5, 6, 8, 4, "f32", 41, with_dy=True)
    G = 3
    qg = x["q"][:, :, None].expand(-1, -1, G, -1).contiguous()
    kg = x["k"][:, :, None].expand(-1, -1, G, -1).contiguous()
    rng = np.random.default_rng(2)
    H0 = rng.uniform(-0.5, 0.5, size=(2, 6, 8, 4))
    a = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], H0=H0)
    b = oracle_mod.fwd(qg, kg, x["v"], x["f"], x["W"], x["w_r"], H0=H0)
    np.testing.assert_allclose(b["y"], a["y"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(b["HT"], a["HT"], rtol=0, atol=1e-15)
    ga = oracle_mod.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"], H0=H0)
    gb = oracle_mod.bwd(qg, kg, x["v"], x["f"], x["W"], x["w_r"], x["dy"], H0=H0)
    assert gb["dq"].shape == (2, 5, G, 8)
    np.testing.assert_allclose(gb["dq"].sum(axis=2), ga["dq"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gb["dk"].sum(axis=2), ga["dk"], rtol=1e-12, atol=1e-14)
    for n in ("dv", "df", "dW", "dw_r", "dH0"):
        np.testing.assert_allclose(gb[n], ga[n], rtol=1e-12, atol=1e-14)


def test_grouped_head_blocks(oracle_mod):
    """Value head n reads group n // (N / G): with N = 4, G = 2, heads 0-1
    use group 0 and heads 2-3 group 1.  Each block run alone as a shared
    problem with its group's q, k gives the same outputs."""
    x = make_inputs(2, 6, 4, 8, 4, "f32", 43, with_dy=True, groups=2)
    o = oracle_mod.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
    for grp, heads in ((0, slice(0, 2)), (1, slice(2, 4))):
        r = oracle_mod.fwd(x["q"][:, :, grp], x["k"][:, :, grp], x["v"][:, :, heads],
                           x["f"][:, :, heads], x["W"][heads], x["w_r"][heads])
        np.testing.assert_array_equal(o["y"][:, :, heads], r["y"])
    # swapping the two groups' q, k changes the outputs (the mapping matters)
    sw = oracle_mod.fwd(x["q"].flip(2), x["k"].flip(2), x["v"], x["f"], x["W"], x["w_r"])
    assert np.abs(sw["y"] - o["y"]).max() > 1e-3


@pytest.mark.parametrize("T", [1, 4])
def test_grouped_backward_matches_central_differences(oracle_mod, T):
    """dq, dk of the grouped backward against brute-force central
    differences of L = sum y (.) dy + sum H_T (.) dH_T in fp64, every
    element of the grouped q and k (N = 4 heads in G = 2 groups)."""
    B, N, K, V, G = 2, 4, 3, 3, 2
    x = make_inputs(B, T, N, K, V, "f32", 350 + T, with_dy=True, groups=G)
    rng = np.random.default_rng(T + 9)
    inp = {n: _np(x[n]).copy() for n in ("q", "k", "v", "f", "W", "w_r")}
    H0 = rng.uniform(-0.5, 0.5, size=(B, N, K, V))
    dy = _np(x["dy"])
    dHT = rng.normal(size=(B, N, K, V))

    def loss():
        o = oracle_mod.fwd(inp["q"], inp["k"], inp["v"], inp["f"], inp["W"], inp["w_r"], H0=H0)
        return float(np.sum(o["y"] * dy) + np.sum(o["HT"] * dHT))

    g = oracle_mod.bwd(inp["q"], inp["k"], inp["v"], inp["f"], inp["W"], inp["w_r"], dy, H0=H0,
                       dHT=dHT)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk")):
        arr = inp[name]
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = loss()
            arr[idx] = old - h
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(g[gname] - fd).max() / max(1.0, np.abs(fd).max())
        assert err <= 1e-6, (gname, err)


# --- readout epilogue (frames "Most of the block can be computed before
# recurrence": x g_t, then RMSNorm; "Backup: RMSNormTP synchronizes per-token
# statistics": the norm and its gradient) ------------------------------------

def _norm_inputs(seed=3, B=2, T=3, N=2, V=4):
    x = make_inputs(B, T, N, 8, V, "f32", seed, with_dy=True, norm=True)
    return _np(x["dy"]) * 0.7, _np(x["g"]), _np(x["w_norm"]), _np(x["dy"])


@pytest.mark.parametrize("eps", [0.0, 1e-3])
def test_readout_norm_matches_library_rms_norm(oracle_mod, eps):
    """The forward against torch.nn.functional.rms_norm over the token's
    N*V features (fp64), applied to y (.) g."""
    y, g, w, _ = _norm_inputs()
    r = oracle_mod.readout_norm(y, g, w, eps)
    o = torch.from_numpy(y * g)
    ref = torch.nn.functional.rms_norm(o, (o.shape[2], o.shape[3]), torch.from_numpy(w), eps=eps)
    np.testing.assert_allclose(r["out"], ref.numpy(), rtol=1e-13, atol=1e-15)


def test_readout_norm_unit_rms_and_scale_invariance(oracle_mod):
    """eps = 0: every token's (out / w) has mean square exactly 1 over its
    N*V features, and scaling y by c > 0 leaves out unchanged."""
    y, g, w, _ = _norm_inputs(seed=5, N=3, V=8)
    r = oracle_mod.readout_norm(y, g, w)
    ms = ((r["out"] / w[None, None]) ** 2).mean(axis=(2, 3))
    np.testing.assert_allclose(ms, 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle_mod.readout_norm(3.7 * y, g, w)["out"], r["out"],
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(r["rstd"], 1 / np.sqrt(((y * g) ** 2).mean(axis=(2, 3))),
                               rtol=1e-13)


@pytest.mark.parametrize("eps", [0.0, 1e-3])
def test_readout_norm_backward_matches_autograd(oracle_mod, eps):
    """dy, dg, dw against fp64 torch.autograd through the library rms_norm."""
    y, g, w, dout = _norm_inputs(seed=9, N=3, V=4)
    r = oracle_mod.readout_norm_bwd(y, g, w, dout, eps)
    yt, gt, wt = (torch.from_numpy(a).requires_grad_() for a in (y, g, w))
    o = yt * gt
    out = torch.nn.functional.rms_norm(o, (o.shape[2], o.shape[3]), wt, eps=eps)
    out.backward(torch.from_numpy(dout))
    for name, t in (("dy", yt), ("dg", gt), ("dw", wt)):
        np.testing.assert_allclose(r[name], t.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_readout_norm_backward_central_differences(oracle_mod):
    """dy, dg, dw against brute-force central differences of
    L = sum out (.) dout on every element (fp64, eps = 0)."""
    y, g, w, dout = _norm_inputs(seed=13, B=1, T=2, N=2, V=3)
    r = oracle_mod.readout_norm_bwd(y, g, w, dout)
    arrs = {"dy": y, "dg": g, "dw": w}
    h = 1e-6
    for name, arr in arrs.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = float((oracle_mod.readout_norm(y, g, w)["out"] * dout).sum())
            arr[idx] = old - h
            lm = float((oracle_mod.readout_norm(y, g, w)["out"] * dout).sum())
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert np.abs(r[name] - fd).max() <= 1e-7 * max(1.0, np.abs(fd).max()), name


def test_fwd_bwd_norm_compose(oracle_mod):
    """fwd_norm / bwd_norm: the recurrence's gradients at dy = the norm's dy
    (checked against a central difference of the whole block in one
    direction of W)."""
    x = make_inputs(1, 4, 2, 8, 4, "f32", 21, with_dy=True, norm=True)
    args = [_np(x[n]) for n in ("q", "k", "v", "f", "W", "w_r")]
    g, w, dout = _np(x["g"]), _np(x["w_norm"]), _np(x["dy"])
    r = oracle_mod.bwd_norm(*args, g, w, dout)
    dirW = np.random.default_rng(0).normal(size=args[4].shape)
    h = 1e-6

    def L(W):
        a = list(args)
        a[4] = W
        return float((oracle_mod.fwd_norm(*a, g, w)["out"] * dout).sum())
    fd = (L(args[4] + h * dirW) - L(args[4] - h * dirW)) / (2 * h)
    assert abs(fd - float((r["dW"] * dirW).sum())) <= 1e-7 * max(1.0, abs(fd))
