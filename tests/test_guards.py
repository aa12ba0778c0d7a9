"""Out-of-bounds writes, checked without a sanitizer: every output buffer
handed to the library is a view into a larger allocation whose guard
regions before and after it hold a sentinel pattern, and every input is
compared with a copy afterwards.  After each call the guards and the inputs
must be untouched.  Shapes are ragged on purpose (T not a multiple of the
ring chunk or the checkpoint interval, odd head counts, K = 16 and 128,
V = 32, grouped q/k, the whole-wave plus tail split)."""
import pytest
import torch

from non_linear_matrix_gb300.inputs import decode_state, make_inputs

pytestmark = pytest.mark.gpu

GUARD = 64          # float32 elements on each side (256 bytes, keeps 16-byte alignment)
SENTINEL = -7.25e33


@pytest.fixture(scope="module")
def m2rnn():
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn as m
    return m


class Guarded:
    """Output tensors carved out of guarded buffers."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype=torch.float32):
        n = 1
        for d in shape:
            n *= d
        per = 4 // torch.tensor([], dtype=dtype).element_size()  # elements per float32 slot
        g = GUARD * per
        buf = torch.full((n + 2 * g,), SENTINEL, dtype=dtype, device="cuda")
        self.bufs.append((buf, g, n))
        return buf[g:g + n].view(*shape)

    def check(self, label):
        torch.cuda.synchronize()
        for i, (buf, g, n) in enumerate(self.bufs):
            lo, hi = buf[:g], buf[g + n:]
            ref = torch.full_like(lo, SENTINEL)
            assert torch.equal(lo, ref) and torch.equal(hi, ref), (label, i, tuple(buf.shape))


def _inputs(B, T, N, K, V, dtype, seed, **kw):
    x = make_inputs(B, T, N, K, V, dtype, seed, with_dy=True, **kw)
    g = {n: t.cuda() for n, t in x.items()}
    return g, {n: t.clone() for n, t in g.items()}


def _inputs_unchanged(g, copies, label):
    torch.cuda.synchronize()
    for n in g:
        assert torch.equal(g[n], copies[n]), (label, n)


@pytest.mark.parametrize("B,T,N,K,V,dtype,C,Nq", [
    (3, 77, 5, 64, 16, "bf16", 24, 1),
    (2, 41, 3, 16, 16, "f32", 16, 1),
    (2, 53, 4, 128, 16, "bf16", 64, 2),
    (2, 35, 3, 64, 32, "bf16", 8, 1),
    (41, 40, 32, 64, 16, "bf16", 16, 4),   # whole-wave + tail launches
])
def test_fwd_bwd_write_only_their_outputs(m2rnn, B, T, N, K, V, dtype, C, Nq):
    g, copies = _inputs(B, T, N, K, V, dtype, 17 + T, groups=Nq)
    G = Guarded()
    td = g["v"].dtype
    nck = -(-T // C)
    qk = tuple(g["q"].shape)
    out = {"y": G((B, T, N, V), td), "HT": G((B, N, K, V)), "ckpt": G((B, N, nck, K, V))}
    y, HT, ck = m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=C, out=out)
    G.check("fwd")
    gout = {"dq": G(qk), "dk": G(qk), "dv": G((B, T, N, V)), "df": G((B, T, N)),
            "dW": G((N, V, V)), "dw_r": G((N, V)), "dH0": G((B, N, K, V)),
            "dckpt": G((B, N, nck, K, V))}
    first = None
    for ckpt in (ck, None):  # caller checkpoints, and recomputed into the workspace
        r = m2rnn.bwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"], ckpt=ckpt,
                      ckpt_every=C, want_dH0=True, want_dckpt=True, out=gout)
        G.check(f"bwd ckpt={'given' if ckpt is not None else 'recomputed'}")
        if first is None:
            first = {n: t.clone() for n, t in r.items()}
    # The recomputed checkpoints come from the same forward kernel, so the two
    # passes differ only in the order of the atomic head and slice sums.
    for n, t in r.items():
        ref = first[n].double()
        err = (t.double() - ref).norm() / ref.norm().clamp_min(1e-30)
        assert err < 1e-5, (n, float(err))
    _inputs_unchanged(g, copies, "fwd/bwd")
    st, _ = m2rnn.device_status()
    assert st == 0


@pytest.mark.parametrize("G", ["4", "14"])
def test_wave_kernel_writes_only_its_outputs(m2rnn, monkeypatch, G):
    """The one-wave forward kernel (CTAs across two batch items with G = 4
    of N = 6 heads; with G = 14 of N = 16 also a last CTA of 6 heads) with
    y, H_T and checkpoints in guarded buffers."""
    monkeypatch.setenv("M2RNN_FWD_WAVE", "1")
    monkeypatch.setenv("M2RNN_FWD_WAVE_G", G)
    B, T, N, C = (5, 77, 6, 24) if G == "4" else (3, 45, 16, 16)
    g, copies = _inputs(B, T, N, 64, 16, "bf16", 90 + T)
    Gd = Guarded()
    nck = -(-T // C)
    out = {"y": Gd((B, T, N, 16), torch.bfloat16), "HT": Gd((B, N, 64, 16)),
           "ckpt": Gd((B, N, nck, 64, 16))}
    m2rnn.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], ckpt_every=C, out=out)
    Gd.check(f"wave G={G}")
    _inputs_unchanged(g, copies, "wave")
    st, _ = m2rnn.device_status()
    assert st == 0


@pytest.mark.parametrize("B,T,N", [(3, 45, 6), (41, 40, 32)])  # the second splits the forward
def test_gated_and_norm_write_only_their_outputs(m2rnn, B, T, N):
    K, V, C = 64, 16, 16
    g, copies = _inputs(B, T, N, K, V, "bf16", 5, gated=True, norm=True)
    G = Guarded()
    td = g["v"].dtype
    nck = -(-T // C)
    gate = (g["a"], g["alpha"], g["beta"])
    r = m2rnn.fwd_norm(g["q"], g["k"], g["v"], None, g["W"], g["w_r"], g["g"], g["w_norm"], 1e-6,
                       gate=gate, ckpt_every=C,
                       out={"y": G((B, T, N, V), td), "out": G((B, T, N, V), td),
                            "rstd": G((B, T)), "HT": G((B, N, K, V)),
                            "ckpt": G((B, N, nck, K, V))})
    G.check("fwd_norm gated")
    gout = {"dq": G((B, T, K)), "dk": G((B, T, K)), "dv": G((B, T, N, V)), "da": G((B, T, N)),
            "dalpha": G((N,)), "dbeta": G((N,)), "dW": G((N, V, V)), "dw_r": G((N, V)),
            "dg": G((B, T, N, V)), "dw_norm": G((N, V)), "dH0": G((B, N, K, V))}
    for ckpt in (r["ckpt"], None):  # given, and recomputed (a checkpoint-only forward)
        m2rnn.bwd_norm(g["q"], g["k"], g["v"], None, g["W"], g["w_r"], g["g"], g["w_norm"],
                       r["y"], r["rstd"], g["dy"], ckpt=ckpt, gate=gate, ckpt_every=C,
                       want_dH0=True, out=gout)
        G.check(f"bwd_norm gated ckpt={'given' if ckpt is not None else 'recomputed'}")
    gg = {"dq": G((B, T, K)), "dk": G((B, T, K)), "dv": G((B, T, N, V)), "da": G((B, T, N)),
          "dalpha": G((N,)), "dbeta": G((N,)), "dW": G((N, V, V)), "dw_r": G((N, V))}
    m2rnn.bwd_gated(g["q"], g["k"], g["v"], *gate, g["W"], g["w_r"], g["dy"], ckpt=r["ckpt"],
                    ckpt_every=C, out=gg)
    G.check("bwd_gated")
    _inputs_unchanged(g, copies, "gated/norm")


@pytest.mark.parametrize("K,V,dtype", [(64, 16, "bf16"), (128, 32, "f32"), (16, 16, "bf16")])
def test_decode_writes_only_its_outputs(m2rnn, K, V, dtype):
    B, N = 7, 5
    x = make_inputs(B, 1, N, K, V, dtype, 23)
    g = {n: (t[:, 0].contiguous() if n in ("q", "k", "v", "f") else t).cuda() for n, t in x.items()}
    copies = {n: t.clone() for n, t in g.items()}
    H = decode_state(B, N, K, V, 3).cuda()
    Hc = H.clone()
    G = Guarded()
    y, Ho = m2rnn.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], H,
                         H_out=G((B, N, K, V)), y=G((B, N, V), g["v"].dtype))
    G.check("decode")
    assert torch.equal(H, Hc)
    _inputs_unchanged(g, copies, "decode")
