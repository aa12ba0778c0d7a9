"""Stored expected values (tests/golden/*.json, written from the oracle by
tests/golden/make_golden.py; the pages print no numeric worked example).

CPU: the oracle still reproduces every stored value (to the 12 stored
digits), so a change to its arithmetic shows up here and must come with
regenerated fixtures.  GPU: the library's outputs on the same seeded inputs
against the stored values, with the parity tolerances (max |.| 2e-3 / 2e-2
on y, H_T and out for fp32 / bf16 operands; relative L2 1e-2 on gradients).
"""
import json
import os
import sys

import numpy as np
import pytest
import torch

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)
import make_golden  # noqa: E402

CASES = sorted(make_golden.CASES)


def _stored(name):
    with open(make_golden.path(name)) as fh:
        rec = json.load(fh)
    return {k: np.asarray(v).reshape(rec["shapes"][k]) for k, v in rec["values"].items()}


@pytest.mark.parametrize("name", CASES)
def test_oracle_reproduces_stored_values(oracle_mod, name):
    stored = _stored(name)
    now = make_golden.expected(name)
    assert sorted(stored) == sorted(now)
    for k, v in now.items():
        scale = max(1e-300, float(np.abs(v).max()))
        assert np.abs(np.asarray(v) - stored[k]).max() <= 1e-11 * scale, (name, k)


@pytest.mark.gpu
@pytest.mark.parametrize("name", CASES)
def test_gpu_matches_stored_values(name):
    import __graft_entry__
    __graft_entry__.build()
    from non_linear_matrix_gb300 import m2rnn
    x = make_golden.inputs(name)
    g = {n: t.cuda() for n, t in x.items()}
    opt = make_golden.CASES[name][7]
    dtype = make_golden.CASES[name][5]
    base = (g["q"], g["k"], g["v"])
    if opt.get("gated"):
        gi = (g["a"], g["alpha"], g["beta"])
        y, HT, ck = m2rnn.fwd_gated(*base, *gi, g["W"], g["w_r"], ckpt_every=4)
        gr = m2rnn.bwd_gated(*base, *gi, g["W"], g["w_r"], g["dy"], ckpt=ck, ckpt_every=4)
        got = {"y": y, "HT": HT, **gr}
    elif opt.get("norm"):
        r = m2rnn.fwd_norm(*base, g["f"], g["W"], g["w_r"], g["g"], g["w_norm"], 1e-6,
                           ckpt_every=4)
        gr = m2rnn.bwd_norm(*base, g["f"], g["W"], g["w_r"], g["g"], g["w_norm"], r["y"],
                            r["rstd"], g["dy"], ckpt=r["ckpt"], ckpt_every=4)
        got = {"y": r["y"], "HT": r["HT"], "out": r["out"], **gr}
    else:
        y, HT, ck = m2rnn.fwd(*base, g["f"], g["W"], g["w_r"], ckpt_every=4)
        gr = m2rnn.bwd(*base, g["f"], g["W"], g["w_r"], g["dy"], ckpt=ck, ckpt_every=4)
        got = {"y": y, "HT": HT, **gr}
    torch.cuda.synchronize()
    st, _ = m2rnn.device_status()
    assert st == 0
    ref = _stored(name)
    tol = 2e-3 if dtype == "f32" else 2e-2
    for k in ("y", "HT", "out"):
        if k in got:
            assert np.abs(got[k].float().cpu().double().numpy() - ref[k]).max() <= tol, (name, k)
    for k in got:
        if k in ("y", "HT", "out") or k not in ref:
            continue
        a = got[k].cpu().double().numpy()
        den = np.linalg.norm(ref[k])
        rel = np.linalg.norm(a - ref[k]) / den if den > 0 else np.linalg.norm(a)
        assert rel <= 1e-2, (name, k, rel)
