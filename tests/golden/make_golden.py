"""Writes the stored expected values under tests/golden/ from the fp64 oracle.

The pages print no numeric worked example for the recurrence, so every value
stored here is the oracle's (this script calls only ``oracle`` and the
seeded input generator).  The oracle itself is pinned by
tests/test_oracle_pins.py; the fixtures freeze its outputs on small cases so
that a later change to its arithmetic shows up as a diff, and give the GPU
tests a comparison that needs no oracle build.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from non_linear_matrix_gb300.inputs import make_inputs  # noqa: E402

# name -> (B, T, N, K, V, dtype, seed, options)
CASES = {
    "plain_f32_b1_t12_n2_k16_v16": (1, 12, 2, 16, 16, "f32", 501, {}),
    "plain_bf16_b1_t12_n2_k16_v16": (1, 12, 2, 16, 16, "bf16", 502, {}),
    "gated_f32_b1_t8_n2_k16_v16": (1, 8, 2, 16, 16, "f32", 503, {"gated": True}),
    "grouped_f32_b1_t8_n4_k16_v16_nq2": (1, 8, 4, 16, 16, "f32", 504, {"groups": 2}),
    "norm_f32_b1_t8_n2_k16_v16": (1, 8, 2, 16, 16, "f32", 505, {"norm": True}),
}
DIGITS = 12  # significant digits stored


def inputs(name):
    B, T, N, K, V, dtype, seed, opt = CASES[name]
    return make_inputs(B, T, N, K, V, dtype, seed, with_dy=True, **opt)


def expected(name):
    """The oracle's outputs for a case, as float64 arrays."""
    x = inputs(name)
    opt = CASES[name][7]
    base = (x["q"], x["k"], x["v"])
    if opt.get("gated"):
        gi = (x["a"], x["alpha"], x["beta"])
        out = oracle.fwd_gated(*base, *gi, x["W"], x["w_r"])
        out.update(oracle.bwd_gated(*base, *gi, x["W"], x["w_r"], x["dy"]))
    elif opt.get("norm"):
        args = (*base, x["f"], x["W"], x["w_r"], x["g"], x["w_norm"])
        out = oracle.fwd_norm(*args, 1e-6)
        out.update(oracle.bwd_norm(*args, x["dy"], 1e-6))
    else:
        out = oracle.fwd(*base, x["f"], x["W"], x["w_r"])
        out.update(oracle.bwd(*base, x["f"], x["W"], x["w_r"], x["dy"]))
    return out


def _rounded(a):
    return [float("%.*g" % (DIGITS, x)) for x in np.asarray(a, dtype=np.float64).ravel()]


def path(name):
    return os.path.join(HERE, name + ".json")


def main():
    for name in CASES:
        out = expected(name)
        rec = {"case": name, "shapes": {k: list(np.shape(v)) for k, v in sorted(out.items())}, "shape_B_T_N_K_V_dtype_seed": list(CASES[name][:7]),
               "options": CASES[name][7], "source": "oracle (fp64), tests/golden/make_golden.py",
               "digits": DIGITS,
               "values": {k: _rounded(v) for k, v in sorted(out.items())}}
        with open(path(name), "w") as fh:
            json.dump(rec, fh)
            fh.write("\n")
        print(path(name))


if __name__ == "__main__":
    main()
