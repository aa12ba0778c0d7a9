"""bench.py's roofline accounting (CPU): the fractions it prints follow from
the stated work counts and the measured peaks, so they can be checked
without a GPU."""
import sys

import pytest

from non_linear_matrix_gb300.inputs import WORKLOADS


@pytest.fixture(scope="module")
def bench():
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = argv
    return b


PEAKS = {"hbm_gbs": 6698.8, "bf16_tflops": 1939.7, "sm_max_mhz": 2070.0, "source": "measured"}


def test_forward_rooflines(bench):
    w = WORKLOADS["fwd_bf16_b64_t4096_n32"]
    ms = 2.78
    north, alu = bench._roofline(w, ms, PEAKS, 5.5e8)
    th = w.B * w.T * w.N
    # the metric's form: max(tensor, HBM) + serial, as throughput
    flops = th * (2 * w.K * w.V * w.V + 4 * w.K * w.V)
    t_tensor = flops / (PEAKS["bf16_tflops"] * 1e12) * 1e3
    t_serial = w.T * bench.STEP_LATENCY_CLK / (PEAKS["sm_max_mhz"] * 1e6) * 1e3
    assert north["t_tensor_ms"] == pytest.approx(t_tensor)
    assert north["t_serial_ms"] == pytest.approx(t_serial)
    t_roof = max(north["t_tensor_ms"], north["t_hbm_ms"]) + t_serial
    assert north["t_roof_ms"] == pytest.approx(t_roof)
    assert north["frac"] == pytest.approx(t_roof / ms)
    assert north["achieved"] / north["peak"] == pytest.approx(north["frac"])
    assert north["achieved"] == pytest.approx(th / (ms * 1e-3))
    assert north["met"] is False and north["target_frac"] == 0.5
    # the SFU form: K*V tanh per token x head at 16 per clock per SM
    peak = bench.NUM_SMS * 16 * PEAKS["sm_max_mhz"] * 1e6
    assert alu["units_per_launch"] == th * w.K * w.V
    assert alu["frac"] == pytest.approx(th * w.K * w.V / (ms * 1e-3) / peak)
    # the ceiling the SFU puts on the metric's fraction
    assert north["frac_ceiling_sfu"] == pytest.approx(t_roof / (th * w.K * w.V / peak * 1e3))
    assert north["frac_ceiling_sfu"] < 0.5


def test_backward_counts_one_recompute(bench):
    w = WORKLOADS["fwdbwd_bf16_b8_t4096_n32"]
    r = bench._fwdbwd_summary(w, 1, 20, 2.37, 0.58, 1.79, PEAKS, 2)
    th = w.B * w.T * w.N
    alu = r["roofline_alu"]
    assert alu["units_per_launch"] == th * w.K * w.V          # the method's work
    assert alu["design_tanh_per_launch"] == 2 * th * w.K * w.V  # this implementation's
    assert alu["design_frac"] == pytest.approx(2 * alu["frac"])
    bwd = r["roofline_bwd"]
    # algorithmic bytes of the backward at bf16: q, k, v, dy, f, checkpoints,
    # W, w_r read; dq, dk (fp32), dv, df, dW, dw_r written
    nck = w.T // w.ckpt_every
    reads = w.B * w.T * 2 * w.K * 2 + th * (2 * w.V * 2 + 2) + w.B * w.N * nck * w.K * w.V * 4 + \
        w.N * (w.V * w.V + w.V) * 2
    writes = w.B * w.T * 2 * w.K * 4 + th * (w.V * 4 + 4) + w.N * (w.V * w.V + w.V) * 4
    assert bwd["algorithmic_bytes"] == reads + writes
    assert bwd["frac"] == pytest.approx(bwd["achieved"] / bwd["peak"])
    step = r["roofline"]
    assert step["t_serial_ms"] == pytest.approx(
        (2 * w.T + w.ckpt_every) * bench.STEP_LATENCY_CLK / (PEAKS["sm_max_mhz"] * 1e6) * 1e3)


def test_clock_samples_go_to_a_temporary_file(bench):
    import os
    import tempfile
    c = bench.ClockSampler(0)
    try:
        assert os.path.dirname(c.path) == tempfile.gettempdir()
        assert "gpurun_out" not in c.path
    finally:
        os.unlink(c.path)
