"""Throughput benchmark of the M2RNN recurrence on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one forward pass of the recurrence over the workload's whole batch
(default: B=64, T=4096, N=32, K=64, V=16, bf16 inputs, fp32 state: the
throughput shape), through the C ABI, with inputs resident in HBM.  The
inputs (~0.32 GB) exceed the 129 MB L2, so no flush is needed between steps;
workloads whose working set fits in L2 write a buffer of twice its size
before every timed step (outside the step's events).
Metric: tokens x heads per second (B*T*N / step time).

Extra keys on the JSON line:
  roofline      the metric's own roofline: the dominant kernel's time against
                max(t_tensor, t_HBM) + t_serial (tensor flops at the measured
                bf16 peak, algorithmic bytes at the measured copy bandwidth,
                T dependent steps at the measured step latency); achieved and
                peak are tokens x heads per second, frac = t_roof / t_kernel.
                While tanh runs on the SFU this fraction cannot exceed about
                0.22 at B=64, T=4096, N=32 (the SFU alone needs 1.71 ms there);
  roofline_alu  the same kernel against the bound it actually meets: the SFU
                tanh rate (K*V tanh per token x head at 16 tanh/clk/SM);
  cpu_baseline  the fp64 oracle (test infrastructure) on a bounded sample of
                the same workload on the host cores;
  e2e           the same metric with host (pinned) inputs: host->device
                copies, the C-ABI call and the device->host copy of y inside
                the timed region;
  clocks        nvidia-smi SM clock samples taken during the timed region;
  fwd_bwd       the backward rows of the path: a forward + backward step of
                B=8, T=4096, N=32 (checkpoints every 64 steps) with its own
                roofline, roofline_bwd, roofline_alu and cpu_baseline (the
                oracle's forward + backward on a bounded sample).
For N > 1 (torchrun) every rank runs its own batch on its own GPU (weak
scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from non_linear_matrix_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

METRIC = ("M2RNN fwd(+bwd) tokens\u00d7heads/s on 1 GB300; % of roofline "
          "(tensor/HBM/serial bound)")
UNIT = "tokens*heads/s"
DEFAULT_WORKLOAD = "fwd_bf16_b64_t4096_n32"
L2_BYTES = 129 * 10**6  # GB300 L2

# Rates measured on this machine's GB300 by non_linear_matrix_gb300/csrc/m2rnn_microbench.cu
# (profiles/microbench_gb300.txt): tanh.approx results per clock per SM (f32,
# bf16x2 and f16x2 alike) and the dependent latency of one recurrence step of
# a 16x16 state tile (mma -> tanh -> blend -> bf16 repack) on one warp.
SFU_TANH_PER_CLK_PER_SM = 16.0
STEP_LATENCY_CLK = 113.3
NUM_SMS = 152
SM_MAX_MHZ = 2070.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "sm_max_mhz": float(d.get("sm_max_mhz", SM_MAX_MHZ)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, sm_max_mhz=SM_MAX_MHZ, source="fallback")


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: per-GPU work is fixed)."""
    return base_seed + 1000 * rank


def max_over_ranks(value: float, device: str = "cuda") -> float:
    """The slowest rank's time (the job finishes when the last rank does)."""
    import torch.distributed as dist
    t = torch.tensor([float(value)], device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms_slowest: float) -> float:
    """Whole-job units per second: all ranks' units over the slowest time."""
    return world * units_per_rank / (ms_slowest * 1e-3)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"m2rnn_clocks_gpu{gpu_index}_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            try:
                os.unlink(self.path)
            except OSError:
                pass
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _tensor_hbm_serial(w, peaks):
    """Terms of the metric's roofline for one forward launch: algorithmic
    bytes and flops, and t_tensor, t_hbm, t_serial in ms."""
    th = w.th
    es = 2 if w.dtype == "bf16" else 4
    # algorithmic bytes: v, f, y per token x head; q, k per token; W, w_r per head; H_T
    bytes_per_launch = th * (2 * w.V * es + es) + w.B * w.T * 2 * w.K * es + \
        w.N * (w.V * w.V + w.V) * es + w.B * w.N * w.K * w.V * 4
    flops_per_launch = th * (2 * w.K * w.V * w.V + 4 * w.K * w.V)
    t_hbm = bytes_per_launch / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_tensor = flops_per_launch / (peaks["bf16_tflops"] * 1e12) * 1e3
    t_serial = w.T * STEP_LATENCY_CLK / (peaks["sm_max_mhz"] * 1e6) * 1e3
    return bytes_per_launch, flops_per_launch, t_tensor, t_hbm, t_serial


def _peak_tanh(peaks):
    return NUM_SMS * SFU_TANH_PER_CLK_PER_SM * peaks["sm_max_mhz"] * 1e6


def _roofline(w, kernel_ms, peaks, traffic):
    """(the metric's roofline, the SFU roofline) of the forward kernel."""
    nbytes, flops, t_tensor, t_hbm, t_serial = _tensor_hbm_serial(w, peaks)
    t_roof = max(t_hbm, t_tensor) + t_serial
    tanh_per_launch = w.th * w.K * w.V
    peak_tanh = _peak_tanh(peaks)
    t_sfu = tanh_per_launch / peak_tanh * 1e3
    achieved_tanh = tanh_per_launch / (kernel_ms * 1e-3)
    src = ("measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
           else "fallback 6.8 TB/s, 1.9 PFLOP/s")
    north = {
        "bound": "tensor+serial" if t_tensor >= t_hbm else "hbm+serial",
        "form": "max(t_tensor, t_hbm) + t_serial",
        "achieved": w.th / (kernel_ms * 1e-3), "peak": w.th / (t_roof * 1e-3),
        "unit": "tokens*heads/s", "frac": t_roof / kernel_ms, "traffic": traffic,
        "traffic_source": _TRAFFIC_SOURCE if traffic is not None else None,
        "t_tensor_ms": t_tensor, "t_hbm_ms": t_hbm, "t_serial_ms": t_serial,
        "t_roof_ms": t_roof, "frac_max_form": max(t_hbm, t_tensor, t_serial) / kernel_ms,
        "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "peaks": src,
        "target_frac": 0.5, "met": t_roof / kernel_ms >= 0.5,
        "frac_ceiling_sfu": t_roof / t_sfu,
        "note": ("tanh runs on the SFU (16/clk/SM measured), which alone needs "
                 f"{t_sfu:.3f} ms here, so this fraction cannot exceed "
                 f"{t_roof / t_sfu:.2f} on this hardware"),
    }
    alu = {"bound": "alu", "achieved": achieved_tanh / 1e12, "peak": peak_tanh / 1e12,
           "unit": "Ttanh/s", "frac": achieved_tanh / peak_tanh, "traffic": traffic,
           "traffic_source": _TRAFFIC_SOURCE if traffic is not None else None,
           "units_per_launch": tanh_per_launch,
           "peak_basis": f"SFU tanh {SFU_TANH_PER_CLK_PER_SM:g}/clk/SM (measured) x {NUM_SMS} SMs x "
                         f"{peaks['sm_max_mhz']:g} MHz"}
    return north, alu


_TRAFFIC_SOURCE = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from a committed "
                   "ncu capture of the same kernel source (sha256 match), not from this run")


def _traffic_record(fname, src_files, workload):
    """DRAM bytes per launch from a committed ncu summary under profiles/,
    if every kernel source it was captured from is unchanged."""
    path = os.path.join(ROOT, "profiles", fname)
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for f in src_files:
            h.update(open(os.path.join(ROOT, "non_linear_matrix_gb300", "csrc", f), "rb").read())
        if rec.get("kernel_source_sha256") == h.hexdigest() and rec.get("workload") == workload:
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


def _traffic(w):
    """DRAM bytes of one forward launch set (committed capture)."""
    return _traffic_record("fwd_dram_traffic.json", ["m2rnn_fwd.cu"], w.name)


def _bwd_traffic(w):
    """DRAM bytes of one backward launch (committed capture)."""
    return _traffic_record("bwd_dram_traffic.json", ["m2rnn_bwd_pipe.cu"], w.name)


def _oracle_rate(w, budget_s: float, seed_offset: int = 0):
    """fp64 oracle on a bounded sample: (th/s, description, threads, seconds)."""
    import oracle
    from non_linear_matrix_gb300.inputs import make_inputs
    oracle.build()
    threads = oracle.threads()
    heads = max(1, min(w.N, threads))

    def run(T_):
        x = make_inputs(1, T_, heads, w.K, w.V, w.dtype, w.seed + seed_offset, w.f_mean,
                        with_dy=w.backward, gated=w.gated, norm=w.norm)
        t0 = time.perf_counter()
        if w.norm:  # the oracle's block: recurrence + readout epilogue (+ backward)
            oracle.fwd_norm(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["g"],
                            x["w_norm"], 1e-6)
            if w.backward:
                oracle.bwd_norm(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["g"],
                                x["w_norm"], x["dy"], 1e-6)
        elif w.gated:  # the oracle's gated forward (+ backward through the gate)
            gi = (x["a"], x["alpha"], x["beta"])
            oracle.fwd_gated(x["q"], x["k"], x["v"], *gi, x["W"], x["w_r"])
            if w.backward:
                oracle.bwd_gated(x["q"], x["k"], x["v"], *gi, x["W"], x["w_r"], x["dy"])
        elif w.backward:  # forward + BPTT backward (the oracle's backward reruns the forward)
            oracle.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
            oracle.bwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], x["dy"])
        else:
            oracle.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"])
        return time.perf_counter() - t0

    T_probe = min(w.T, 256)
    rate = heads * T_probe / max(run(T_probe), 1e-6)
    T_s = int(max(16, min(w.T, budget_s * rate / heads)))
    dt = run(T_s)
    what = "fwd+bwd" if w.backward else "fwd"
    desc = f"{what} of 1 batch item x {heads} heads x {T_s} steps of {w.name} (K={w.K}, V={w.V})"
    return heads * T_s / dt, desc, threads, dt


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return
    per_step_budget = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    rate_fn = _oracle_decode_rate if w.decode else _oracle_rate
    for _ in range(args.warmup):
        rate_fn(w, per_step_budget / 4)
    times, th = [], 0.0
    desc, threads = "", 0
    for _ in range(args.steps):
        rate, desc, threads, dt = rate_fn(w, per_step_budget)
        times.append(dt)
        th += rate * dt
    value = th / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "N": w.N, "K": w.K, "V": w.V,
                       "inputs": w.dtype, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def _count_launches(fn):
    """Kernels of this library one call of fn launches (torch profiler)."""
    try:
        from torch.profiler import ProfilerActivity, profile
        n = 0
        for _ in range(2):  # the first session may start recording late
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                fn()
                torch.cuda.synchronize()
            n = max(n, sum(1 for e in prof.events()
                           if e.device_type == torch.autograd.DeviceType.CUDA
                           and "m2rnn" in e.name))
        return n
    except Exception:  # profiler unavailable
        return None


class Runner:
    """Preallocated buffers and the step of one workload on this rank."""

    def __init__(self, w, m2rnn, rank):
        from non_linear_matrix_gb300.inputs import make_inputs
        self.w, self.m = w, m2rnn
        seed = rank_seed(w.seed, rank)
        self.x = make_inputs(w.B, w.T, w.N, w.K, w.V, w.dtype, seed, w.f_mean,
                             with_dy=w.backward, gated=w.gated, norm=w.norm)
        self.g = {n: t.cuda() for n, t in self.x.items()}
        g = self.g
        f32 = dict(device="cuda", dtype=torch.float32)
        self.out = {"y": torch.empty_like(g["v"]),
                    "HT": torch.empty(w.B, w.N, w.K, w.V, **f32)}
        if w.norm:
            self.out.update(out=torch.empty_like(g["v"]), rstd=torch.empty(w.B, w.T, **f32))
        if w.backward:
            nck = -(-w.T // w.ckpt_every)
            self.out["ckpt"] = torch.empty(w.B, w.N, nck, w.K, w.V, **f32)
            self.gout = {"dq": torch.empty(w.B, w.T, w.K, **f32),
                         "dk": torch.empty(w.B, w.T, w.K, **f32),
                         "dv": torch.empty(w.B, w.T, w.N, w.V, **f32),
                         "dW": torch.empty(w.N, w.V, w.V, **f32),
                         "dw_r": torch.empty(w.N, w.V, **f32)}
            if w.norm:
                self.gout.update(dg=torch.empty(w.B, w.T, w.N, w.V, **f32),
                                 dw_norm=torch.empty(w.N, w.V, **f32))
            if w.gated:
                self.gout.update(da=torch.empty(w.B, w.T, w.N, **f32),
                                 dalpha=torch.empty(w.N, **f32), dbeta=torch.empty(w.N, **f32))
            else:
                self.gout["df"] = torch.empty(w.B, w.T, w.N, **f32)
            shape = m2rnn.make_shape(g["q"], g["v"], w.ckpt_every)
            ws = (m2rnn.lib().m2rnn_bwd_norm_workspace_size(ctypes.byref(shape), 1) if w.norm
                  else m2rnn.bwd_workspace_size(shape, True))
            self.ws = torch.empty(max(16, ws), device="cuda", dtype=torch.uint8)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        # bytes a step reads or writes (all its device tensors); below the L2
        # size the timed steps are separated by an L2 flush
        tensors = list(self.g.values()) + list(self.out.values())
        if w.backward:
            tensors += list(self.gout.values()) + [self.ws]
        self.working_set = sum(t.numel() * t.element_size() for t in tensors)
        self.flush = (torch.empty(2 * L2_BYTES, device="cuda", dtype=torch.uint8)
                      if self.working_set <= L2_BYTES else None)

    def l2_note(self):
        mb = self.working_set / 1e6
        if self.flush is None:
            return "working set %.0f MB larger than L2 (129 MB); no flush" % mb
        return ("working set %.0f MB fits in L2 (129 MB): a %.0f MB buffer is written "
                "before every timed step, outside its events" % (mb, self.flush.numel() / 1e6))

    def fwd(self):
        g = self.g
        if self.w.norm:
            self.m.fwd_norm(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["g"], g["w_norm"],
                            1e-6, out=self.out, ckpt_every=self.w.ckpt_every)
        elif self.w.gated:
            self.m.fwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                             g["w_r"], out=self.out, ckpt_every=self.w.ckpt_every)
        else:
            self.m.fwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], out=self.out,
                       ckpt_every=self.w.ckpt_every)

    def bwd(self):
        g = self.g
        if self.w.norm:
            o = self.out
            self.m.bwd_norm(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["g"],
                            g["w_norm"], o["y"], o["rstd"], g["dy"], ckpt=o["ckpt"],
                            ckpt_every=self.w.ckpt_every, out=self.gout, workspace=self.ws)
        elif self.w.gated:
            self.m.bwd_gated(g["q"], g["k"], g["v"], g["a"], g["alpha"], g["beta"], g["W"],
                             g["w_r"], g["dy"], ckpt=self.out["ckpt"],
                             ckpt_every=self.w.ckpt_every, out=self.gout, workspace=self.ws)
        else:
            self.m.bwd(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], g["dy"],
                       ckpt=self.out["ckpt"], ckpt_every=self.w.ckpt_every, out=self.gout,
                       workspace=self.ws)

    def step(self):
        self.fwd()
        if self.w.backward:
            self.bwd()

    def timed(self, steps, stream):
        """Times `steps` steps; returns (ms/step, fwd ms/step, bwd ms/step)."""
        e0, e1, e2 = self.ev
        tot = fw = bw = 0.0
        if self.flush is not None:  # L2-resident working set: flush, then time each step
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
            for a, b, c in evs:
                self.flush.fill_(1)
                a.record(stream)
                self.fwd()
                b.record(stream)
                if self.w.backward:
                    self.bwd()
                c.record(stream)
            torch.cuda.synchronize()
            for a, b, c in evs:
                fw += a.elapsed_time(b)
                bw += b.elapsed_time(c)
            return (fw + bw) / steps, fw / steps, bw / steps
        if not self.w.backward:
            e0.record(stream)
            for _ in range(steps):
                self.fwd()
            e1.record(stream)
            torch.cuda.synchronize()
            tot = fw = e0.elapsed_time(e1)
        else:
            # per-step events split fwd and bwd; all steps are queued back to
            # back and read after one synchronize, so no step waits for the
            # host to enqueue it
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
            for a, b, c in evs:
                a.record(stream)
                self.fwd()
                b.record(stream)
                self.bwd()
                c.record(stream)
            torch.cuda.synchronize()
            for a, b, c in evs:
                fw += a.elapsed_time(b)
                bw += b.elapsed_time(c)
            tot = evs[0][0].elapsed_time(evs[-1][2])
        return tot / steps, fw / steps, bw / steps


class DecodeRunner:
    """Single-step decode of B sequences: the state stays in HBM and is
    updated in place by every step."""

    def __init__(self, w, m2rnn, rank):
        from non_linear_matrix_gb300.inputs import decode_state, make_inputs
        self.w, self.m = w, m2rnn
        seed = rank_seed(w.seed, rank)
        x = make_inputs(w.B, 1, w.N, w.K, w.V, w.dtype, seed, w.f_mean)
        self.x = {n: (t[:, 0].contiguous() if n in ("q", "k", "v", "f") else t)
                  for n, t in x.items()}
        self.g = {n: t.cuda() for n, t in self.x.items()}
        self.H = decode_state(w.B, w.N, w.K, w.V, seed).cuda()
        self.out = {"y": torch.empty_like(self.g["v"])}
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(self):
        g = self.g
        self.m.decode(g["q"], g["k"], g["v"], g["f"], g["W"], g["w_r"], self.H, H_out=self.H,
                      y=self.out["y"])

    def timed(self, steps, stream):
        e0, e1, _ = self.ev
        e0.record(stream)
        for _ in range(steps):
            self.step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        return ms, ms, 0.0


def _decode_roofline(w, ms, peaks):
    """Decode is bound by HBM: the state is read and written once per step."""
    es = 2 if w.dtype == "bf16" else 4
    heads = w.B * w.N
    bytes_step = heads * (2 * w.K * w.V * 4 + 2 * w.V * es + es) + w.B * 2 * w.K * es + \
        w.N * (w.V * w.V + w.V) * es
    achieved = bytes_step / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes": bytes_step,
            "peak_basis": ("measured copy bandwidth (MEASURED_PEAKS.json)"
                           if peaks["source"] == "measured" else "fallback 6.8 TB/s")}


def _oracle_decode_rate(w, budget_s: float):
    """fp64 oracle at T = 1 on a sample of sequences: (units/s, desc, threads)."""
    import oracle
    from non_linear_matrix_gb300.inputs import decode_state, make_inputs
    oracle.build()
    threads = oracle.threads()

    def run(Bs):
        x = make_inputs(Bs, 1, w.N, w.K, w.V, w.dtype, w.seed, w.f_mean)
        H = decode_state(Bs, w.N, w.K, w.V, w.seed)
        t0 = time.perf_counter()
        oracle.fwd(x["q"], x["k"], x["v"], x["f"], x["W"], x["w_r"], H0=H)
        return time.perf_counter() - t0

    Bp = min(w.B, 64)
    rate = Bp * w.N / max(run(Bp), 1e-6)
    Bs = int(max(1, min(w.B, budget_s * rate / w.N)))
    dt = run(Bs)
    desc = f"one decode step of {Bs} sequences x {w.N} heads of {w.name} (K={w.K}, V={w.V})"
    return Bs * w.N / dt, desc, threads, dt


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-bwd-line", action="store_true",
                    help="skip the nested fwd+bwd measurement of the default line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from non_linear_matrix_gb300 import m2rnn
    m2rnn.lib()
    stream = torch.cuda.current_stream()

    def check_status(where):
        st, detail = m2rnn.device_status(clear=True)
        if st != 0:
            raise RuntimeError(f"device status {st} ({detail}) {where}")

    run = DecodeRunner(w, m2rnn, rank) if w.decode else Runner(w, m2rnn, rank)
    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    check_status("after warm-up")
    launches = _count_launches(run.step)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms, fwd_ms, bwd_ms = run.timed(args.steps, stream)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    check_status("in the timed region")
    ms_max = max_over_ranks(ms)
    value = job_throughput(w.th, world, ms_max)

    # End to end through the public API with host inputs.
    e2e = None
    if not args.no_e2e:
        # decode: the step's inputs are q, k, v, f (the carried state and the
        # weights stay on the device); every step returns y
        hx = {n: t.pin_memory() for n, t in run.x.items()
              if (not w.decode or n in ("q", "k", "v", "f")) and not (w.gated and n == "f")}
        res = [run.out["y"]] if not w.backward else [run.gout[n] for n in sorted(run.gout)]
        hres = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in res]
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for t in hres)

        # at least 50 pipelined steps: the first batch's copy in and the
        # last batch's copy out are not overlapped, and over 20 steps that
        # fill and drain alone add ~0.15 ms per step at B=64
        e_steps = max(50, min(args.steps, 200))
        if w.decode:
            # one decode stream: each step needs the state the previous step wrote
            def e2e_step():
                for n in hx:
                    run.g[n].copy_(hx[n], non_blocking=True)
                run.step()
                for h, r in zip(hres, res):
                    h.copy_(r, non_blocking=True)

            for _ in range(2):
                e2e_step()
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            e0, e1, _ = run.ev
            e0.record(stream)
            for _ in range(e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize()
        else:
            # Independent batches: two device buffer sets, so that the next
            # batch's host->device copy and the previous batch's
            # device->host copy run on their own streams while this batch
            # computes (the copies stay inside the timed region).
            sets = [run, Runner(w, m2rnn, rank)]
            outs = [res, [sets[1].out["y"]] if not w.backward
                    else [sets[1].gout[n] for n in sorted(sets[1].gout)]]
            houts = [hres, [torch.empty(r.shape, dtype=r.dtype, pin_memory=True)
                            for r in outs[1]]]
            h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
            ev = lambda: torch.cuda.Event()  # noqa: E731
            in_ready = [ev(), ev()]
            computed = [ev(), ev()]
            copied_out = [ev(), ev()]

            def e2e_run(nsteps, e_start=None, e_end=None):
                if e_start is not None:
                    e_start.record(h2d_s)
                for i in range(nsteps):
                    k = i % 2
                    r = sets[k]
                    if i >= 2:  # buffer set k's previous batch has been consumed
                        h2d_s.wait_event(computed[k])
                    with torch.cuda.stream(h2d_s):
                        for n in hx:
                            r.g[n].copy_(hx[n], non_blocking=True)
                    in_ready[k].record(h2d_s)
                    stream.wait_event(in_ready[k])
                    if i >= 2:  # its previous results have been copied out
                        stream.wait_event(copied_out[k])
                    r.step()
                    computed[k].record(stream)
                    d2h_s.wait_event(computed[k])
                    with torch.cuda.stream(d2h_s):
                        for h, o in zip(houts[k], outs[k]):
                            h.copy_(o, non_blocking=True)
                    copied_out[k].record(d2h_s)
                if e_end is not None:
                    d2h_s.wait_event(computed[(nsteps - 1) % 2])
                    e_end.record(d2h_s)

            e2e_run(4)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            e0, e1, _ = run.ev
            e2e_run(e_steps, e0, e1)
            torch.cuda.synchronize()
            del sets[1]
        e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps)
        e2e = {"value": job_throughput(w.th, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": e_ms,
               "pipelining": ("none (the carried state orders the steps)" if w.decode else
                              "two buffer sets; batch i+1's host->device copy and batch "
                              "i-1's device->host copy overlap batch i's compute")}

    # Nested fwd+bwd measurement (the backward rows of the path).
    nested = None
    if not w.backward and not w.decode and not args.no_bwd_line:
        wb = WORKLOADS["fwdbwd_bf16_b8_t4096_n32"]
        rb = Runner(wb, m2rnn, rank)
        for _ in range(args.warmup):
            rb.step()
        torch.cuda.synchronize()
        check_status("after fwd+bwd warm-up")
        nb_steps = max(3, min(args.steps, 20))
        if world > 1:
            torch.distributed.barrier()
        b_ms, b_fwd, b_bwd = rb.timed(nb_steps, stream)
        check_status("in the fwd+bwd timed region")
        b_ms = max_over_ranks(b_ms)
        peaks = _peaks()
        nested = _fwdbwd_summary(wb, world, nb_steps, b_ms, b_fwd, b_bwd, peaks,
                                 _count_launches(rb.step))
        del rb

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks = _peaks()
    extra = {}
    if w.backward:
        nested_main = _fwdbwd_summary(w, world, args.steps, ms_max, fwd_ms, bwd_ms, peaks,
                                      launches)
        roof = nested_main["roofline"]
        extra = {"roofline_bwd": nested_main["roofline_bwd"],
                 "roofline_alu": nested_main["roofline_alu"]}
    elif w.decode:
        roof = _decode_roofline(w, fwd_ms, peaks)
    else:
        roof, alu = _roofline(w, fwd_ms, peaks, _traffic(w))
        extra = {"roofline_alu": alu}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "N": w.N, "K": w.K, "V": w.V,
                   "inputs": w.dtype, "state": "f32", "global_batch": w.B * world,
                   "seq_len": w.T, "parallelism": f"replicas{world}" if world > 1 else "1 GPU",
                   "step": ("forward + backward" + (" (fused input gate)" if w.gated else "")
                            + (" (readout epilogue: x g, RMSNorm)" if w.norm else "")
                            if w.backward else
                            "decode (one step, state updated in place)" if w.decode else
                            "forward"),
                   "l2": ("state (%.0f MB) larger than L2 (129 MB); no flush"
                          % (w.B * w.N * w.K * w.V * 4 / 1e6) if w.decode else
                          run.l2_note())},
        "roofline": roof, **extra,
        "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches * args.steps if launches is not None else args.steps,
        "gpu_launches_per_step": launches,
    }
    if w.backward:
        line["fwd_ms"], line["bwd_ms"] = fwd_ms, bwd_ms
    if nested is not None:
        line["fwd_bwd"] = nested
    if not args.no_cpu:
        rate, desc, threads, _ = (_oracle_decode_rate(w, 12.0) if w.decode else
                                  _oracle_rate(w, 12.0))
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": desc}
        if nested is not None:  # the fwd+bwd step's own oracle baseline (forward + backward)
            rate, desc, threads, _ = _oracle_rate(WORKLOADS["fwdbwd_bf16_b8_t4096_n32"], 12.0)
            nested["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads,
                                      "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _bwd_terms(w, peaks):
    """Algorithmic bytes and flops of the method's backward for one launch
    (one recompute of every interval from its checkpoint, then the reverse
    sweep), with t_tensor and t_hbm in ms."""
    es = 2 if w.dtype == "bf16" else 4
    th = w.th
    nck = -(-w.T // w.ckpt_every)
    reads = w.B * w.T * 2 * w.K * es + th * (2 * w.V * es + es) + \
        w.B * w.N * nck * w.K * w.V * 4 + w.N * (w.V * w.V + w.V) * es
    writes = w.B * w.T * 2 * w.K * 4 + th * (w.V * 4 + 4) + w.N * (w.V * w.V + w.V) * 4
    # recompute H W, reverse D W^T and H^T D (2 K V^2 each); k v^T, D v, H u, D^T k
    flops = th * (3 * 2 * w.K * w.V * w.V + 8 * w.K * w.V)
    t_hbm = (reads + writes) / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    return reads + writes, flops, t_tensor, t_hbm


def _fwdbwd_summary(w, world, steps, ms, fwd_ms, bwd_ms, peaks, launches):
    """Metric and rooflines of a forward + backward step.

    The method's backward recomputes every interval once from its checkpoint
    (K*V tanh per token x head, like the forward).  This implementation's
    backward recomputes twice (sub-checkpoints, then each sub-interval), so
    it evaluates 2*K*V: reported as design_tanh, not counted as work.
    Serial bound: T forward steps, T reverse steps and one interval of
    recompute before the first reverse step, each at the measured step
    latency."""
    th = w.th * world
    peak_tanh = _peak_tanh(peaks)
    method_tanh, design_tanh = w.th * w.K * w.V, 2 * w.th * w.K * w.V
    fb, ff, ft_tensor, ft_hbm, _ = _tensor_hbm_serial(w, peaks)
    nck = -(-w.T // w.ckpt_every)
    fb += w.B * w.N * nck * w.K * w.V * 4  # checkpoints written by the forward
    ft_hbm = fb / (peaks["hbm_gbs"] * 1e9) * 1e3
    bb, bf, bt_tensor, bt_hbm = _bwd_terms(w, peaks)
    clk = peaks["sm_max_mhz"] * 1e6
    t_ser_bwd = (w.T + w.ckpt_every) * STEP_LATENCY_CLK / clk * 1e3
    t_ser_step = (2 * w.T + w.ckpt_every) * STEP_LATENCY_CLK / clk * 1e3
    t_roof_step = max(ft_tensor + bt_tensor, ft_hbm + bt_hbm) + t_ser_step
    t_roof_bwd = max(bt_tensor, bt_hbm) + t_ser_bwd
    traffic = _bwd_traffic(w)
    achieved = method_tanh / (bwd_ms * 1e-3)
    return {
        "workload": w.name, "value": th / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "steps": steps, "ckpt_every": w.ckpt_every,
        "gpu_launches_per_step": launches,
        "roofline": {
            "bound": "tensor+serial" if ft_tensor + bt_tensor >= ft_hbm + bt_hbm else "hbm+serial",
            "form": "max(t_tensor, t_hbm) + t_serial over the fwd+bwd step",
            "achieved": w.th / (ms * 1e-3), "peak": w.th / (t_roof_step * 1e-3),
            "unit": "tokens*heads/s", "frac": t_roof_step / ms,
            "t_tensor_ms": ft_tensor + bt_tensor, "t_hbm_ms": ft_hbm + bt_hbm,
            "t_serial_ms": t_ser_step, "t_roof_ms": t_roof_step},
        "roofline_bwd": {
            "bound": "tensor+serial" if bt_tensor >= bt_hbm else "hbm+serial",
            "form": "max(t_tensor, t_hbm) + t_serial of the backward kernel",
            "achieved": w.th / (bwd_ms * 1e-3), "peak": w.th / (t_roof_bwd * 1e-3),
            "unit": "tokens*heads/s", "frac": t_roof_bwd / bwd_ms, "traffic": traffic,
            "traffic_source": _TRAFFIC_SOURCE if traffic is not None else None,
            "t_tensor_ms": bt_tensor, "t_hbm_ms": bt_hbm, "t_serial_ms": t_ser_bwd,
            "algorithmic_bytes": bb, "algorithmic_flops": bf},
        "roofline_alu": {
            "bound": "alu", "kernel": "bwd", "achieved": achieved / 1e12,
            "peak": peak_tanh / 1e12, "unit": "Ttanh/s", "frac": achieved / peak_tanh,
            "traffic": traffic,
            "traffic_source": _TRAFFIC_SOURCE if traffic is not None else None,
            "units_per_launch": method_tanh,
            "units_basis": "the method's K*V tanh per token x head (one recompute)",
            "design_tanh_per_launch": design_tanh,
            "design_frac": design_tanh / (bwd_ms * 1e-3) / peak_tanh},
    }


if __name__ == "__main__":
    main()
