"""Seeded synthetic inputs for the M2RNN recurrence.

This module holds no arithmetic of the method itself: it only draws random
tensors in a fixed order, so that the CUDA path and the fp64 oracle can be fed
identical values.  It imports nothing from the CUDA binding.

Recipe (shapes and distributions follow the paper's workloads: K=64, V=16 per
value head, frame "Shared queries and keys buy more recurrent capacity";
4,096-token training sequences and BF16 training, frame "Two model scales
share a 100B-token training protocol"; long contexts to 16K and beyond):

  torch CPU generator seeded with ``seed``; draws in this order, all fp32:
    q  ~ N(0,1) [B,T,K], then L2-normalised over K (shared by all heads);
                            [B,T,G,K] with G > 1 query/key groups
    k  ~ N(0,1) [B,T,K] (or [B,T,G,K]), then L2-normalised over K
    v  ~ N(0,1)/4 [B,T,N,V]
    f  = sigmoid(N(f_mean, 1)) [B,T,N]
    W  ~ N(0, 1/V) [N,V,V]
    w_r ~ N(0,1) [N,V]
    dy ~ N(0,1) [B,T,N,V]   (only when requested)
    a  ~ N(0,1) [B,T,N], alpha ~ U(0.5, 1.5) [N], beta ~ N(-2, 0.5) [N]
                            (only for the fused input gate)
    g  ~ U(0, 1) [B,T,N,V], w_norm ~ N(1, 0.1) [N,V]
                            (drawn last, only for the readout epilogue)
  then every tensor is cast to the workload's input dtype (round to nearest
  even for bf16).  H0 = 0 unless a test supplies one.

  Decode workloads (T = 1, state carried between calls) draw the state with
  ``decode_state``: U(-0.9, 0.9) fp32 [B,N,K,V] from a generator seeded with
  ``seed + 1`` (any reachable state has |H| <= 1).
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    N: int
    K: int
    V: int
    dtype: str          # "f32" or "bf16": dtype of q, k, v, f, W, w_r, y
    seed: int
    f_mean: float = 2.0
    backward: bool = False
    ckpt_every: int = 0  # checkpoint interval C for the backward (0 = none)
    decode: bool = False  # single-step decode (T = 1, state carried in HBM)
    gated: bool = False   # f computed from a, alpha, beta by the fused input gate
    norm: bool = False    # readout epilogue: out = RMSNorm(y (.) g)

    @property
    def th(self) -> int:
        """tokens x heads processed by one pass."""
        return self.B * self.T * self.N


# The workloads the recurrence is exercised and measured on.
WORKLOADS = {
    w.name: w for w in (
        Workload("fwd_f32_b1_t64_n4", 1, 64, 4, 64, 16, "f32", 0),
        Workload("fwd_bf16_b8_t2048_n32", 8, 2048, 32, 64, 16, "bf16", 1),
        Workload("fwd_bf16_b1_t65536_n64", 1, 65536, 64, 64, 16, "bf16", 2, f_mean=3.0),
        Workload("fwd_bf16_b64_t4096_n32", 64, 4096, 32, 64, 16, "bf16", 3),
        Workload("fwd_bf16_b64_t4096_n32_k128", 64, 4096, 32, 128, 16, "bf16", 3),
        Workload("fwd_bf16_b64_t4096_n32_v32", 64, 4096, 32, 64, 32, "bf16", 3),
        Workload("fwdbwd_bf16_b8_t4096_n32", 8, 4096, 32, 64, 16, "bf16", 4,
                 backward=True, ckpt_every=64),
        Workload("fwdbwd_gated_bf16_b8_t4096_n32", 8, 4096, 32, 64, 16, "bf16", 4,
                 backward=True, ckpt_every=64, gated=True),
        Workload("fwdbwd_norm_bf16_b8_t4096_n32", 8, 4096, 32, 64, 16, "bf16", 4,
                 backward=True, ckpt_every=64, norm=True),
        Workload("decode_bf16_b2048_n32", 2048, 1, 32, 64, 16, "bf16", 6, decode=True),
    )
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_inputs(B: int, T: int, N: int, K: int, V: int, dtype: str = "bf16",
                seed: int = 0, f_mean: float = 2.0, with_dy: bool = False,
                gated: bool = False, groups: int = 1, norm: bool = False) -> dict:
    """Draw one seeded input set on the CPU (see the module docstring)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    qk_shape = (B, T, K) if groups == 1 else (B, T, groups, K)
    q = torch.randn(*qk_shape, generator=g)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k = torch.randn(*qk_shape, generator=g)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn(B, T, N, V, generator=g) / 4.0
    f = torch.sigmoid(torch.randn(B, T, N, generator=g) + f_mean)
    W = torch.randn(N, V, V, generator=g) / (V ** 0.5)
    w_r = torch.randn(N, V, generator=g)
    out = {"q": q, "k": k, "v": v, "f": f, "W": W, "w_r": w_r}
    if with_dy:
        out["dy"] = torch.randn(B, T, N, V, generator=g)
    if gated:
        out["a"] = torch.randn(B, T, N, generator=g)
        out["alpha"] = torch.rand(N, generator=g) + 0.5
        out["beta"] = torch.randn(N, generator=g) * 0.5 - 2.0
    if norm:
        out["g"] = torch.rand(B, T, N, V, generator=g)
        out["w_norm"] = torch.randn(N, V, generator=g) * 0.1 + 1.0
    td = TORCH_DTYPES[dtype]
    return {name: t.to(td).contiguous() for name, t in out.items()}


def decode_state(B: int, N: int, K: int, V: int, seed: int) -> torch.Tensor:
    """A state to decode from (see the module docstring)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 1)
    return (torch.rand(B, N, K, V, generator=g) * 2 - 1) * 0.9


def workload_inputs(w: Workload, with_dy: bool | None = None) -> dict:
    return make_inputs(w.B, w.T, w.N, w.K, w.V, w.dtype, w.seed, w.f_mean,
                       with_dy=w.backward if with_dy is None else with_dy, gated=w.gated,
                       norm=w.norm)
