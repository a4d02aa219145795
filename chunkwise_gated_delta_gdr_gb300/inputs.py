"""Seeded synthetic inputs for the gated delta rule forward pass.

This module only draws random tensors; it holds none of the method's
arithmetic (no normalisation, cumsum, decay or solve). Both the CUDA path and
the float64 oracle read the tensors it returns, so the two always see the same
bits.

Recipe (one CPU ``torch.Generator`` per workload, seeded; every tensor drawn in
float32 in the order q, k, v, g, beta, initial state; then cast with
round-to-nearest-even to the workload's q/k/v dtype; g, beta and the state stay
float32):

  q, k, v ~ N(0, 1)
  g       = logsigmoid(N(mu_g, sd_g)) per token and value head (scalar gate),
            or per token, value head and key channel (per-key gate, KDA)
  beta    = sigmoid(N(0, 1))
  S0      = 0, or N(0, sd_s0) when the workload carries a state

``N(m, s)`` is a normal distribution with mean m and standard deviation s.
logsigmoid and sigmoid only shape the distributions of the log-decay and the
write strength; they are part of the input recipe, not of the method.

The five named workloads follow the benchmark configurations of the gated
delta rule forward pass; ``make_inputs`` can shrink any of them (fewer tokens,
batches or heads) while keeping its distributions and seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    C: int
    dtype: torch.dtype          # q, k, v element type
    gate_mode: int              # 0: scalar gate [B,T,HV]; 1: per-key gate [B,T,HV,K]
    g_mean: float
    g_std: float
    s0_std: Optional[float]     # None: zero initial state
    seed: int
    use_qk_l2norm: bool = True
    description: str = ""
    segments: int = 1           # > 1: the forward runs as a segmented scan of this many parts

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.K)

    @property
    def n_chunks(self) -> int:
        return (self.T + self.C - 1) // self.C


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", B=1, T=128, H=2, HV=2, K=32, V=32, C=16, dtype=torch.float32,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=None, seed=0,
        description="tiny scalar-gate forward, fp32 q/k/v, K=V=32, C=16"),
    "gdn_t4096_h12": Workload(
        "gdn_t4096_h12", B=1, T=4096, H=12, HV=12, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=None, seed=1,
        description="scalar-gate forward, bf16 q/k/v, T=4096, 12 heads, K=V=128, C=64"),
    "kda_gqa_t8192": Workload(
        "kda_gqa_t8192", B=2, T=8192, H=16, HV=32, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=1, g_mean=3.0, g_std=1.0, s0_std=None, seed=2,
        description="per-key-gate (KDA) forward, 16 q/k heads shared by 32 value heads"),
    "gdn_long_t65000": Workload(
        "gdn_long_t65000", B=1, T=65000, H=32, HV=32, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=1.0, g_std=1.0, s0_std=0.02, seed=3,
        description="scalar-gate forward, T=65000 (ragged last chunk), carried fp32 state"),
    "kda_many_b64": Workload(
        "kda_many_b64", B=64, T=1024, H=16, HV=16, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=1, g_mean=0.0, g_std=2.0, s0_std=None, seed=4,
        description="per-key-gate forward, 64 short sequences, strong decay"),
}

# The workload the throughput figure is quoted on.
# The token-by-token (decode) form: one new token per sequence, carried state.
DECODE_WORKLOADS = {
    "decode_b64_h16": Workload(
        "decode_b64_h16", B=64, T=1, H=16, HV=16, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=0.02, seed=5,
        description="decode step: 64 sequences x 16 heads, one token each, fp32 state in place"),
}

# Few, long sequences: the case the segmented scan of the chunk recurrence serves
# (16 state chains for 152 SMs unsegmented).
SEGMENTED_WORKLOADS = {
    "gdn_h2_t65536": Workload(
        "gdn_h2_t65536", B=1, T=65536, H=2, HV=2, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=1.0, g_std=1.0, s0_std=0.02, seed=7, segments=8,
        description="scalar-gate forward, 2 heads x 65536 tokens, carried state, 8 segments"),
}

# The Mamba2 SSD recurrence on the headline shape (beta is drawn but not used).
SSD_WORKLOADS = {
    "ssd_t4096_h12": Workload(
        "ssd_t4096_h12", B=1, T=4096, H=12, HV=12, K=128, V=128, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=None, seed=6,
        description="Mamba2 SSD forward on the headline shape"),
}

# The headline shape with a chunk size or head dims outside the tensor-core
# path (C = 128; K = V = 64): the general fp32 path.
GENERAL_WORKLOADS = {
    "gdn_c128_t4096_h12": Workload(
        "gdn_c128_t4096_h12", B=1, T=4096, H=12, HV=12, K=128, V=128, C=128, dtype=torch.bfloat16,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=None, seed=1,
        description="the headline shape with chunk size 128"),
    "gdn_k64_t4096_h12": Workload(
        "gdn_k64_t4096_h12", B=1, T=4096, H=12, HV=12, K=64, V=64, C=64, dtype=torch.bfloat16,
        gate_mode=0, g_mean=0.0, g_std=1.0, s0_std=None, seed=1,
        description="the headline shape with head dims K = V = 64"),
}

HEADLINE = "gdn_t4096_h12"


def shrink(w: Workload, **overrides) -> Workload:
    """Same workload with some sizes replaced (distributions and seed unchanged)."""
    return dataclasses.replace(w, **overrides)


def make_inputs(w: Workload, device: str = "cpu", **overrides):
    """Draw the workload's tensors. Returns a dict with q, k, v, g, beta, s0 (or None).

    Tensors are generated on the CPU (so every device sees identical values)
    and then moved to ``device``.
    """
    if overrides:
        w = shrink(w, **overrides)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    f32 = torch.float32
    q = torch.randn(w.B, w.T, w.H, w.K, generator=gen, dtype=f32)
    k = torch.randn(w.B, w.T, w.H, w.K, generator=gen, dtype=f32)
    v = torch.randn(w.B, w.T, w.HV, w.V, generator=gen, dtype=f32)
    gshape = (w.B, w.T, w.HV) if w.gate_mode == 0 else (w.B, w.T, w.HV, w.K)
    g = torch.nn.functional.logsigmoid(
        torch.randn(*gshape, generator=gen, dtype=f32) * w.g_std + w.g_mean)
    beta = torch.sigmoid(torch.randn(w.B, w.T, w.HV, generator=gen, dtype=f32))
    s0 = None
    if w.s0_std is not None:
        s0 = torch.randn(w.B, w.HV, w.K, w.V, generator=gen, dtype=f32) * w.s0_std
    q, k, v = (x.to(w.dtype) for x in (q, k, v))
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta, s0=s0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out
