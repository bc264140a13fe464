"""Seeded synthetic inputs for attention workloads.

This module holds no attention arithmetic: it only draws random tensors.  It is
the one piece shared by the CUDA path's tests/benchmark and by the oracle's
tests, so that both sides see the same bf16 bytes.

Recipe (one per workload): a CPU ``torch.Generator`` seeded with the
workload's seed draws, in this order, Q, K, V and (for backward workloads) dO,
each as ``torch.randn(B, H, N, d)`` in float32.  Q and K are multiplied by
``qk_mult`` (3 for the peaked-softmax workload) and then every tensor is
rounded to the storage dtype (bfloat16 by default).  Layout is contiguous
[B, H, N, d].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool
    seed: int
    qk_mult: float = 1.0
    description: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    def flops_fwd(self) -> float:
        """4 B H N^2 d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_fwd_bwd(self) -> float:
        """10 B H N^2 d (forward 4 + backward 6 by this count), halved when causal."""
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f


# The five workloads: a tiny forward check, a short-sequence d=64 training
# shape, two d=128 causal training shapes (the second with Q, K scaled by 3 to
# make softmax rows peaked) and a long-sequence causal shape.
WORKLOADS = {
    w.name: w
    for w in (
        Workload("fwd_b1_h2_n256_d64", 1, 2, 256, 64, False, False, 1001,
                 description="forward only, non-causal, B=1 H=2 N=256 d=64"),
        Workload("fwdbwd_b8_h16_n1024_d64", 8, 16, 1024, 64, False, True, 1002,
                 description="forward+backward, non-causal, B=8 H=16 N=1024 d=64"),
        Workload("fwdbwd_causal_b4_h32_n4096_d128", 4, 32, 4096, 128, True, True, 1003,
                 description="forward+backward, causal, B=4 H=32 N=4096 d=128"),
        Workload("fwdbwd_causal_peaked_b2_h16_n8192_d128", 2, 16, 8192, 128, True, True, 1004,
                 qk_mult=3.0,
                 description="forward+backward, causal, B=2 H=16 N=8192 d=128, Q,K x3"),
        Workload("fwdbwd_causal_b1_h8_n32768_d128", 1, 8, 32768, 128, True, True, 1005,
                 description="long-sequence forward+backward, causal, B=1 H=8 N=32768 d=128"),
    )
}

HEADLINE = "fwdbwd_causal_peaked_b2_h16_n8192_d128"


def make_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0,
                with_grad: bool = True, dtype: torch.dtype = torch.bfloat16):
    """Return a dict of contiguous CPU tensors q, k, v (and dO) of shape [B,H,N,d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    out = {}
    for name in ("q", "k", "v") + (("dO",) if with_grad else ()):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x = x * qk_mult
        out[name] = x.to(dtype).contiguous()
    return out


def workload_inputs(w: Workload, with_grad=None, dtype: torch.dtype = torch.bfloat16):
    wg = w.backward if with_grad is None else with_grad
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, wg, dtype)
