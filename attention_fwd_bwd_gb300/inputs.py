"""Seeded synthetic inputs and the workload table.

This module holds no attention arithmetic: it only draws random tensors, so the
CUDA path and the fp64 oracle can be fed identical inputs without sharing any
of the method's code.

Recipe: a CPU torch.Generator seeded with `seed` draws N(0,1) float32 tensors
in the order Q, K, V, dO; Q and K are multiplied by `qk_std` (2 for the
sharper-softmax 70B-shaped workload, 1 elsewhere) and every tensor is then
rounded to bfloat16 (round to nearest even). Layout is [B, S, H, D],
contiguous.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    causal: bool
    qk_std: float = 1.0
    seed: int = 1234
    window: int = 0  # > 0: sliding-window causal attention over the last `window` keys

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops_fwd(self) -> float:
        """4 * B * Hq * S^2 * D, halved when causal; with a window of W keys,
        4 * B * Hq * D times the visible (query, key) pairs, sum_i min(i+1, W)."""
        if self.window > 0:
            W, S = min(self.window, self.S), self.S
            pairs = W * (W + 1) / 2 + (S - W) * W
            return 4.0 * self.B * self.Hq * self.D * pairs
        f = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        """2.5 times the forward count."""
        return 2.5 * self.flops_fwd()


# The five workloads: shapes and value distributions of the attention layers of
# the models the pages train (Llama 3 8B / 70B shapes, GQA), a head-dim-64 MHA
# case, a long-context case and a tiny one. Seeds are 1234 + index.
WORKLOADS = [
    Workload("tiny_s128_d64", 1, 1, 1, 128, 64, False, 1.0, 1234),
    Workload("llama3_8b_s4096", 2, 32, 8, 4096, 128, True, 1.0, 1235),
    Workload("mha_d64_s2048", 8, 16, 16, 2048, 64, True, 1.0, 1236),
    Workload("llama3_70b_s8192", 1, 64, 8, 8192, 128, True, 2.0, 1237),
    Workload("long_s32768", 1, 32, 8, 32768, 128, True, 1.0, 1238),
]
# Beyond those: sliding-window causal attention with a 128-key window and 64
# query heads, the dense part (cr0) of the sparse attention the pages study
# (Table 7: "Flash cr0", 64 heads, every query over a 128-token window), at
# the Llama-3-8B sequence length.
EXTRA_WORKLOADS = [
    Workload("swa_w128_s4096", 2, 64, 8, 4096, 128, True, 1.0, 1240, 128),
]
BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def make_inputs(B, Hq, Hkv, S, D, seed, qk_std=1.0):
    """Return bf16 CPU tensors (q, k, v, do) drawn as the module docstring says."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn(B, S, Hq, D, generator=g, dtype=torch.float32)
    k = torch.randn(B, S, Hkv, D, generator=g, dtype=torch.float32)
    v = torch.randn(B, S, Hkv, D, generator=g, dtype=torch.float32)
    do = torch.randn(B, S, Hq, D, generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        q.mul_(qk_std)
        k.mul_(qk_std)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, do))


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.Hq, w.Hkv, w.S, w.D, w.seed, w.qk_std)
