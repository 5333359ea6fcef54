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


# ---------------------------------------------------------------- sparse top-k
# Synthetic stand-in for the top-k lists of the pages' compressed sparse
# attention (Table 7, "cr4": every query attends to a 128-token sliding window
# plus the top-k rows of a pool compressed 4:1). No trained model or real
# top-k map is available, so the lists are drawn at random with the same
# structure:
#   * pool rows 0..T-1 are the tokens' own rows; rows T..T+T/r-1 are the
#     compressed rows, row T+c summarising tokens r*c..r*c+r-1;
#   * token t's list is its window, rows t-W+1..t (-1 where negative), then
#     `topk` compressed rows: all visible ones (those whose r tokens end at or
#     before t) when there are at most `topk`, else a uniformly random subset
#     of `topk` of them, in ascending order; -1 pads the rest.
# q, kp, vp and dO are N(0,1) draws rounded to bf16, in that order, from the
# same seeded generator, followed by the random keys that pick the subsets.


@dataclass(frozen=True)
class SparseWorkload:
    name: str
    B: int
    T: int
    H: int
    DK: int
    DV: int
    window: int
    topk: int
    ratio: int
    seed: int = 2024

    @property
    def P(self) -> int:
        return self.T + self.T // self.ratio

    @property
    def K(self) -> int:
        return self.window + self.topk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.DK)


SPARSE_WORKLOADS = [
    # Pro cr4 (Table 7): 128 heads, top-k 1152 = 128 window + top-1024 of T/4.
    SparseWorkload("csa_pro_cr4_t16384", 1, 16384, 128, 128, 128, 128, 1024, 4, 2024),
    # Flash cr4 (Table 7): 64 heads, top-k 640 = 128 window + top-512 of T/4.
    SparseWorkload("csa_flash_cr4_t8192", 1, 8192, 64, 128, 128, 128, 512, 4, 2025),
    # Small case the oracle finishes in seconds; d_v != d.
    SparseWorkload("csa_small_t512", 2, 512, 128, 128, 64, 128, 96, 4, 2026),
    # The Pro cr4 list structure at a quarter of the tokens (top-1024 of T/4:
    # the later tokens' lists are full), a size for detailed profiler captures.
    SparseWorkload("csa_pro_cr4_t4096", 1, 4096, 128, 128, 128, 128, 1024, 4, 2027),
]
SPARSE_BY_NAME = {w.name: w for w in SPARSE_WORKLOADS}


def make_sparse_index(T, window, topk, ratio, g):
    """idx [T, window + topk] int32 as the recipe above says (torch.Generator g)."""
    nc = T // ratio
    idx = torch.full((T, window + topk), -1, dtype=torch.int32)
    t = torch.arange(T, dtype=torch.int64)
    w = t[:, None] - (window - 1) + torch.arange(window, dtype=torch.int64)[None, :]
    idx[:, :window] = torch.where(w >= 0, w, torch.full_like(w, -1)).to(torch.int32)
    if nc == 0 or topk == 0:
        return idx
    keys = torch.rand(T, nc, generator=g, dtype=torch.float32)
    visible = (torch.arange(nc, dtype=torch.int64)[None, :] + 1) * ratio <= (t[:, None] + 1)
    keys = torch.where(visible, keys, torch.full_like(keys, -1.0))
    n_vis = visible.sum(dim=1)
    kk = min(topk, nc)
    pick = keys.topk(kk, dim=1).indices  # the kk largest keys; invisible rows rank last
    pick, _ = pick.sort(dim=1)
    # Rows that are not visible only fill lists with fewer than kk visible rows:
    # drop them, keeping the visible ones in ascending order.
    ok = visible.gather(1, pick)
    rows = torch.where(ok, pick + T, torch.full_like(pick, -1))
    # Move the filled entries to the front (stable), -1 after them.
    order = torch.argsort((~ok).to(torch.int8), dim=1, stable=True)
    rows = rows.gather(1, order)
    idx[:, window:window + kk] = rows.to(torch.int32)
    assert int((rows >= 0).sum(dim=1).max()) <= int(n_vis.max())
    return idx


def make_sparse_inputs(w: SparseWorkload):
    """bf16 CPU tensors (q [B,T,H,DK], kp [B,P,DK], vp [B,P,DV], do [B,T,H,DV])
    and idx [B,T,K] int32, drawn as the recipe above says."""
    g = torch.Generator(device="cpu").manual_seed(int(w.seed))
    q = torch.randn(w.B, w.T, w.H, w.DK, generator=g, dtype=torch.float32)
    kp = torch.randn(w.B, w.P, w.DK, generator=g, dtype=torch.float32)
    vp = torch.randn(w.B, w.P, w.DV, generator=g, dtype=torch.float32)
    do = torch.randn(w.B, w.T, w.H, w.DV, generator=g, dtype=torch.float32)
    idx = torch.stack([make_sparse_index(w.T, w.window, w.topk, w.ratio, g) for _ in range(w.B)])
    return tuple(t.to(torch.bfloat16) for t in (q, kp, vp, do)) + (idx,)
