"""GPU parity of sparse top-k gather attention (attn_sparse_fwd) against the
fp64 oracle.

Element-by-element on every output for small cases that span several 128-slot
chunks, a ragged last chunk, head counts below 128, every (DK, DV) pair, empty
slots (negative entries and entries past the pool), tokens with no filled slot,
repeated rows and a negative scale; the full-size CSA Pro cr4 workload is
checked on sampled tokens.
"""
import numpy as np
import pytest
import torch

import attention_fwd_bwd_gb300 as attn
from attention_fwd_bwd_gb300.inputs import SPARSE_BY_NAME, make_sparse_inputs
from oracle.sparse import sparse_ref_fwd, sparse_ref_tokens_fwd
from tests.helpers import TOL_LSE, TOL_O, np64

pytestmark = pytest.mark.gpu

# o + o_lo carries O to about 16 significant bits (P enters the P.V product as
# a bf16 hi/lo pair, accumulation is fp32).
TOL_O_SPLIT = 2e-3


def gpu_sparse_fwd(q, kp, vp, idx, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, kp, vp))
    idd = idx.to(dev).contiguous()
    B, T, H, _ = q.shape
    DV = vp.shape[2]
    o = torch.empty(B, T, H, DV, dtype=torch.bfloat16, device=dev)
    o_lo = torch.empty_like(o)
    lse = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    attn.attn_sparse_fwd(qd, kd, vd, idd, o, lse, scale, o_lo=o_lo)
    torch.cuda.synchronize()
    assert attn.attn_check_status(None) == 0
    return o.cpu(), o_lo.cpu(), lse.cpu()


def check(o, o_lo, lse, o_ref, lse_ref, what):
    eo = float(np.max(np.abs(np64(o) - o_ref)))
    es = float(np.max(np.abs(np64(o) + np64(o_lo) - o_ref)))
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(np64(lse)), fin), f"{what}: LSE finiteness differs"
    el = float(np.max(np.abs(np64(lse)[fin] - lse_ref[fin]))) if fin.any() else 0.0
    assert eo <= TOL_O, f"{what}: O max-abs error {eo:.3e} > {TOL_O}"
    assert es <= TOL_O_SPLIT, f"{what}: o + o_lo max-abs error {es:.3e} > {TOL_O_SPLIT}"
    assert el <= TOL_LSE, f"{what}: LSE max-abs error {el:.3e} > {TOL_LSE}"


def rand_case(B, T, H, P, K, DK, DV, seed, empty_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, DK, generator=g).to(torch.bfloat16)
    kp = torch.randn(B, P, DK, generator=g).to(torch.bfloat16)
    vp = torch.randn(B, P, DV, generator=g).to(torch.bfloat16)
    idx = torch.randint(0, P, (B, T, K), generator=g, dtype=torch.int32)
    drop = torch.rand(B, T, K, generator=g) < empty_frac
    idx[drop] = -1
    return q, kp, vp, idx


CASES = [
    # B, T, H, P, K, DK, DV
    (1, 7, 128, 300, 128, 128, 128),
    (2, 5, 128, 700, 516, 128, 64),    # five chunks, ragged (4 slots in the last)
    (1, 9, 64, 400, 260, 64, 128),     # 64 heads: rows 64..127 of the tile are not stored
    (1, 6, 100, 257, 384, 64, 64),
    (1, 3, 1, 50, 4, 128, 128),        # one head, one chunk of 4 slots
    (3, 4, 128, 1000, 1152, 128, 128),  # the CSA Pro list length
]


@pytest.mark.parametrize("B,T,H,P,K,DK,DV", CASES)
def test_sparse_elementwise(B, T, H, P, K, DK, DV):
    q, kp, vp, idx = rand_case(B, T, H, P, K, DK, DV, seed=B * 1000 + T * 17 + K)
    scale = 1.0 / np.sqrt(DK)
    o, o_lo, lse = gpu_sparse_fwd(q, kp, vp, idx, scale)
    o_ref, lse_ref = sparse_ref_fwd(np64(q), np64(kp), np64(vp), idx.numpy(), scale)
    check(o, o_lo, lse, o_ref, lse_ref, f"B{B} T{T} H{H} P{P} K{K} DK{DK} DV{DV}")


def test_sparse_edge_cases():
    B, T, H, P, K, DK, DV = 1, 8, 128, 64, 260, 128, 128
    q, kp, vp, idx = rand_case(B, T, H, P, K, DK, DV, seed=9)
    idx[0, 0] = -1                       # a token with no filled slot: O = 0, LSE = -inf
    idx[0, 1, :] = -1
    idx[0, 1, 259] = 5                   # one filled slot, in the ragged chunk
    idx[0, 2, :130] = -1                 # whole first chunk empty for this token
    idx[0, 3, 10:20] = idx[0, 3, 0]      # one row listed 11 times
    idx[0, 4, ::3] = P + 7               # entries past the pool are empty slots
    idx[0, 5, 128:] = 2147483647
    for scale in (1.0 / np.sqrt(DK), -0.2):
        o, o_lo, lse = gpu_sparse_fwd(q, kp, vp, idx, scale)
        o_ref, lse_ref = sparse_ref_fwd(np64(q), np64(kp), np64(vp), np.where(idx.numpy() >= P, -1, idx.numpy()),
                                        scale)
        check(o, o_lo, lse, o_ref, lse_ref, f"edge cases, scale {scale}")
        assert torch.all(o[0, 0] == 0)


def test_sparse_small_workload():
    w = SPARSE_BY_NAME["csa_small_t512"]
    q, kp, vp, do, idx = make_sparse_inputs(w)
    o, o_lo, lse = gpu_sparse_fwd(q, kp, vp, idx, w.scale)
    o_ref, lse_ref = sparse_ref_fwd(np64(q), np64(kp), np64(vp), idx.numpy(), w.scale)
    check(o, o_lo, lse, o_ref, lse_ref, w.name)


def test_sparse_full_size_sampled():
    w = SPARSE_BY_NAME["csa_pro_cr4_t16384"]
    q, kp, vp, do, idx = make_sparse_inputs(w)
    o, o_lo, lse = gpu_sparse_fwd(q, kp, vp, idx, w.scale)
    tokens = [0, 1, 127, 128, 4095, 4096, 9000, w.T - 1]
    o_ref, lse_ref = sparse_ref_tokens_fwd(np64(q), np64(kp), np64(vp), idx.numpy(), w.scale, 0, tokens)
    check(o[0, tokens], o_lo[0, tokens], lse[0][:, tokens], o_ref, lse_ref, w.name + " (sampled tokens)")
