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


# ---------------------------------------------------------------- backward
from oracle.sparse import sparse_ref_bwd  # noqa: E402
from tests.helpers import assert_close_grad  # noqa: E402


def gpu_sparse_fwd_bwd(q, kp, vp, idx, do, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev).contiguous() for t in (q, kp, vp, do))
    idd = idx.to(dev).contiguous()
    B, T, H, DK = q.shape
    P, DV = kp.shape[1], vp.shape[2]
    o = torch.empty(B, T, H, DV, dtype=torch.bfloat16, device=dev)
    o_lo = torch.empty_like(o)
    lse = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    attn.attn_sparse_fwd(qd, kd, vd, idd, o, lse, scale, o_lo=o_lo)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dkp, dvp = torch.empty(B, T, H, DK, **f32), torch.empty(B, P, DK, **f32), torch.empty(B, P, DV, **f32)
    ws = torch.empty(attn.attn_sparse_bwd_workspace_size(B, T, H), dtype=torch.uint8, device=dev)
    attn.attn_sparse_bwd(qd, kd, vd, idd, o, dod, lse, dq, dkp, dvp, scale, ws, o_lo=o_lo)
    torch.cuda.synchronize()
    assert attn.attn_check_status(ws) == 0
    return {n: t.cpu() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dkp", dkp), ("dvp", dvp))}


def check_grads(got, q, kp, vp, idx, do, scale, what):
    dq_ref, dkp_ref, dvp_ref = sparse_ref_bwd(np64(q), np64(kp), np64(vp), idx, np64(do), scale)
    assert_close_grad(got["dq"], dq_ref, "dq", what)
    assert_close_grad(got["dkp"], dkp_ref, "dkp", what)
    assert_close_grad(got["dvp"], dvp_ref, "dvp", what)


@pytest.mark.parametrize("B,T,H,P,K,DK,DV", CASES)
def test_sparse_bwd_elementwise(B, T, H, P, K, DK, DV):
    q, kp, vp, idx = rand_case(B, T, H, P, K, DK, DV, seed=B * 1000 + T * 17 + K)
    g = torch.Generator().manual_seed(T + K)
    do = torch.randn(B, T, H, DV, generator=g).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(DK)
    got = gpu_sparse_fwd_bwd(q, kp, vp, idx, do, scale)
    check_grads(got, q, kp, vp, idx.numpy(), do, scale, f"B{B} T{T} H{H} P{P} K{K} DK{DK} DV{DV}")


def test_sparse_bwd_edge_cases():
    B, T, H, P, K, DK, DV = 1, 8, 128, 64, 260, 128, 128
    q, kp, vp, idx = rand_case(B, T, H, P, K, DK, DV, seed=9)
    idx[0, 0] = -1                       # no filled slot: zero gradient
    idx[0, 1, :] = -1
    idx[0, 1, 259] = 5                   # one filled slot: dS = 0, dvp[5] = sum of dO
    idx[0, 2, :130] = -1
    idx[0, 3, 10:20] = idx[0, 3, 0]      # one row listed 11 times
    idx[0, 4, ::3] = P + 7               # entries past the pool are empty slots
    do = torch.randn(B, T, H, DV, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    ref_idx = np.where(idx.numpy() >= P, -1, idx.numpy())
    for scale in (1.0 / np.sqrt(DK), -0.2):
        got = gpu_sparse_fwd_bwd(q, kp, vp, idx, do, scale)
        check_grads(got, q, kp, vp, ref_idx, do, scale, f"edge cases, scale {scale}")
        assert torch.all(got["dq"][0, 0] == 0)


def test_sparse_bwd_small_workload():
    w = SPARSE_BY_NAME["csa_small_t512"]
    q, kp, vp, do, idx = make_sparse_inputs(w)
    got = gpu_sparse_fwd_bwd(q, kp, vp, idx, do, w.scale)
    check_grads(got, q, kp, vp, idx.numpy(), do, w.scale, w.name)


def test_sparse_bwd_full_size_sampled():
    """Full CSA Pro cr4 size: dq of sampled tokens against the oracle (a token's
    dq depends on that token alone), and the pool gradients through invariants
    that hold at any size: summed over pool rows, dvp equals the sum of dO over
    every head of every token with a filled slot (each token's probabilities
    sum to 1), and dkp sums to zero (each row of dS sums to zero)."""
    w = SPARSE_BY_NAME["csa_pro_cr4_t16384"]
    q, kp, vp, do, idx = make_sparse_inputs(w)
    got = gpu_sparse_fwd_bwd(q, kp, vp, idx, do, w.scale)
    tokens = [0, 1, 127, 128, 4095, 4096, 9000, w.T - 1]
    dq_ref, _, _ = sparse_ref_bwd(np64(q[:, tokens]), np64(kp), np64(vp), idx[:, tokens].numpy(),
                                  np64(do[:, tokens]), w.scale)
    assert_close_grad(got["dq"][:, tokens], dq_ref, "dq", w.name + " (sampled tokens)")
    has = (idx >= 0).any(dim=2)  # [B, T]
    sum_do = (np64(do) * has.numpy()[:, :, None, None]).sum(axis=(1, 2))  # [B, DV]
    sum_dvp = np64(got["dvp"]).sum(axis=1)
    scale_do = np.abs(np64(do)).sum(axis=(1, 2))
    assert np.max(np.abs(sum_dvp - sum_do) / scale_do) < 1e-4
    sum_dkp = np64(got["dkp"]).sum(axis=1)
    mag_dkp = np.abs(np64(got["dkp"])).sum(axis=1)
    assert np.max(np.abs(sum_dkp) / mag_dkp) < 1e-3
    # Pool rows j < T are token j's own row, which only the windows of
    # tokens j .. j+127 list (the compressed rows are T and beyond); the
    # oracle over those tokens gives their dkp and dvp row in full.
    rows = [0, 1, 127, 5000, 9000, w.T - 128, w.T - 1]
    dk_got, dv_got, dk_ref, dv_ref = [], [], [], []
    for j in rows:
        toks = list(range(j, min(j + w.window, w.T)))
        sel = idx[:, toks].numpy()
        assert not np.isin(j, np.delete(idx.numpy(), toks, axis=1)), "row listed outside its window"
        _, dkp_r, dvp_r = sparse_ref_bwd(np64(q[:, toks]), np64(kp), np64(vp), sel, np64(do[:, toks]), w.scale)
        dk_ref.append(dkp_r[:, j]); dv_ref.append(dvp_r[:, j])
        dk_got.append(np64(got["dkp"][:, j])); dv_got.append(np64(got["dvp"][:, j]))
    assert_close_grad(np.stack(dk_got), np.stack(dk_ref), "dkp", w.name + " (window-only pool rows)")
    assert_close_grad(np.stack(dv_got), np.stack(dv_ref), "dvp", w.name + " (window-only pool rows)")
