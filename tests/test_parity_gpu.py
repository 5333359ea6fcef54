"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes are compared element by element on every output; they span
several tiles and ragged tails, GQA and MHA, causal and not, D = 64 and 128.
The five named workloads run at full size in the same launch configuration
the benchmark uses, and are compared on seeded samples of rows that the
oracle computes one by one, plus exact gradient invariants over every row.
"""
import numpy as np
import pytest
import torch

from attention_fwd_bwd_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from oracle import attn_ref_bwd, attn_ref_fwd, attn_ref_keys_dkdv, attn_ref_rows_dq, attn_ref_rows_fwd
from tests.helpers import (TOL_GRAD_REL_RMS, assert_close_fwd, assert_close_grad, gpu_fwd_bwd, np64)

pytestmark = pytest.mark.gpu

SMALL = [
    # B, Hq, Hkv, S, D, causal
    (1, 1, 1, 128, 64, False),
    (1, 1, 1, 128, 128, True),
    (1, 2, 1, 384, 128, True),
    (2, 4, 2, 256, 64, True),
    (1, 4, 1, 512, 128, False),
    (1, 2, 2, 300, 128, True),    # ragged tail
    (2, 2, 1, 200, 64, False),    # ragged tail, non-causal
    (1, 3, 3, 129, 64, True),     # one row into a second tile
    (1, 2, 1, 1, 128, True),      # single row
    (1, 2, 2, 77, 128, False),    # shorter than one tile
    (1, 8, 2, 640, 128, True),
]


# residual=True: the training pair attn_fwd_residual -> attn_bwd(o_lo);
# residual=False: the plain pair attn_fwd -> attn_bwd(o_lo = NULL).
@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", SMALL)
def test_small_shapes_elementwise(B, Hq, Hkv, S, D, causal, residual):
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=100 + S + D + Hq)
    got = gpu_fwd_bwd(q, k, v, do, causal, scale, residual=residual)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), causal, scale)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), causal, scale)
    what = f"B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} residual={residual}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


@pytest.mark.parametrize("scale", [0.0, -0.25, 1e-35, 0.6])
@pytest.mark.parametrize("causal", [True, False])
def test_special_scales(scale, causal):
    # scale 0: uniform attention over the visible keys (dQ = dK = 0); a
    # negative scale flips which keys dominate; 1e-35 is below the forward's
    # smallest exponent scale; 0.6 gives a sharp softmax.
    B, Hq, Hkv, S, D = 1, 2, 1, 200, 128
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=7)
    got = gpu_fwd_bwd(q, k, v, do, causal, scale)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), causal, scale)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), causal, scale)
    what = f"scale={scale} causal={causal}"
    for name in ("o", "lse", "dq", "dk", "dv"):
        assert np.isfinite(np64(got[name])).all(), f"{what}: non-finite {name}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
def test_tiny_workload_full(residual):
    w = WORKLOADS[0]
    q, k, v, do = workload_inputs(w)
    got = gpu_fwd_bwd(q, k, v, do, w.causal, w.scale, residual=residual)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), w.causal, w.scale)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), w.causal, w.scale)
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, w.name)
    assert_close_grad(got["dq"], dq_ref, "dQ", w.name)
    assert_close_grad(got["dk"], dk_ref, "dK", w.name)
    assert_close_grad(got["dv"], dv_ref, "dV", w.name)


def _sampled_check(w, n_rows=64, n_key_groups=1, residual=True):
    q, k, v, do = workload_inputs(w)
    got = gpu_fwd_bwd(q, k, v, do, w.causal, w.scale, residual=residual)
    do_t = do
    # float32 copies are exact for bf16 values; the oracle upcasts to fp64.
    q, k, v, do = (t.float().numpy() for t in (q, k, v, do))
    rng = np.random.default_rng(w.seed)
    rows = [(int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(w.S))) for _ in range(n_rows)]
    # always include the first and last rows of the first head
    rows[0] = (0, 0, 0)
    rows[1] = (w.B - 1, w.Hq - 1, w.S - 1)
    o_ref, lse_ref = attn_ref_rows_fwd(q, k, v, w.causal, w.scale, rows)
    dq_ref = attn_ref_rows_dq(q, k, v, do, w.causal, w.scale, rows)
    o_g = np.stack([np64(got["o"][b, i, h]) for b, h, i in rows])
    l_g = np.array([float(got["lse"][b, h, i]) for b, h, i in rows])
    dq_g = np.stack([np64(got["dq"][b, i, h]) for b, h, i in rows])
    what = f"{w.name} residual={residual}"
    assert_close_fwd(o_g, l_g, o_ref, lse_ref, what)
    assert_close_grad(dq_g, dq_ref, "dQ rows", what)
    for _ in range(n_key_groups):
        b, g = int(rng.integers(w.B)), int(rng.integers(w.Hkv))
        keys = sorted(set(int(x) for x in rng.integers(0, w.S, 64)) | {0, w.S - 1})
        dk_ref, dv_ref = attn_ref_keys_dkdv(q, k, v, do, w.causal, w.scale, b, g, keys)
        assert_close_grad(np64(got["dk"][b, keys, g]), dk_ref, "dK rows", what)
        assert_close_grad(np64(got["dv"][b, keys, g]), dv_ref, "dV rows", what)
    # Exact invariants over all rows: sum_j dK_j = 0, sum_j dV_j = sum of the group's dO.
    G = w.Hq // w.Hkv
    dk_sum = got["dk"].to(torch.float64).sum(dim=1)          # [B, Hkv, D]
    dv_sum = got["dv"].to(torch.float64).sum(dim=1)
    do_sum = do_t.to(torch.float64).sum(dim=1).reshape(w.B, w.Hkv, G, w.D).sum(dim=2)
    dk_rms = float(got["dk"].to(torch.float64).pow(2).mean().sqrt())
    dv_rms = float(got["dv"].to(torch.float64).pow(2).mean().sqrt())
    # bf16 rounding of each dK/dV row is an independent error of about
    # 2^-9 * rms, so the row sums drift by about sqrt(S) of that.
    bound_k = 4 * np.sqrt(w.S) * 2.0 ** -8 * dk_rms
    bound_v = 4 * np.sqrt(w.S) * 2.0 ** -8 * dv_rms + 1e-3 * float(do_sum.abs().max())
    assert float(dk_sum.abs().max()) <= bound_k, (float(dk_sum.abs().max()), bound_k)
    assert float((dv_sum - do_sum).abs().max()) <= bound_v, (float((dv_sum - do_sum).abs().max()), bound_v)


@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("name", [w.name for w in WORKLOADS[1:]])
def test_workload_sampled(name, residual):
    w = {x.name: x for x in WORKLOADS}[name]
    _sampled_check(w, residual=residual)


def test_plain_forward_matches_residual_forward():
    """attn_fwd and attn_fwd_residual run the same arithmetic (the residual
    form only stores o_lo as well), so o and lse agree bit for bit."""
    for (B, Hq, Hkv, S, D, causal) in ((1, 4, 2, 384, 128, True), (2, 2, 2, 200, 64, False)):
        q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=11 + S)
        a = gpu_fwd_bwd(q, k, v, do, causal, D ** -0.5, with_bwd=False, residual=True)
        b = gpu_fwd_bwd(q, k, v, do, causal, D ** -0.5, with_bwd=False, residual=False)
        assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])


def test_repeatable_outputs():
    """O, LSE, dK and dV are bitwise repeatable; dQ (fp32 reductions in
    varying order) agrees within the gradient tolerance."""
    q, k, v, do = make_inputs(1, 4, 2, 512, 128, seed=7)
    a = gpu_fwd_bwd(q, k, v, do, True, 128 ** -0.5)
    b = gpu_fwd_bwd(q, k, v, do, True, 128 ** -0.5)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    rms = float(a["dq"].float().pow(2).mean().sqrt())
    assert float((a["dq"].float() - b["dq"].float()).abs().max()) <= TOL_GRAD_REL_RMS * rms


# Shapes where the backward splits each key tile's query heads over two CTAs
# (an even group, >= 512 (head, query tile) iterations in the longest key
# tile, at most four waves of key tiles): 16 heads x 32 query tiles. The two
# halves of dK and dV are added into zeroed rows.
@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("S", [2048, 2000])
def test_split_heads_elementwise(S, residual):
    B, Hq, Hkv, D = 1, 16, 1, 128
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=31 + S)
    got = gpu_fwd_bwd(q, k, v, do, True, scale, residual=residual)
    again = gpu_fwd_bwd(q, k, v, do, True, scale, residual=residual)
    # Two additions onto zero give the same sum in either order.
    assert torch.equal(got["dk"], again["dk"]) and torch.equal(got["dv"], again["dv"])
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), True, scale)
    what = f"split heads S{S} residual={residual}"
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


def test_empty_inputs_are_noops():
    # B == 0 or S == 0 returns ATTN_OK without reading any pointer.
    import attention_fwd_bwd_gb300 as attn
    L = attn.lib()
    for B, S in ((0, 128), (1, 0)):
        assert L.attn_fwd(None, None, None, None, None, B, 2, 1, S, 64, 1, 0.125, None) == 0
        assert L.attn_bwd(*([None] * 10), B, 2, 1, S, 64, 1, 0.125, None, 0, None) == 0
    torch.cuda.synchronize()


# A longer causal sequence compared element by element: key tiles far below
# the diagonal, where every P is small (below 1/16 in most 64 x 128 tiles,
# measured on the oracle's P), so the rounding of small P and dS values is
# checked on every output, not on samples.
@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("D", [128, 64])
def test_long_causal_elementwise(D, residual):
    B, Hq, Hkv, S = 1, 2, 1, 3072
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=57 + D)
    got = gpu_fwd_bwd(q, k, v, do, True, scale, residual=residual)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), True, scale)
    q64, k64 = np64(q), np64(k)
    small = total = 0
    for h in range(Hq):
        s = scale * (q64[0, :, h] @ k64[0, :, 0].T) - lse_ref[0, h][:, None]
        s[np.triu_indices(S, 1)] = -np.inf
        tmax = np.exp(s).reshape(S // 64, 64, S // 128, 128).max(axis=(1, 3))
        visible = np.arange(S // 128)[None, :] * 128 <= np.arange(S // 64)[:, None] * 64 + 63
        small += int((tmax[visible] <= 1 / 16).sum())
        total += int(visible.sum())
    assert small >= total // 2, (small, total)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(q64, k64, np64(v), np64(do), True, scale)
    what = f"S{S} D{D} residual={residual}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


# The staged entry points (preprocess, optionally the Dvec pass, then the
# main kernel) compute what attn_bwd computes, and can run again on the same
# workspace: the preprocess restarts the main kernel's item counter each time
# (short items, D = 64: one CTA per SM taking items from that counter; long
# items, D = 128: one CTA per item).
@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(2, 4, 4, 1024, 64), (1, 8, 2, 2048, 128)])
def test_staged_backward_matches_attn_bwd(B, Hq, Hkv, S, D, residual):
    import attention_fwd_bwd_gb300 as attn
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = (t.cuda() for t in make_inputs(B, Hq, Hkv, S, D, seed=91 + D))
    o, o_lo = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    attn.attn_fwd_residual(q, k, v, o, o_lo, lse, True, scale)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, Hq, Hkv, S, D), dtype=torch.uint8, device=q.device)
    f32 = lambda t: torch.empty(t.shape, dtype=torch.float32, device=t.device)
    ref = [f32(q), f32(k), f32(k)]
    attn.attn_bwd(q, k, v, o, do, lse, *ref, True, scale, ws, o_lo=o_lo if residual else None)
    rms = float(ref[0].double().pow(2).mean().sqrt())
    for _ in range(2):
        got = [f32(q), f32(k), f32(k)]
        attn.attn_bwd_preprocess(q, k, o, do, lse, got[0], ws, o_lo=o_lo if residual else None)
        if not residual:
            attn.attn_bwd_dvec(q, k, v, do, True, scale, ws)
        attn.attn_bwd_main(q, k, v, do, *got, True, scale, ws)
        torch.cuda.synchronize()
        assert attn.attn_check_status(ws) == 0
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        # dq: fp32 reductions in varying order
        assert float((got[0] - ref[0]).abs().max()) <= 1e-5 * rms


# Non-causal attention over a long sequence, element by element: every key
# tile sees every query tile, so the backward's items are long (G x 64
# iterations) and run as one CTA per item -- the launch the short shapes
# above do not reach without the causal mask.
@pytest.mark.parametrize("Hq,Hkv,D", [(4, 1, 128), (4, 2, 64)])
def test_long_noncausal_elementwise(Hq, Hkv, D):
    B, S = 1, 4096
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=211 + D)
    got = gpu_fwd_bwd(q, k, v, do, False, scale)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), False, scale)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), False, scale)
    what = f"non-causal S{S} Hq{Hq} Hkv{Hkv} D{D}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


@pytest.mark.parametrize("D,window", [(128, 0), (128, 200), (64, 0), (64, 77)])
def test_head_pairing_leaves_rows_unchanged(D, window):
    # With causal masking and an even number of query heads per kv head, a
    # forward item holds the same rows of two heads; with one query head per
    # kv head it holds two consecutive row blocks of one head. Each row's
    # arithmetic is the same either way, so GQA equals the same problem with
    # K/V repeated per query head, bit for bit.
    B, Hq, Hkv, S = 1, 4, 2, 520
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=900 + D + window)
    kr, vr = (t.repeat_interleave(Hq // Hkv, dim=2).contiguous() for t in (k, v))
    for residual in (True, False):
        a = gpu_fwd_bwd(q, k, v, do, True, scale, with_bwd=False, window=window, residual=residual)
        b = gpu_fwd_bwd(q, kr, vr, do, True, scale, with_bwd=False, window=window, residual=residual)
        assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"]), (D, window, residual)
