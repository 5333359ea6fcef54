"""Pins for the fp64 oracle, checked against facts that do not come from the
oracle itself: a hand-derived closed-form example, closed forms of special
inputs, central finite differences of the forward, exact invariants of the
gradient, an independent log-sum-exp routine, and a brute-force loop.

Every test here runs on the CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import (
    attn_ref_bwd,
    attn_ref_fwd,
    attn_ref_keys_dkdv,
    attn_ref_probs,
    attn_ref_rows_dq,
    attn_ref_rows_fwd,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _expr(s):
    """Evaluate a fixture expression: numbers, + - * /, and ln()."""
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


# --------------------------------------------------------------------------
# 1. Hand-derived worked example (Eq. (1), section 2.1).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["noncausal", "causal"])
def test_golden_closed_form(mode):
    with open(os.path.join(GOLDEN, "closed_form_s3_d1.json")) as f:
        fx = json.load(f)
    as3 = lambda key: np.array([_expr(s) for s in fx[key]]).reshape(1, 3, 1, 1)
    q, k, v, do = as3("q"), as3("k"), as3("v"), as3("do")
    causal = mode == "causal"
    exp = {n: np.array([_expr(s) for s in fx[mode][n]]) for n in fx[mode]}
    o, lse = attn_ref_fwd(q, k, v, causal, fx["scale"])
    dq, dk, dv = attn_ref_bwd(q, k, v, do, causal, fx["scale"])
    np.testing.assert_allclose(o.ravel(), exp["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.ravel(), exp["lse"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq.ravel(), exp["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.ravel(), exp["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.ravel(), exp["dv"], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# 2. Softmax rows: sum to one; masked entries exactly zero.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_probs_rows_sum_to_one_and_mask(causal):
    rng = np.random.default_rng(1)
    q, k = _rand(rng, 1, 37, 2, 8), _rand(rng, 1, 37, 1, 8)
    p = attn_ref_probs(q, k, causal, 0.35, b=0, h=1)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p >= 0)
    if causal:
        assert np.all(p[np.triu_indices(37, k=1)] == 0.0)
        assert np.all(p[np.tril_indices(37)] > 0.0)


# --------------------------------------------------------------------------
# 3. Closed forms for special inputs.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_running_mean_of_values(causal):
    rng = np.random.default_rng(2)
    S, D = 23, 6
    q = _rand(rng, 2, S, 2, D)
    k = np.broadcast_to(_rand(rng, 1, 1, 1, D), (2, S, 1, D)).copy()
    v = _rand(rng, 2, S, 1, D)
    o, lse = attn_ref_fwd(q, k, v, causal, 0.7)
    for b in range(2):
        for h in range(2):
            for i in range(S):
                n = i + 1 if causal else S
                np.testing.assert_allclose(o[b, i, h], v[b, :n, 0].mean(axis=0), atol=1e-12)
                s0 = 0.7 * q[b, i, h] @ k[b, 0, 0]
                np.testing.assert_allclose(lse[b, h, i], s0 + math.log(n), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_pass_through(causal):
    rng = np.random.default_rng(3)
    S, D = 19, 5
    q, k = _rand(rng, 1, S, 3, D, std=3), _rand(rng, 1, S, 3, D, std=3)
    c = _rand(rng, D)
    v = np.broadcast_to(c, (1, S, 3, D)).copy()
    o, _ = attn_ref_fwd(q, k, v, causal, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-12)


def test_causal_first_row_sees_only_first_key():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 2, 9, 4, 7), _rand(rng, 2, 9, 2, 7), _rand(rng, 2, 9, 2, 7)
    o, lse = attn_ref_fwd(q, k, v, True, 0.3)
    for b in range(2):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(o[b, 0, h], v[b, 0, g], atol=1e-13)
            np.testing.assert_allclose(lse[b, h, 0], 0.3 * q[b, 0, h] @ k[b, 0, g], atol=1e-13)


def test_single_key_uniform_special_case():
    # S = 1, non-causal: softmax over one key is 1, so O = V and LSE = the score.
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, 3, 1, 2, 4), _rand(rng, 3, 1, 2, 4), _rand(rng, 3, 1, 2, 4)
    o, lse = attn_ref_fwd(q, k, v, False, 1.3)
    np.testing.assert_allclose(o, v, atol=1e-14)
    np.testing.assert_allclose(lse, 1.3 * np.einsum("bshd,bshd->bhs", q, k), atol=1e-13)


# --------------------------------------------------------------------------
# 4. LSE against an independent stable log-sum-exp routine.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_lse_matches_scipy_logsumexp(causal):
    rng = np.random.default_rng(6)
    S, D = 41, 16
    q, k = _rand(rng, 1, S, 2, D, std=4), _rand(rng, 1, S, 1, D, std=4)
    v = _rand(rng, 1, S, 1, D)
    _, lse = attn_ref_fwd(q, k, v, causal, 0.25)
    for h in range(2):
        s = 0.25 * np.einsum("id,jd->ij", q[0, :, h], k[0, :, 0])
        for i in range(S):
            row = s[i, : i + 1] if causal else s[i]
            assert abs(lse[0, h, i] - logsumexp(row)) < 1e-12


# --------------------------------------------------------------------------
# 5. Brute force with scalar loops on a tiny input.
# --------------------------------------------------------------------------
def test_forward_brute_force_loops():
    rng = np.random.default_rng(7)
    S, D = 5, 3
    q, k, v = _rand(rng, 1, S, 2, D), _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D)
    for causal in (False, True):
        o, lse = attn_ref_fwd(q, k, v, causal, 0.9)
        for h in range(2):
            for i in range(S):
                ws, tot = [], 0.0
                for j in range(S):
                    if causal and j > i:
                        ws.append(0.0)
                        continue
                    e = math.exp(0.9 * sum(q[0, i, h, d] * k[0, j, 0, d] for d in range(D)))
                    ws.append(e)
                    tot += e
                for d in range(D):
                    ref = sum(ws[j] * v[0, j, 0, d] for j in range(S)) / tot
                    assert abs(o[0, i, h, d] - ref) < 1e-12
                assert abs(lse[0, h, i] - math.log(tot)) < 1e-12


# --------------------------------------------------------------------------
# 6. Central finite differences of L = sum(dO * O) pin the backward.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(causal):
    rng = np.random.default_rng(8)
    B, S, Hq, Hkv, D = 1, 8, 2, 1, 4
    scale = 0.6
    q, k, v = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D)
    do = _rand(rng, B, S, Hq, D)
    dq, dk, dv = attn_ref_bwd(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        o, _ = attn_ref_fwd(qq, kk, vv, causal, scale)
        return float(np.sum(do * o))

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]})
                       - loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * eps)
        rel = np.max(np.abs(fd - g)) / np.max(np.abs(g))
        assert rel < 1e-7, (name, rel)


# --------------------------------------------------------------------------
# 7. Exact invariants of the gradient.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_invariants(causal):
    # sum_j dS_ij = 0 for every row, so sum_j dK_j = 0 per kv head; and
    # sum_j dV_j = sum over the group's query heads and rows of dO_i.
    rng = np.random.default_rng(9)
    B, S, Hq, Hkv, D = 2, 29, 4, 2, 6
    q, k, v = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D)
    do = _rand(rng, B, S, Hq, D)
    _, dk, dv = attn_ref_bwd(q, k, v, do, causal, 0.4)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    G = Hq // Hkv
    for g in range(Hkv):
        np.testing.assert_allclose(dv[:, :, g].sum(axis=1),
                                   do[:, :, g * G:(g + 1) * G].sum(axis=(1, 2)), atol=1e-12)


def test_key_shift_invariance():
    # K -> K + 1 c^T adds scale * q_i . c to every score of row i: O and dK are
    # unchanged and LSE_i shifts by scale * q_i . c.
    rng = np.random.default_rng(10)
    B, S, Hq, Hkv, D = 1, 17, 2, 2, 5
    q, k, v = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D)
    do = _rand(rng, B, S, Hq, D)
    c = _rand(rng, D)
    for causal in (False, True):
        o1, l1 = attn_ref_fwd(q, k, v, causal, 0.5)
        o2, l2 = attn_ref_fwd(q, k + c, v, causal, 0.5)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, 0.5 * np.einsum("bshd,d->bhs", q, c), atol=1e-12)
        _, dk1, _ = attn_ref_bwd(q, k, v, do, causal, 0.5)
        _, dk2, _ = attn_ref_bwd(q, k + c, v, do, causal, 0.5)
        np.testing.assert_allclose(dk2, dk1, atol=1e-12)


# --------------------------------------------------------------------------
# 8. Grouped-query attention equals multi-head attention on repeated K/V,
#    with the gradients of the repeated heads summed (contiguous groups).
# --------------------------------------------------------------------------
def test_gqa_equals_repeated_mha():
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, D = 2, 13, 6, 2, 4
    G = Hq // Hkv
    q, k, v = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D)
    do = _rand(rng, B, S, Hq, D)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    for causal in (False, True):
        o, lse = attn_ref_fwd(q, k, v, causal, 0.45)
        o2, lse2 = attn_ref_fwd(q, kr, vr, causal, 0.45)
        np.testing.assert_allclose(o, o2, atol=1e-13)
        np.testing.assert_allclose(lse, lse2, atol=1e-13)
        dq, dk, dv = attn_ref_bwd(q, k, v, do, causal, 0.45)
        dq2, dkr, dvr = attn_ref_bwd(q, kr, vr, do, causal, 0.45)
        np.testing.assert_allclose(dq, dq2, atol=1e-13)
        np.testing.assert_allclose(dk, dkr.reshape(B, S, Hkv, G, D).sum(axis=3), atol=1e-13)
        np.testing.assert_allclose(dv, dvr.reshape(B, S, Hkv, G, D).sum(axis=3), atol=1e-13)


# --------------------------------------------------------------------------
# 9. Causal masking: row i of causal attention equals non-causal attention over
#    the prefix 0..i; and a uniform rescaling of Q moves into `scale`.
# --------------------------------------------------------------------------
def test_causal_prefix_property_and_scale():
    rng = np.random.default_rng(12)
    S, D = 11, 4
    q, k, v = _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D)
    o, lse = attn_ref_fwd(q, k, v, True, 0.8)
    for i in range(S):
        op, lp = attn_ref_fwd(q[:, : i + 1], k[:, : i + 1], v[:, : i + 1], False, 0.8)
        np.testing.assert_allclose(o[0, i], op[0, i], atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], lp[0, 0, i], atol=1e-13)
    o2, lse2 = attn_ref_fwd(q * 0.8, k, v, True, 1.0)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_noncausal_key_permutation_invariance():
    rng = np.random.default_rng(13)
    S, D = 16, 4
    q, k, v = _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D)
    perm = rng.permutation(S)
    o, lse = attn_ref_fwd(q, k, v, False, 0.5)
    o2, lse2 = attn_ref_fwd(q, k[:, perm], v[:, perm], False, 0.5)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


# --------------------------------------------------------------------------
# 10. The row-subset forms agree with the full oracle.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_forms_match_full(causal):
    rng = np.random.default_rng(14)
    B, S, Hq, Hkv, D = 2, 70, 4, 2, 8
    q, k, v = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D)
    do = _rand(rng, B, S, Hq, D)
    o, lse = attn_ref_fwd(q, k, v, causal, 0.3)
    dq, dk, dv = attn_ref_bwd(q, k, v, do, causal, 0.3)
    rows = [(0, 0, 0), (1, 3, 69), (0, 2, 33), (1, 1, 5)]
    ro, rl = attn_ref_rows_fwd(q, k, v, causal, 0.3, rows)
    rdq = attn_ref_rows_dq(q, k, v, do, causal, 0.3, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], o[b, i, h], atol=1e-13)
        np.testing.assert_allclose(rl[n], lse[b, h, i], atol=1e-13)
        np.testing.assert_allclose(rdq[n], dq[b, i, h], atol=1e-13)
    keys = [0, 1, 31, 69]
    rdk, rdv = attn_ref_keys_dkdv(q, k, v, do, causal, 0.3, 1, 1, keys, row_block=16)
    np.testing.assert_allclose(rdk, dk[1, keys, 1], atol=1e-12)
    np.testing.assert_allclose(rdv, dv[1, keys, 1], atol=1e-12)
