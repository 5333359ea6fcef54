"""Pins for the oracle's sliding-window form (key j visible to query i iff
i - W < j <= i), checked against facts that do not come from the oracle: a
brute-force loop over the visibility rule, the closed form of a one-key
window, translation invariance, the plain causal case, per-row visible-key
counts, central finite differences, and planted mistakes that these catch.

CPU only.
"""
import math
import types

import numpy as np
import pytest

import oracle.ref as ref_mod
from oracle import attn_ref_bwd, attn_ref_fwd, attn_ref_keys_dkdv, attn_ref_probs, attn_ref_rows_dq, attn_ref_rows_fwd


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _brute_ok(m, S=9, W=3, D=3, scale=0.7):
    rng = np.random.default_rng(21)
    q, k, v = _rand(rng, 1, S, 2, D), _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D)
    o, lse = m.attn_ref_fwd(q, k, v, True, scale, window=W)
    for h in range(2):
        for i in range(S):
            ws = [math.exp(scale * sum(q[0, i, h, d] * k[0, j, 0, d] for d in range(D)))
                  if i - W < j <= i else 0.0 for j in range(S)]
            tot = sum(ws)
            for d in range(D):
                if abs(o[0, i, h, d] - sum(ws[j] * v[0, j, 0, d] for j in range(S)) / tot) > 1e-12:
                    return False
            if abs(lse[0, h, i] - math.log(tot)) > 1e-12:
                return False
    return True


def _one_key_ok(m):
    # W = 1: each query sees only its own key, so O_i = v_i, LSE_i = scale q_i.k_i,
    # dS = 0 (dQ = dK = 0) and dV_j = sum over the group's heads of dO_j.
    rng = np.random.default_rng(22)
    B, S, Hq, Hkv, D = 1, 6, 4, 2, 3
    q, k, v, do = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hq, D)
    o, lse = m.attn_ref_fwd(q, k, v, True, 0.8, window=1)
    dq, dk, dv = m.attn_ref_bwd(q, k, v, do, True, 0.8, window=1)
    G = Hq // Hkv
    for h in range(Hq):
        g = h // G
        if not np.allclose(o[0, :, h], v[0, :, g], atol=1e-13):
            return False
        if not np.allclose(lse[0, h], 0.8 * np.sum(q[0, :, h] * k[0, :, g], axis=1), atol=1e-13):
            return False
    if not (np.allclose(dq, 0, atol=1e-13) and np.allclose(dk, 0, atol=1e-13)):
        return False
    for g in range(Hkv):
        if not np.allclose(dv[0, :, g], do[0, :, g * G:(g + 1) * G].sum(axis=1), atol=1e-13):
            return False
    return True


def _translation_ok(m, W=4):
    # Prepending one token shifts every full window by one position.
    rng = np.random.default_rng(23)
    S, D = 12, 5
    q, k, v = _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D), _rand(rng, 1, S, 1, D)
    o, lse = m.attn_ref_fwd(q, k, v, True, 0.5, window=W)
    pre = lambda x: np.concatenate([_rand(rng, 1, 1, 1, D), x], axis=1)
    o2, lse2 = m.attn_ref_fwd(pre(q), pre(k), pre(v), True, 0.5, window=W)
    return (np.allclose(o2[0, W:, 0], o[0, W - 1:, 0], atol=1e-13)
            and np.allclose(lse2[0, 0, W:], lse[0, 0, W - 1:], atol=1e-13))


def _fd_ok(m, W=3):
    rng = np.random.default_rng(24)
    q, k, v, do = _rand(rng, 1, 7, 2, 3), _rand(rng, 1, 7, 1, 3), _rand(rng, 1, 7, 1, 3), _rand(rng, 1, 7, 2, 3)
    dq, dk, dv = m.attn_ref_bwd(q, k, v, do, True, 0.6, window=W)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-6
            xm[idx] -= 1e-6
            a = {"q": q, "k": k, "v": v}
            b = dict(a)
            a[name], b[name] = xp, xm
            fp = np.sum(do * m.attn_ref_fwd(a["q"], a["k"], a["v"], True, 0.6, window=W)[0])
            fm = np.sum(do * m.attn_ref_fwd(b["q"], b["k"], b["v"], True, 0.6, window=W)[0])
            if abs((fp - fm) / 2e-6 - g[idx]) > 1e-6 * max(1.0, np.max(np.abs(g))):
                return False
    return True


def _window_pins_pass(m):
    return _brute_ok(m) and _one_key_ok(m) and _translation_ok(m) and _fd_ok(m)


def test_brute_force_loops():
    assert _brute_ok(ref_mod)
    assert _brute_ok(ref_mod, S=10, W=7, D=2, scale=-0.4)


def test_one_key_window_closed_form():
    assert _one_key_ok(ref_mod)


def test_translation_invariance():
    assert _translation_ok(ref_mod, W=4)
    assert _translation_ok(ref_mod, W=1)


def test_gradients_match_finite_differences():
    assert _fd_ok(ref_mod, W=3)


@pytest.mark.parametrize("W", [1, 3, 64])
def test_visible_key_counts(W):
    rng = np.random.default_rng(25)
    S = 40
    p = attn_ref_probs(_rand(rng, 1, S, 1, 4), _rand(rng, 1, S, 1, 4), True, 0.5, window=W)
    for i in range(S):
        assert np.count_nonzero(p[i]) == min(i + 1, W)
        np.testing.assert_allclose(p[i].sum(), 1.0, atol=1e-14)


def test_window_at_least_sequence_is_plain_causal():
    rng = np.random.default_rng(26)
    q, k, v, do = _rand(rng, 1, 9, 2, 3), _rand(rng, 1, 9, 1, 3), _rand(rng, 1, 9, 1, 3), _rand(rng, 1, 9, 2, 3)
    for W in (9, 10, 1000):
        for a, b in zip(attn_ref_fwd(q, k, v, True, 0.5, window=W), attn_ref_fwd(q, k, v, True, 0.5)):
            np.testing.assert_array_equal(a, b)
        for a, b in zip(attn_ref_bwd(q, k, v, do, True, 0.5, window=W), attn_ref_bwd(q, k, v, do, True, 0.5)):
            np.testing.assert_array_equal(a, b)


def test_gradient_sum_invariants():
    rng = np.random.default_rng(27)
    B, S, Hq, Hkv, D = 2, 23, 4, 2, 5
    q, k, v, do = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hq, D)
    _, dk, dv = attn_ref_bwd(q, k, v, do, True, 0.4, window=5)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    G = Hq // Hkv
    for g in range(Hkv):
        np.testing.assert_allclose(dv[:, :, g].sum(axis=1), do[:, :, g * G:(g + 1) * G].sum(axis=(1, 2)), atol=1e-12)


def test_row_subset_forms_match_full():
    rng = np.random.default_rng(28)
    B, S, Hq, Hkv, D = 1, 50, 2, 1, 4
    q, k, v, do = _rand(rng, B, S, Hq, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hkv, D), _rand(rng, B, S, Hq, D)
    W = 9
    o, lse = attn_ref_fwd(q, k, v, True, 0.3, window=W)
    dq, dk, dv = attn_ref_bwd(q, k, v, do, True, 0.3, window=W)
    rows = [(0, 0, 0), (0, 1, 49), (0, 0, 8), (0, 1, 9)]
    ro, rl = attn_ref_rows_fwd(q, k, v, True, 0.3, rows, window=W)
    rdq = attn_ref_rows_dq(q, k, v, do, True, 0.3, rows, window=W)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], o[b, i, h], atol=1e-13)
        np.testing.assert_allclose(rl[n], lse[b, h, i], atol=1e-13)
        np.testing.assert_allclose(rdq[n], dq[b, i, h], atol=1e-13)
    keys = [0, 7, 40, 49]
    rdk, rdv = attn_ref_keys_dkdv(q, k, v, do, True, 0.3, 0, 0, keys, row_block=16, window=W)
    np.testing.assert_allclose(rdk, dk[0, keys, 0], atol=1e-12)
    np.testing.assert_allclose(rdv, dv[0, keys, 0], atol=1e-12)


def test_window_needs_causal():
    with pytest.raises(ValueError):
        attn_ref_fwd(np.zeros((1, 4, 1, 2)), np.zeros((1, 4, 1, 2)), np.zeros((1, 4, 1, 2)), False, 1.0, window=2)


SRC = open(ref_mod.__file__).read()
WINDOW_MUTATIONS = [
    ("window boundary off by one (too wide)", "s[cols <= rows - window] = -np.inf", "s[cols < rows - window] = -np.inf"),
    ("window boundary off by one (too narrow)", "s[cols <= rows - window] = -np.inf", "s[cols <= rows - window + 1] = -np.inf"),
    ("window dropped in the backward", "p, _ = _softmax_rows(_scores(qh, kh, scale, causal, window=window))\n            dp = doh",
     "p, _ = _softmax_rows(_scores(qh, kh, scale, causal))\n            dp = doh"),
]


def _load_mutant(old, new):
    assert old in SRC, old
    m = types.ModuleType("oracle_window_mutant")
    exec(compile(SRC.replace(old, new, 1), "oracle_window_mutant", "exec"), m.__dict__)
    return m


def test_unmutated_oracle_passes_window_pins():
    assert _window_pins_pass(ref_mod)


@pytest.mark.parametrize("label,old,new", WINDOW_MUTATIONS, ids=[m[0] for m in WINDOW_MUTATIONS])
def test_window_pins_catch_planted_mistake(label, old, new):
    m = _load_mutant(old, new)
    try:
        caught = not _window_pins_pass(m)
    except Exception:
        caught = True
    assert caught, f"planted mistake not caught: {label}"
