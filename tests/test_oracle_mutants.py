"""Plant plausible mistakes in a copy of the oracle's source and check that the
pins catch every one: a pin set that a dropped term, a wrong sign, a wrong
index or a transposed operand slips through is not a pin.

The mutants are built on the CPU from the oracle's source text; nothing here
touches a GPU or the CUDA library.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle.ref as ref_mod

SRC = open(ref_mod.__file__).read()
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MUTATIONS = [
    ("causal mask off by one", "s[cols > rows] = -np.inf", "s[cols >= rows] = -np.inf"),
    ("causal mask reversed", "s[cols > rows] = -np.inf", "s[cols < rows] = -np.inf"),
    ("scale dropped from scores", "s = scale * (qh @ kh.T)", "s = (qh @ kh.T)"),
    ("softmax not normalised", "    p /= l[:, None]\n", "    pass\n"),
    ("lse in base 2", "return p, m + np.log(l)", "return p, m + np.log2(l)"),
    ("lse missing max", "return p, m + np.log(l)", "return p, np.log(l)"),
    ("PV transposed", "o[b, :, h, :] = p @ v[b, :, g, :]", "o[b, :, h, :] = p.T @ v[b, :, g, :]"),
    ("GQA interleaved", "            g = h // G\n            p, lse[b, h]", "            g = h % k.shape[2]\n            p, lse[b, h]"),
    ("dQ scale dropped", "dq[b, :, h, :] = scale * (ds @ kh)", "dq[b, :, h, :] = (ds @ kh)"),
    ("dK uses dS not dS^T", "dk[b, :, g, :] += scale * (ds.T @ qh)", "dk[b, :, g, :] += scale * (ds @ qh)"),
    ("dV uses P not P^T", "dv[b, :, g, :] += p.T @ doh", "dv[b, :, g, :] += p @ doh"),
    ("dS sign flipped", "ds = p * (dp - dvec[:, None])\n            dq[b", "ds = p * (dvec[:, None] - dp)\n            dq[b"),
    ("Dvec term dropped", "ds = p * (dp - dvec[:, None])\n            dq[b", "ds = p * dp\n            dq[b"),
    ("dV not accumulated over group", "dv[b, :, g, :] += p.T @ doh", "dv[b, :, g, :] = p.T @ doh"),
    ("dP uses K instead of V", "dp = doh @ vh.T\n            dvec", "dp = doh @ kh.T\n            dvec"),
]


def _load_mutant(old, new):
    assert old in SRC, old
    m = types.ModuleType("oracle_mutant")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant", "exec"), m.__dict__)
    return m


def _expr(s):
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


def _golden_ok(m):
    with open(os.path.join(GOLDEN, "closed_form_s3_d1.json")) as f:
        fx = json.load(f)
    as3 = lambda key: np.array([_expr(s) for s in fx[key]]).reshape(1, 3, 1, 1)
    for mode in ("noncausal", "causal"):
        causal = mode == "causal"
        o, lse = m.attn_ref_fwd(as3("q"), as3("k"), as3("v"), causal, 1.0)
        dq, dk, dv = m.attn_ref_bwd(as3("q"), as3("k"), as3("v"), as3("do"), causal, 1.0)
        for name, got in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            exp = np.array([_expr(s) for s in fx[mode][name]])
            if not np.allclose(got.ravel(), exp, rtol=0, atol=1e-12):
                return False
    return True


def _fd_ok(m):
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((1, 6, 2, 3)), rng.standard_normal((1, 6, 1, 3)), rng.standard_normal((1, 6, 1, 3))
    do = rng.standard_normal((1, 6, 2, 3))
    for causal in (False, True):
        dq, dk, dv = m.attn_ref_bwd(q, k, v, do, causal, 0.6)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += 1e-6
                xm[idx] -= 1e-6
                a = {"q": q, "k": k, "v": v}
                b = dict(a)
                a[name], b[name] = xp, xm
                fp = np.sum(do * m.attn_ref_fwd(a["q"], a["k"], a["v"], causal, 0.6)[0])
                fm = np.sum(do * m.attn_ref_fwd(b["q"], b["k"], b["v"], causal, 0.6)[0])
                if abs((fp - fm) / 2e-6 - g[idx]) > 1e-6 * max(1.0, np.max(np.abs(g))):
                    return False
    return True


def _gqa_ok(m):
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, D = 1, 7, 4, 2, 3
    q, k, v = rng.standard_normal((B, S, Hq, D)), rng.standard_normal((B, S, Hkv, D)), rng.standard_normal((B, S, Hkv, D))
    # reference: each query head run alone against its contiguous-group kv head
    o, _ = m.attn_ref_fwd(q, k, v, True, 0.5)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        oh, _ = m.attn_ref_fwd(q[:, :, h:h + 1], k[:, :, g:g + 1], v[:, :, g:g + 1], True, 0.5)
        if not np.allclose(o[:, :, h], oh[:, :, 0], atol=1e-12):
            return False
    return True


def _lse_ok(m):
    from scipy.special import logsumexp
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal((1, 9, 1, 4)) * 3, rng.standard_normal((1, 9, 1, 4)) * 3, rng.standard_normal((1, 9, 1, 4))
    _, lse = m.attn_ref_fwd(q, k, v, True, 0.25)
    s = 0.25 * q[0, :, 0] @ k[0, :, 0].T
    return all(abs(lse[0, 0, i] - logsumexp(s[i, : i + 1])) < 1e-12 for i in range(9))


def _pins_pass(m):
    return _golden_ok(m) and _lse_ok(m) and _gqa_ok(m) and _fd_ok(m)


def test_unmutated_oracle_passes_pins():
    assert _pins_pass(ref_mod)


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(label, old, new):
    m = _load_mutant(old, new)
    try:
        caught = not _pins_pass(m)
    except Exception:
        caught = True
    assert caught, f"planted mistake not caught: {label}"
