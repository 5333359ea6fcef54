"""Pins for the sparse top-k gather oracle, checked against facts that do not
come from it: the dense oracle (itself pinned) when every list names every
pool row in order, or a token's sliding window; a brute-force loop over the
slots; the closed form of a one-slot list; invariance under slot order and
under empty slots; a repeated row against a pool that holds the row twice;
central finite differences of the loss with d_v != d; and planted mistakes
that these catch.

CPU only.
"""
import math
import types

import numpy as np
import pytest

import oracle.sparse as sparse_mod
from oracle import attn_ref_bwd, attn_ref_fwd

SRC = open(sparse_mod.__file__).read()


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _case(rng, B=1, T=5, H=3, P=7, K=4, DK=3, DV=2):
    q, kp, vp, do = _rand(rng, B, T, H, DK), _rand(rng, B, P, DK), _rand(rng, B, P, DV), _rand(rng, B, T, H, DV)
    idx = np.stack([np.stack([rng.permutation(P)[:K] for _ in range(T)]) for _ in range(B)]).astype(np.int32)
    return q, kp, vp, do, idx


def _dense_all_rows_ok(m, scale=0.45):
    """Every list = all pool rows in order: dense non-causal attention with one
    kv head (T = P so the dense oracle applies)."""
    rng = np.random.default_rng(3)
    B, T, H, D = 2, 6, 3, 4
    q, kp, vp, do = _rand(rng, B, T, H, D), _rand(rng, B, T, D), _rand(rng, B, T, D), _rand(rng, B, T, H, D)
    idx = np.tile(np.arange(T, dtype=np.int32), (B, T, 1))
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, scale)
    od, lsed = attn_ref_fwd(q, kp[:, :, None], vp[:, :, None], False, scale)
    dq, dkp, dvp = m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    dqd, dkd, dvd = attn_ref_bwd(q, kp[:, :, None], vp[:, :, None], do, False, scale)
    return (np.allclose(o, od, atol=1e-12) and np.allclose(lse, lsed, atol=1e-12)
            and np.allclose(dq, dqd, atol=1e-12) and np.allclose(dkp, dkd[:, :, 0], atol=1e-12)
            and np.allclose(dvp, dvd[:, :, 0], atol=1e-12))


def _window_ok(m, W=3, scale=0.8):
    """idx[t] = rows t-W+1..t (-1 where negative): the dense sliding window."""
    rng = np.random.default_rng(4)
    B, T, H, D = 1, 8, 2, 3
    q, kp, vp, do = _rand(rng, B, T, H, D), _rand(rng, B, T, D), _rand(rng, B, T, D), _rand(rng, B, T, H, D)
    t = np.arange(T)[:, None] - (W - 1) + np.arange(W)[None, :]
    idx = np.where(t >= 0, t, -1).astype(np.int32)[None]
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, scale)
    od, lsed = attn_ref_fwd(q, kp[:, :, None], vp[:, :, None], True, scale, window=W)
    dq, dkp, dvp = m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    dqd, dkd, dvd = attn_ref_bwd(q, kp[:, :, None], vp[:, :, None], do, True, scale, window=W)
    return (np.allclose(o, od, atol=1e-12) and np.allclose(lse, lsed, atol=1e-12)
            and np.allclose(dq, dqd, atol=1e-12) and np.allclose(dkp, dkd[:, :, 0], atol=1e-12)
            and np.allclose(dvp, dvd[:, :, 0], atol=1e-12))


def _brute_ok(m, scale=0.6):
    """Scalar loops over heads, slots and dims, with idx holding empty slots."""
    rng = np.random.default_rng(5)
    q, kp, vp, do, idx = _case(rng, T=3, K=5, P=6)
    idx[0, 1, 2] = -1
    idx[0, 2, 0] = -1
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, scale)
    H, DK, DV = q.shape[2], q.shape[3], vp.shape[2]
    for t in range(3):
        for h in range(H):
            ws = []
            for j in range(5):
                r = idx[0, t, j]
                if r < 0:
                    continue
                ws.append((math.exp(scale * sum(q[0, t, h, d] * kp[0, r, d] for d in range(DK))), r))
            tot = sum(w for w, _ in ws)
            for e in range(DV):
                if abs(o[0, t, h, e] - sum(w * vp[0, r, e] for w, r in ws) / tot) > 1e-12:
                    return False
            if abs(lse[0, h, t] - math.log(tot)) > 1e-12:
                return False
    return True


def _one_slot_ok(m, scale=1.3):
    rng = np.random.default_rng(6)
    q, kp, vp, do, idx = _case(rng, K=3)
    idx[:] = -1
    idx[0, :, 1] = 4
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, scale)
    dq, dkp, dvp = m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    s = scale * np.einsum("thd,d->ht", q[0], kp[0, 4])
    # One key: the output is its value, LSE its score, and the softmax
    # Jacobian vanishes (dq = dkp = 0); dvp[4] = sum of dO over tokens and heads.
    exp_dv = np.zeros_like(dvp)
    exp_dv[0, 4] = do[0].sum(axis=(0, 1))
    return (np.allclose(o[0], np.broadcast_to(vp[0, 4], o[0].shape), atol=1e-12)
            and np.allclose(lse[0], s, atol=1e-12) and np.allclose(dq, 0, atol=1e-12)
            and np.allclose(dkp, 0, atol=1e-12) and np.allclose(dvp, exp_dv, atol=1e-12))


def _order_and_padding_ok(m, scale=0.5):
    """Permuting a token's slots or inserting empty slots changes nothing."""
    rng = np.random.default_rng(7)
    q, kp, vp, do, idx = _case(rng, T=4, K=4, P=9)
    ref = m.sparse_ref_fwd(q, kp, vp, idx, scale) + m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    perm = idx[:, :, ::-1].copy()
    pad = np.concatenate([np.full((1, 4, 2), -1, np.int32), idx, np.full((1, 4, 3), -1, np.int32)], axis=2)
    for alt in (perm, pad):
        got = m.sparse_ref_fwd(q, kp, vp, alt, scale) + m.sparse_ref_bwd(q, kp, vp, alt, do, scale)
        if not all(np.allclose(a, b, atol=1e-12) for a, b in zip(ref, got)):
            return False
    return True


def _repeat_ok(m, scale=0.7):
    """A row listed twice equals a pool holding that row twice, listed once each;
    its gradient is the sum of the two copies' gradients."""
    rng = np.random.default_rng(8)
    q, kp, vp, do, idx = _case(rng, T=3, K=3, P=5)
    idx[0, :, 1] = idx[0, :, 0]
    P = kp.shape[1]
    kp2 = np.concatenate([kp, kp[:, :1] * 0], axis=1)
    vp2 = np.concatenate([vp, vp[:, :1] * 0], axis=1)
    idx2 = idx.copy()
    # Per token, the second listing points at a copy of the first row.
    for t in range(3):
        r = idx[0, t, 0]
        kp2t, vp2t = kp2.copy(), vp2.copy()
        kp2t[0, P], vp2t[0, P] = kp[0, r], vp[0, r]
        i2 = idx2[:, t:t + 1].copy()
        i2[0, 0, 1] = P
        o, lse = m.sparse_ref_fwd(q[:, t:t + 1], kp, vp, idx[:, t:t + 1], scale)
        o2, lse2 = m.sparse_ref_fwd(q[:, t:t + 1], kp2t, vp2t, i2, scale)
        dq, dkp, dvp = m.sparse_ref_bwd(q[:, t:t + 1], kp, vp, idx[:, t:t + 1], do[:, t:t + 1], scale)
        dq2, dkp2, dvp2 = m.sparse_ref_bwd(q[:, t:t + 1], kp2t, vp2t, i2, do[:, t:t + 1], scale)
        def fold(g):  # add the copy's row back onto row r
            f = g[:, :P].copy()
            f[:, r] += g[:, P]
            return f
        if not (np.allclose(o, o2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)
                and np.allclose(dq, dq2, atol=1e-12) and np.allclose(dkp, fold(dkp2), atol=1e-12)
                and np.allclose(dvp, fold(dvp2), atol=1e-12)):
            return False
    return True


def _fd_ok(m, scale=0.9, eps=1e-6):
    """Central differences of L = sum(dO * O) with DK = 3 != DV = 2 and an
    empty slot, against the analytic gradients."""
    rng = np.random.default_rng(9)
    q, kp, vp, do, idx = _case(rng, T=2, H=2, P=5, K=4)
    idx[0, 1, 3] = -1
    dq, dkp, dvp = m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    loss = lambda q_, kp_, vp_: float((m.sparse_ref_fwd(q_, kp_, vp_, idx, scale)[0] * do).sum())
    for arr, grad, pos in ((q, dq, 0), (kp, dkp, 1), (vp, dvp, 2)):
        for i in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[i] += eps
            a2[i] -= eps
            args1 = [q, kp, vp]
            args2 = [q, kp, vp]
            args1[pos], args2[pos] = a1, a2
            fd = (loss(*args1) - loss(*args2)) / (2 * eps)
            if abs(fd - grad[i]) > 1e-6:
                return False
    return True


def _empty_token_ok(m, scale=1.0):
    rng = np.random.default_rng(10)
    q, kp, vp, do, idx = _case(rng, T=3)
    idx[0, 1] = -1
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, scale)
    dq, _, _ = m.sparse_ref_bwd(q, kp, vp, idx, do, scale)
    return (np.all(o[0, 1] == 0) and np.all(np.isneginf(lse[0, :, 1])) and np.all(dq[0, 1] == 0)
            and np.all(np.isfinite(lse[0, :, 0])))


PINS = [_dense_all_rows_ok, _window_ok, _brute_ok, _one_slot_ok, _order_and_padding_ok, _repeat_ok,
        _fd_ok, _empty_token_ok]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_sparse_oracle_pin(pin):
    assert pin(sparse_mod)


def test_sparse_rows_beyond_pool_rejected():
    rng = np.random.default_rng(11)
    q, kp, vp, do, idx = _case(rng)
    idx[0, 0, 0] = kp.shape[1]
    with pytest.raises(ValueError):
        sparse_mod.sparse_ref_fwd(q, kp, vp, idx, 1.0)


MUTATIONS = [
    ("empty slots read the last row", "filled = np.nonzero(idx_bt >= 0)[0]", "filled = np.arange(idx_bt.size)"),
    ("scale dropped", "s = scale * (q_bt @ kg.T)", "s = q_bt @ kg.T"),
    ("softmax over heads", "m = s.max(axis=1, keepdims=True)\n    e = np.exp(s - m)\n    return e / e.sum(axis=1, keepdims=True)",
     "m = s.max(axis=0, keepdims=True)\n    e = np.exp(s - m)\n    return e / e.sum(axis=0, keepdims=True)"),
    ("lse missing max", "lse[:, n] = m + np.log(", "lse[:, n] = np.log("),
    ("dS sign flipped", "ds = p * (dp - dvec)", "ds = p * (dvec - dp)"),
    ("Dvec dropped", "ds = p * (dp - dvec)", "ds = p * dp"),
    ("dq scale dropped", "dq[b, t] = scale * (ds @ kg)", "dq[b, t] = ds @ kg"),
    ("dK uses P", "np.add.at(dkp[b], rows, scale * (ds.T @ q[b, t]))", "np.add.at(dkp[b], rows, scale * (p.T @ q[b, t]))"),
    ("repeated rows lose a term", "np.add.at(dvp[b], rows, p.T @ do[b, t])", "dvp[b][rows] += p.T @ do[b, t]"),
    ("dP uses K", "dp = do[b, t] @ vg.T", "dp = do[b, t] @ kg[:, :do.shape[3]].T"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_sparse_pins_catch_mutant(name, old, new):
    assert old in SRC, old
    m = types.ModuleType("sparse_mutant")
    exec(compile(SRC.replace(old, new, 1), "sparse_mutant", "exec"), m.__dict__)
    caught = []
    for pin in PINS:
        try:
            caught.append(not pin(m))
        except Exception:
            caught.append(True)
    assert any(caught), name


def _golden_ok(m):
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "sparse_closed_form_t3_d1.json")
    with open(path) as f:
        fx = json.load(f)
    ev = lambda s: float(eval(s, {"__builtins__": {}}, {"ln": math.log, "inf": math.inf}))
    vec = lambda key: np.array([ev(s) for s in fx[key]])
    q = vec("q").reshape(1, 3, 1, 1)
    do = vec("do").reshape(1, 3, 1, 1)
    kp, vp = vec("kp").reshape(1, 3, 1), vec("vp").reshape(1, 3, 1)
    idx = np.array(fx["idx"], dtype=np.int32)[None]
    o, lse = m.sparse_ref_fwd(q, kp, vp, idx, fx["scale"])
    dq, dkp, dvp = m.sparse_ref_bwd(q, kp, vp, idx, do, fx["scale"])
    lse_exp = vec("lse")
    fin = np.isfinite(lse_exp)
    return (np.allclose(o.ravel(), vec("o"), atol=1e-12)
            and np.array_equal(np.isfinite(lse.ravel()), fin)
            and np.allclose(lse.ravel()[fin], lse_exp[fin], atol=1e-12)
            and np.allclose(dq.ravel(), vec("dq"), atol=1e-12)
            and np.allclose(dkp.ravel(), vec("dkp"), atol=1e-12)
            and np.allclose(dvp.ravel(), vec("dvp"), atol=1e-12))


PINS.append(_golden_ok)


def test_sparse_oracle_golden_worked_example():
    assert _golden_ok(sparse_mod)
