"""Plain, slow, fp64 CPU sparse top-k gather attention: the oracle for the
sparse attention kernels.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
leg of the benchmark may import this module. The product path never calls it,
and it imports nothing from the product.

Source: "Scheduling Data to Compute: Hierarchical Data Pipelining for LLM
Training on AMD GPUs" (Rao et al.), §2.1 (Compressed Sparse Attention: every
query token receives a top-k list; the forward gathers those vectors, scores
them and streams the matching values into the output; the backward gathers
the same vectors for dQ and reduces a per-slot dKV intermediate through the
inverse of the top-k map), §3 (a token's top-k list is a list of KV row
indices) and §4.1 Table 7 (each query attends to a 128-token window plus its
top-k compressed-pool rows). Eq. (1) of §2.1 gives the attention itself:
O = softmax(Q K^T / sqrt(d)) V, with d_v allowed to differ from d.

Readings where the pages are silent (listed with reasons in the design notes):
  * One gathered key/value source per batch, shared by every query head of a
    token (the top-k list belongs to the token, not to a head): a key pool
    kp [B, P, DK] and a value pool vp [B, P, DV]; the window rows and the
    compressed rows are both rows of that pool.
  * idx [B, T, K] int32: slot j of token t reads pool row idx[b, t, j]; a
    negative entry is an empty slot and contributes nothing. Slots are
    independent: a row listed twice counts twice.
  * scale is an explicit argument (Eq. (1) fixes 1/sqrt(DK)).
  * LSE[b, h, t] = ln sum_j exp(scale * q . kp[idx_j]) over the filled slots;
    a token with no filled slot has O = 0 and LSE = -inf (and zero gradient).
  * backward: the exact gradient of the loss sum(dO * O). With
    P = softmax over the slots, S_hj = scale * q_h . k_j:
        dP_hj = dO_h . v_j,  Dvec_h = sum_j P_hj dP_hj,  dS = P * (dP - Dvec),
        dq_h = scale * sum_j dS_hj k_j,
        per-slot dK_j = scale * sum_h dS_hj q_h,  dV_j = sum_h P_hj dO_h,
    and dkp / dvp of a pool row sum the per-slot terms of every (token, slot)
    that lists it (the inverse of the top-k map).

Layouts: q, o, dO, dq: [B, T, H, D*] (DK for q and dq, DV for o and dO);
kp, dkp: [B, P, DK]; vp, dvp: [B, P, DV]; lse: [B, H, T].
"""
import numpy as np

__all__ = ["sparse_ref_fwd", "sparse_ref_bwd", "sparse_ref_tokens_fwd"]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _token(q_bt, kp_b, vp_b, idx_bt, scale):
    """One token: q_bt [H, DK], kp_b [P, DK], vp_b [P, DV], idx_bt [K].

    Returns (P [H, n], rows [n], s [H, n]) over the filled slots, in slot order,
    or None when no slot is filled."""
    filled = np.nonzero(idx_bt >= 0)[0]
    if filled.size == 0:
        return None
    rows = idx_bt[filled].astype(np.int64)
    kg = kp_b[rows]  # [n, DK] gathered keys
    s = scale * (q_bt @ kg.T)  # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True), rows, s


def _check(q, kp, vp, idx):
    B, T, H, DK = q.shape
    if kp.shape[0] != B or kp.shape[2] != DK or vp.shape[:2] != kp.shape[:2]:
        raise ValueError("kp [B, P, DK] and vp [B, P, DV] must match q [B, T, H, DK]")
    if idx.shape[:2] != (B, T):
        raise ValueError("idx must be [B, T, K]")
    if np.any(idx >= kp.shape[1]):
        raise ValueError("idx holds a row beyond the pool")


def sparse_ref_tokens_fwd(q, kp, vp, idx, scale, b, tokens):
    """O [len(tokens), H, DV] and LSE [H, len(tokens)] of the listed tokens of
    batch b (the whole-array function below calls this token by token)."""
    q, kp, vp = _f64(q), _f64(kp), _f64(vp)
    idx = np.asarray(idx)
    _check(q, kp, vp, idx)
    H, DV = q.shape[2], vp.shape[2]
    o = np.zeros((len(tokens), H, DV))
    lse = np.full((H, len(tokens)), -np.inf)
    for n, t in enumerate(tokens):
        r = _token(q[b, t], kp[b], vp[b], idx[b, t], scale)
        if r is None:
            continue
        p, rows, s = r
        o[n] = p @ vp[b][rows]
        m = s.max(axis=1)
        lse[:, n] = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    return o, lse


def sparse_ref_fwd(q, kp, vp, idx, scale):
    """O [B, T, H, DV] and LSE [B, H, T] (fp64)."""
    B, T = q.shape[0], q.shape[1]
    H, DV = q.shape[2], np.shape(vp)[2]
    o = np.zeros((B, T, H, DV))
    lse = np.zeros((B, H, T))
    for b in range(B):
        o[b], lse[b] = sparse_ref_tokens_fwd(q, kp, vp, idx, scale, b, range(T))
    return o, lse


def sparse_ref_bwd(q, kp, vp, idx, do, scale):
    """(dq [B, T, H, DK], dkp [B, P, DK], dvp [B, P, DV]) for the loss sum(dO * O),
    fp64, probabilities recomputed from the inputs."""
    q, kp, vp, do = _f64(q), _f64(kp), _f64(vp), _f64(do)
    idx = np.asarray(idx)
    _check(q, kp, vp, idx)
    B, T = q.shape[:2]
    dq = np.zeros_like(q)
    dkp = np.zeros_like(kp)
    dvp = np.zeros_like(vp)
    for b in range(B):
        for t in range(T):
            r = _token(q[b, t], kp[b], vp[b], idx[b, t], scale)
            if r is None:
                continue
            p, rows, _ = r
            kg, vg = kp[b][rows], vp[b][rows]
            dp = do[b, t] @ vg.T  # [H, n]
            dvec = (p * dp).sum(axis=1, keepdims=True)
            ds = p * (dp - dvec)
            dq[b, t] = scale * (ds @ kg)
            # Per-slot terms, reduced into the pool through the inverse map;
            # np.add.at adds every occurrence of a repeated row.
            np.add.at(dkp[b], rows, scale * (ds.T @ q[b, t]))
            np.add.at(dvp[b], rows, p.T @ do[b, t])
    return dq, dkp, dvp
