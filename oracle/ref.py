"""Plain, slow, fp64 CPU attention: the oracle for the fused attention kernels.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
leg of the benchmark may import this module. The product path (the CUDA
library and its Python binding) never calls it, and it imports nothing from the
product: it is written from the definition of attention alone.

Source: "Scheduling Data to Compute: Hierarchical Data Pipelining for LLM
Training on AMD GPUs" (Rao et al.), §2.1 Eq. (1): O = softmax(Q K^T / sqrt(d)) V
for one head, with the softmax taken over keys. Algorithm 0 on the same page
(FlashAttention-style streaming with online softmax) reaches this same result
up to rounding order, so the oracle is the definition written out, with the
score matrix materialised.

Readings where the page is silent (each one is listed with its reason in the
design notes of the repository):
  * scale is an explicit argument (Eq. (1) fixes it to 1/sqrt(d); every
    workload here passes exactly that value).
  * causal: key j is visible to query i iff j <= i (equal query and key
    lengths, so no row is fully masked).
  * sliding window (the dense part of the sparse attention on the same page:
    §4.1, Table 7 caption, "every query attends to a 128-token sliding
    window", and §3's cr0 kernels, where consecutive tokens attend to almost
    the same window rows): with window W > 0 and causal, key j is visible to
    query i iff i - W < j <= i, so a query sees at most W keys, its own
    included. window = 0 means no window; a window needs causal.
  * grouped-query attention: query head h reads key/value head h // (Hq/Hkv).
  * LSE_i = ln sum_j exp(scale * q_i . k_j) over the visible keys: the natural
    log-sum-exp of the scaled, masked scores.
  * backward: the exact analytic gradient of Eq. (1) for the loss
    L = sum(dO * O); the page gives no backward equations. With
    P = softmax(S), S = scale * Q K^T:
        dV = P^T dO,  dP = dO V^T,  Dvec_i = sum_j P_ij dP_ij,
        dS = P * (dP - Dvec),  dQ = scale * dS K,  dK = scale * dS^T Q,
    and dK, dV of a key/value head sum over the query heads of its group.

Layout of every tensor argument (numpy arrays of any float dtype; they are
upcast exactly to float64): q, o, dO, dq: [B, S, Hq, D]; k, v, dk, dv:
[B, S, Hkv, D]; lse: [B, Hq, S].
"""
import numpy as np

__all__ = [
    "attn_ref_probs",
    "attn_ref_fwd",
    "attn_ref_bwd",
    "attn_ref_rows_fwd",
    "attn_ref_rows_dq",
    "attn_ref_keys_dkdv",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _group(Hq, Hkv):
    """Query heads per key/value head; query head h reads kv head h // G."""
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} is not a multiple of Hkv={Hkv}")
    return Hq // Hkv


def _check_window(causal, window):
    if window < 0 or (window > 0 and not causal):
        raise ValueError(f"window={window} needs causal attention and must be >= 0")


def _scores(qh, kh, scale, causal, row0=0, window=0):
    """S = scale * Q K^T for query rows row0.. of one head, masked entries -inf.

    qh: [n, D] query rows (absolute positions row0..row0+n-1), kh: [S, D].
    """
    _check_window(causal, window)
    s = scale * (qh @ kh.T)
    if causal:
        rows = row0 + np.arange(qh.shape[0])[:, None]
        cols = np.arange(kh.shape[0])[None, :]
        s[cols > rows] = -np.inf
        if window > 0:
            s[cols <= rows - window] = -np.inf
    return s


def _softmax_rows(s):
    """Row softmax of a score block, and the natural log-sum-exp of each row."""
    m = np.max(s, axis=1)
    p = np.exp(s - m[:, None])          # masked entries: exp(-inf) = 0 exactly
    l = np.sum(p, axis=1)
    p /= l[:, None]
    return p, m + np.log(l)


def attn_ref_probs(q, k, causal, scale, b=0, h=0, window=0):
    """The full attention-probability matrix P = softmax(scale Q K^T) of one
    (batch, query head), Eq. (1). Returned for the oracle's own pins."""
    q, k = _f64(q), _f64(k)
    G = _group(q.shape[2], k.shape[2])
    p, _ = _softmax_rows(_scores(q[b, :, h, :], k[b, :, h // G, :], scale, causal, window=window))
    return p


def attn_ref_fwd(q, k, v, causal, scale, window=0):
    """Forward attention, Eq. (1), per (batch, query head).

    Returns (o [B,S,Hq,D] float64, lse [B,Hq,S] float64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, D = q.shape
    G = _group(Hq, k.shape[2])
    o = np.zeros((B, S, Hq, v.shape[3]))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p, lse[b, h] = _softmax_rows(_scores(q[b, :, h, :], k[b, :, g, :], scale, causal,
                                                 window=window))
            o[b, :, h, :] = p @ v[b, :, g, :]
    return o, lse


def attn_ref_bwd(q, k, v, do, causal, scale, window=0):
    """Exact gradients of L = sum(dO * O) with respect to q, k, v.

    Recomputes P from q, k (it takes nothing from a forward run) and returns
    (dq [B,S,Hq,D], dk [B,S,Hkv,D], dv [B,S,Hkv,D]) in float64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = _group(Hq, Hkv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            qh, kh, vh, doh = q[b, :, h, :], k[b, :, g, :], v[b, :, g, :], do[b, :, h, :]
            p, _ = _softmax_rows(_scores(qh, kh, scale, causal, window=window))
            dp = doh @ vh.T
            dvec = np.sum(p * dp, axis=1)
            ds = p * (dp - dvec[:, None])
            dq[b, :, h, :] = scale * (ds @ kh)
            dk[b, :, g, :] += scale * (ds.T @ qh)
            dv[b, :, g, :] += p.T @ doh
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Row-subset forms for sequence lengths where the full S x S oracle is too slow.
# Each computes exactly the same quantities as the full functions above for the
# selected rows; the test suite checks that agreement at moderate sizes.
# ---------------------------------------------------------------------------

def attn_ref_rows_fwd(q, k, v, causal, scale, rows, window=0):
    """O_i and LSE_i for selected query rows.

    rows: iterable of (b, h, i). Returns (o [n, D], lse [n]) in float64.
    """
    G = _group(q.shape[2], k.shape[2])
    out_o, out_l = [], []
    for b, h, i in rows:
        g = h // G
        qi = _f64(q[b, i, h, :])[None, :]
        kh = _f64(k[b, :, g, :])
        p, l = _softmax_rows(_scores(qi, kh, scale, causal, row0=i, window=window))
        out_o.append((p @ _f64(v[b, :, g, :]))[0])
        out_l.append(l[0])
    return np.array(out_o), np.array(out_l)


def attn_ref_rows_dq(q, k, v, do, causal, scale, rows, window=0):
    """dQ_i for selected query rows: scale * sum_j P_ij (dP_ij - Dvec_i) k_j.

    Row i's gradient needs only that row's probabilities, so each row is
    computed on its own. rows: iterable of (b, h, i). Returns [n, D].
    """
    G = _group(q.shape[2], k.shape[2])
    out = []
    for b, h, i in rows:
        g = h // G
        kh, vh = _f64(k[b, :, g, :]), _f64(v[b, :, g, :])
        qi = _f64(q[b, i, h, :])[None, :]
        p, _ = _softmax_rows(_scores(qi, kh, scale, causal, row0=i, window=window))
        dp = _f64(do[b, i, h, :])[None, :] @ vh.T
        dvec = np.sum(p * dp, axis=1)
        ds = p * (dp - dvec[:, None])
        out.append(scale * (ds @ kh)[0])
    return np.array(out)


def attn_ref_keys_dkdv(q, k, v, do, causal, scale, b, g, keys, row_block=512, window=0):
    """dK_j and dV_j for selected key rows j of key/value head g in batch b.

    The gradients of a key row sum over every query row of the G query heads
    that read head g, so all of those rows' probabilities are recomputed, one
    block of query rows at a time. Returns (dk [n, D], dv [n, D]).
    """
    B, S, Hq, D = q.shape
    G = _group(Hq, k.shape[2])
    keys = np.asarray(list(keys), dtype=np.int64)
    kh, vh = _f64(k[b, :, g, :]), _f64(v[b, :, g, :])
    dk = np.zeros((keys.size, kh.shape[1]))
    dv = np.zeros((keys.size, vh.shape[1]))
    for h in range(g * G, (g + 1) * G):
        for r0 in range(0, S, row_block):
            r1 = min(S, r0 + row_block)
            qh = _f64(q[b, r0:r1, h, :])
            doh = _f64(do[b, r0:r1, h, :])
            p, _ = _softmax_rows(_scores(qh, kh, scale, causal, row0=r0, window=window))
            dp = doh @ vh.T
            dvec = np.sum(p * dp, axis=1)
            ds = p * (dp - dvec[:, None])
            dk += scale * (ds[:, keys].T @ qh)
            dv += p[:, keys].T @ doh
    return dk, dv
