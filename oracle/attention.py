"""Monolithic masked softmax attention in float64.  TEST INFRASTRUCTURE ONLY.

Definition followed (ring attention computes exactly this, per the NVSHMEM/XLA
page, section "Paralelismo de contexto y atencion en anillo": the ring keeps
mathematical equivalence with standard attention):

For a packed batch in THD layout with document boundaries ``cu_seqlens``
(Dynamic-CP page, "Reprogramacion dinamica y empaquetado de datos"), query
head h reads key/value head g = h // (Hq // Hkv) (contiguous GQA groups), and
query i sees key j iff both lie in the same document and, when causal, j <= i
(Accelerate guide: SDPA "sem mascara ou com mascara causal").

    s_ij  = scale * <q_i, k_j>                       visible j only
    LSE_i = ln sum_j exp(s_ij)                       natural log
    P_ij  = exp(s_ij - LSE_i)
    O_i   = sum_j P_ij v_j

Backward of f = <dO, O>:

    Delta_i = <dO_i, O_i>,  dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - Delta_i)
    dq_i = scale sum_j dS_ij k_j
    dk_j = scale sum_{h in group} sum_i dS_ij q_i
    dv_j = sum_{h in group} sum_i P_ij dO_i

Rows are processed in blocks only to bound memory; every row's softmax is
taken over all of its visible keys at once (no online softmax, no ring).
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def _docs(cu_seqlens):
    cu = [int(c) for c in cu_seqlens]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1) if cu[i + 1] > cu[i]]


def _block_scores(q, k, h, g, r0, r1, b, e, causal, scale):
    """Scores of query rows [r0, r1) against the keys they may see, masked."""
    kend = r1 if causal else e
    s = scale * (q[r0:r1, h, :] @ k[b:kend, g, :].T)
    if causal:
        qpos = np.arange(r0, r1)[:, None]
        kpos = np.arange(b, kend)[None, :]
        s = np.where(kpos <= qpos, s, -np.inf)
    return s, kend


def _softmax_lse(s):
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    return lse, np.exp(s - lse[:, None])


def attention_fwd(q, k, v, cu_seqlens, causal=True, scale=None, heads=None,
                  row_block=256):
    """O [T,Hq,d] and LSE [Hq,T] (natural log), float64.

    ``heads`` restricts the computation to some query heads (the others are
    left at O = 0, LSE = -inf).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    heads = range(Hq) if heads is None else heads
    o = np.zeros((T, Hq, v.shape[2]))
    lse = np.full((Hq, T), -np.inf)
    for b, e in _docs(cu_seqlens):
        for h in heads:
            g = h // G
            for r0 in range(b, e, row_block):
                r1 = min(r0 + row_block, e)
                s, kend = _block_scores(q, k, h, g, r0, r1, b, e, causal, scale)
                l, p = _softmax_lse(s)
                o[r0:r1, h, :] = p @ v[b:kend, g, :]
                lse[h, r0:r1] = l
    return o, lse


def attention_bwd(q, k, v, do, cu_seqlens, causal=True, scale=None, heads=None,
                  row_block=256):
    """(dq, dk, dv, o, lse) in float64 for upstream gradient ``do``.

    With ``heads`` given, only those query heads contribute (dk/dv then hold
    the contribution of those heads only).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    heads = range(Hq) if heads is None else heads
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros((T, Hq, v.shape[2]))
    lse = np.full((Hq, T), -np.inf)
    for b, e in _docs(cu_seqlens):
        for h in heads:
            g = h // G
            for r0 in range(b, e, row_block):
                r1 = min(r0 + row_block, e)
                s, kend = _block_scores(q, k, h, g, r0, r1, b, e, causal, scale)
                l, p = _softmax_lse(s)
                vb = v[b:kend, g, :]
                ob = p @ vb
                o[r0:r1, h, :] = ob
                lse[h, r0:r1] = l
                dob = do[r0:r1, h, :]
                delta = (dob * ob).sum(axis=1)
                dp = dob @ vb.T
                ds = p * (dp - delta[:, None])
                dq[r0:r1, h, :] = scale * (ds @ k[b:kend, g, :])
                dk[b:kend, g, :] += scale * (ds.T @ q[r0:r1, h, :])
                dv[b:kend, g, :] += p.T @ dob
    return dq, dk, dv, o, lse


def attention_rows(q, k, v, cu_seqlens, rows, head, causal=True, scale=None):
    """O and LSE of single query rows of one head (exact, O(L d) per row).

    Used to check outputs sampled from workloads too large for the full
    oracle.  Returns (o [len(rows), d], lse [len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    g = head // G
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    cu = np.asarray([int(c) for c in cu_seqlens])
    o = np.zeros((len(rows), v.shape[2]))
    lse = np.zeros(len(rows))
    for n, i in enumerate(rows):
        doc = int(np.searchsorted(cu, i, side="right") - 1)
        b, e = int(cu[doc]), int(cu[doc + 1])
        kend = i + 1 if causal else e
        s = scale * (k[b:kend, g, :] @ q[i, head, :])
        m = s.max()
        lse[n] = m + np.log(np.exp(s - m).sum())
        o[n] = np.exp(s - lse[n]) @ v[b:kend, g, :]
    return o, lse


def attention_keys_dkdv(q, k, v, do, cu_seqlens, keys, kv_head, causal=True, scale=None):
    """dk and dv of single key rows of one key/value head (exact).

    For a key j of document [b, e) the gradients are sums over the queries
    that see it (i >= j when causal, the whole document otherwise) and over
    the query heads h of the key/value head's group:

        dv_j = sum_h sum_i P_ij dO_i,   dk_j = scale sum_h sum_i dS_ij q_i,
        dS_ij = P_ij (<dO_i, v_j> - Delta_i),   Delta_i = <dO_i, O_i>,

    where every P_ij needs the whole softmax row of query i (its LSE and O).
    So the cost is the number of queries seeing the keys times the document
    length: cheap for keys near a document's end under a causal mask, which
    is what the tests at full size ask for.  Returns (dk [len(keys), d],
    dv [len(keys), d]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    g = kv_head
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    cu = np.asarray([int(c) for c in cu_seqlens])
    keys = [int(j) for j in keys]
    dk = np.zeros((len(keys), d))
    dv = np.zeros((len(keys), v.shape[2]))
    # group the keys by document: one pass over the queries that see them
    by_doc = {}
    for n, j in enumerate(keys):
        by_doc.setdefault(int(np.searchsorted(cu, j, side="right") - 1), []).append(n)
    for doc, idx in by_doc.items():
        b, e = int(cu[doc]), int(cu[doc + 1])
        jpos = np.asarray([keys[n] for n in idx])
        i0 = int(jpos.min()) if causal else b   # first query that sees any of the keys
        for h in range(g * G, (g + 1) * G):
            for r0 in range(i0, e, 256):
                r1 = min(r0 + 256, e)
                # whole softmax rows of queries [r0, r1): LSE, O and Delta
                s, kend = _block_scores(q, k, h, g, r0, r1, b, e, causal, scale)
                lse, p = _softmax_lse(s)
                o = p @ v[b:kend, g, :]
                dob = do[r0:r1, h, :]
                delta = (dob * o).sum(axis=1)
                # probabilities and dS of these queries against the chosen keys
                sj = scale * (q[r0:r1, h, :] @ k[jpos, g, :].T)
                if causal:
                    sj = np.where(jpos[None, :] <= np.arange(r0, r1)[:, None], sj, -np.inf)
                pj = np.exp(sj - lse[:, None])
                dpj = dob @ v[jpos, g, :].T
                dsj = pj * (dpj - delta[:, None])
                dv[idx] += pj.T @ dob
                dk[idx] += scale * (dsj.T @ q[r0:r1, h, :])
    return dk, dv


def attention_rows_dq(q, k, v, do, cu_seqlens, rows, head, causal=True, scale=None):
    """dq of single query rows of one head (exact, O(L d) per row).

    Each row's softmax, its Delta = <dO_i, O_i> and its dq_i = scale sum_j
    P_ij (<dO_i, v_j> - Delta_i) k_j need only that row.  Returns [len(rows), d].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    g = head // G
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    cu = np.asarray([int(c) for c in cu_seqlens])
    dq = np.zeros((len(rows), d))
    for n, i in enumerate(rows):
        doc = int(np.searchsorted(cu, i, side="right") - 1)
        b, e = int(cu[doc]), int(cu[doc + 1])
        kend = i + 1 if causal else e
        s = scale * (k[b:kend, g, :] @ q[i, head, :])
        m = s.max()
        p = np.exp(s - m)
        p /= p.sum()
        vb = v[b:kend, g, :]
        o = p @ vb
        dp = vb @ do[i, head, :]
        ds = p * (dp - do[i, head, :] @ o)
        dq[n] = scale * (ds @ k[b:kend, g, :])
    return dq
