"""Ring-decomposed attention in float64.  TEST INFRASTRUCTURE ONLY.

The same result as ``oracle.attention`` reached the way ring attention
reaches it, used to pin the invariant that ring attention equals standard
attention (NVSHMEM/XLA page, "Paralelismo de contexto y atencion en anillo").

Steps, in the pages' order:

1. Shard Q, K, V along the sequence into cp parts (Accelerate guide,
   "Detalhes tecnicos": sharding dimension D over N ranks gives parts of
   size D//N).  Two layouts, read per document of length L:
   * contiguous: boundaries floor(k L / cp), k = 0..cp; shard r is
     [b_r, b_{r+1});
   * zigzag (load-balanced for causal masks; not on the pages): boundaries
     floor(k L / (2 cp)), k = 0..2cp, chunks C_k = [b_k, b_{k+1}); shard r is
     C_r united with C_{2cp-1-r}.
2. Ring: at step s, shard r holds key/value shard (r - s) mod cp (each rank
   receives from its left neighbour every step; the guide's pseudocode loops
   j over all shards).  Step 0 is the local shard.
3. Each step computes a partial attention of Q_r against K_j, V_j with the
   mask taken on global positions (same document, key <= query when causal),
   giving a normalised partial output and its log-sum-exp (-inf and O = 0 for
   rows that see no key in that shard).
4. ``combine`` (undefined on the pages; read as the exact merge):
   lse = max(a, b) + ln(1 + exp(-|a - b|)), O = exp(a - lse) O_a + exp(b - lse) O_b,
   where a merge with an -inf side returns the other side.

The backward is decomposed the same way: with the final LSE and
Delta = <dO, O> known, each (query shard, key/value shard) pair contributes its
own exact share of dq, dk and dv.
"""

from __future__ import annotations

import numpy as np


def chunk_bounds(L: int, cp: int, layout: str) -> list:
    """Document-local boundaries of the layout's chunks (step 1)."""
    n = 2 * cp if layout == "zigzag" else cp
    return [(k * L) // n for k in range(n + 1)]


def shard_ranges(L: int, cp: int, layout: str, r: int) -> list:
    """Document-local [begin, end) ranges making up shard r (step 1)."""
    b = chunk_bounds(L, cp, layout)
    if layout == "zigzag":
        return [(b[r], b[r + 1]), (b[2 * cp - 1 - r], b[2 * cp - r])]
    return [(b[r], b[r + 1])]


def ring_source(r: int, s: int, cp: int) -> int:
    """Key/value shard that shard r holds at ring step s (step 2)."""
    return (r - s) % cp


def _positions(ranges, base):
    if not ranges:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(base + a, base + b) for a, b in ranges]).astype(np.int64)


def partial_attention(q_rows, k_rows, v_rows, qpos, kpos, causal, scale):
    """Step 3: normalised partial O [n, d] and LSE [n] of one shard pair."""
    n = q_rows.shape[0]
    o = np.zeros((n, v_rows.shape[1]))
    lse = np.full(n, -np.inf)
    if n == 0 or k_rows.shape[0] == 0:
        return o, lse
    s = scale * (q_rows @ k_rows.T)
    if causal:
        s = np.where(kpos[None, :] <= qpos[:, None], s, -np.inf)
    seen = np.isfinite(s).any(axis=1)
    if not seen.any():
        return o, lse
    ss = s[seen]
    m = ss.max(axis=1, keepdims=True)
    lse[seen] = m[:, 0] + np.log(np.exp(ss - m).sum(axis=1))
    o[seen] = np.exp(ss - lse[seen][:, None]) @ v_rows
    return o, lse


def merge(o_a, lse_a, o_b, lse_b):
    """Step 4, row by row: exact merge of two normalised partials."""
    o = o_a.copy()
    lse = lse_a.copy()
    only_b = np.isneginf(lse_a) & ~np.isneginf(lse_b)
    o[only_b] = o_b[only_b]
    lse[only_b] = lse_b[only_b]
    both = ~np.isneginf(lse_a) & ~np.isneginf(lse_b)
    a, b = lse_a[both], lse_b[both]
    new = np.maximum(a, b) + np.log1p(np.exp(-np.abs(a - b)))
    o[both] = np.exp(a - new)[:, None] * o_a[both] + np.exp(b - new)[:, None] * o_b[both]
    lse[both] = new
    return o, lse


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def ring_attention_fwd(q, k, v, cu_seqlens, cp_per_doc, layout, causal=True, scale=None):
    """O [T,Hq,d] and LSE [Hq,T] reached by running the ring, float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.zeros((T, Hq, v.shape[2]))
    lse = np.full((Hq, T), -np.inf)
    cu = [int(c) for c in cu_seqlens]
    for doc in range(len(cu) - 1):
        base, L, cp = cu[doc], cu[doc + 1] - cu[doc], int(cp_per_doc[doc])
        if L == 0:
            continue
        for r in range(cp):
            qpos = _positions(shard_ranges(L, cp, layout, r), base)
            for h in range(Hq):
                g = h // G
                run_o = np.zeros((len(qpos), v.shape[2]))
                run_l = np.full(len(qpos), -np.inf)
                for s in range(cp):
                    j = ring_source(r, s, cp)
                    kpos = _positions(shard_ranges(L, cp, layout, j), base)
                    po, pl = partial_attention(q[qpos, h], k[kpos, g], v[kpos, g],
                                               qpos, kpos, causal, scale)
                    run_o, run_l = merge(run_o, run_l, po, pl)
                o[qpos, h] = run_o
                lse[h, qpos] = run_l
    return o, lse


def ring_attention_bwd(q, k, v, do, o, lse, cu_seqlens, cp_per_doc, layout,
                       causal=True, scale=None):
    """(dq, dk, dv) summed over ring steps, given the final O and LSE."""
    q, k, v, do, o, lse = (_f64(x) for x in (q, k, v, do, o, lse))
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    cu = [int(c) for c in cu_seqlens]
    for doc in range(len(cu) - 1):
        base, L, cp = cu[doc], cu[doc + 1] - cu[doc], int(cp_per_doc[doc])
        if L == 0:
            continue
        for s in range(cp):
            for r in range(cp):
                j = ring_source(r, s, cp)
                qpos = _positions(shard_ranges(L, cp, layout, r), base)
                kpos = _positions(shard_ranges(L, cp, layout, j), base)
                if len(qpos) == 0 or len(kpos) == 0:
                    continue
                for h in range(Hq):
                    g = h // G
                    s_ij = scale * (q[qpos, h] @ k[kpos, g].T)
                    if causal:
                        s_ij = np.where(kpos[None, :] <= qpos[:, None], s_ij, -np.inf)
                    p = np.exp(s_ij - lse[h, qpos][:, None])
                    delta = (do[qpos, h] * o[qpos, h]).sum(axis=1)
                    dp = do[qpos, h] @ v[kpos, g].T
                    ds = p * (dp - delta[:, None])
                    dq[qpos, h] += scale * (ds @ k[kpos, g])
                    dk[kpos, g] += scale * (ds.T @ q[qpos, h])
                    dv[kpos, g] += p.T @ do[qpos, h]
    return dq, dk, dv
