"""Workload definitions and seeded bf16 inputs for ring attention.

Shapes follow the five synthetic workloads the build is measured on: a tiny
multi-head case, the Llama-3-8B attention shape (32 query heads, 8 key/value
heads, head_dim 128) at 32K, 128K and 256K tokens, and a packed
variable-length batch in THD layout with ``cu_seqlens`` (the Dynamic-CP page,
section "Reprogramacion dinamica y empaquetado de datos").

Every tensor is drawn as float32 N(0, 1) from ``numpy.random.default_rng(seed)``
in the order q, k, v, dO and rounded to bf16 (round to nearest even).  The
same host tensors feed the GPU library and the oracle.

Nothing here computes attention.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                     # total packed tokens
    Hq: int                    # query heads
    Hkv: int                   # key/value heads (GQA groups of Hq // Hkv)
    d: int                     # head_dim
    cu_seqlens: tuple          # int prefix sums, len = num_docs + 1, last == T
    cp_per_doc: tuple          # ring size (cp_size) of every document
    layout: str                # "zigzag" or "contiguous"
    causal: bool
    seed: int
    scale: float = field(default=0.0)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.d)

    @property
    def num_docs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def doc_lengths(self) -> list:
        cu = self.cu_seqlens
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    def with_layout(self, layout: str) -> "Workload":
        return Workload(self.name + "_" + layout, self.T, self.Hq, self.Hkv, self.d,
                        self.cu_seqlens, self.cp_per_doc, layout, self.causal,
                        self.seed, self.scale)


def varlen_doc_lengths(n_docs: int = 40, total: int = 65536, mu: float = 7.5,
                       sigma: float = 1.2, lo: int = 128, hi: int = 32768,
                       seed: int = 1234) -> list:
    """Lognormal document lengths rescaled to sum to exactly ``total``.

    Draw ``n_docs`` lengths round(exp(N(mu, sigma^2))), clip them to
    [lo, hi], scale them proportionally (floor) so they sum to ``total``,
    re-clip, then hand the remaining tokens one by one to the largest
    documents (or take them back, if clipping overshot).
    """
    rng = np.random.default_rng(seed)
    raw = np.clip(np.rint(np.exp(rng.normal(mu, sigma, n_docs))), lo, hi)
    lens = np.floor(raw * total / raw.sum()).astype(np.int64)
    lens = np.clip(lens, lo, hi)
    order = np.argsort(-lens, kind="stable")
    diff = int(total - lens.sum())
    i = 0
    while diff != 0:
        idx = order[i % n_docs]
        step = 1 if diff > 0 else -1
        if lo <= lens[idx] + step <= hi:
            lens[idx] += step
            diff -= step
        i += 1
    return [int(x) for x in lens]


def _single(name, T, Hq, Hkv, d, cp, layout, seed, scale=0.0):
    return Workload(name, T, Hq, Hkv, d, (0, T), (cp,), layout, True, seed, scale)


def _varlen():
    lens = varlen_doc_lengths()
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    cps = tuple(min(8, -(-L // 4096)) for L in lens)
    return Workload("varlen_65k", cu[-1], 32, 8, 128, tuple(cu), cps, "zigzag", True, 4)


CONFIGS = {
    "tiny": _single("tiny", 512, 2, 2, 64, 4, "zigzag", 1, 1.0 / 8.0),
    "llama3_8b_32k": _single("llama3_8b_32k", 32768, 32, 8, 128, 8, "zigzag", 2),
    "long_128k": _single("long_128k", 131072, 32, 8, 128, 16, "zigzag", 3),
    "varlen_65k": _varlen(),
    "max_256k": _single("max_256k", 262144, 32, 8, 128, 32, "zigzag", 5),
    # beyond the five parity configurations: the no-mask mode and head_dim 64 / 256 at 128K
    "long_128k_noncausal": Workload("long_128k_noncausal", 131072, 32, 8, 128, (0, 131072), (16,), "zigzag",
                                    False, 6),
    "long_128k_d64": _single("long_128k_d64", 131072, 32, 8, 64, 16, "zigzag", 7),
    # head_dim 256 at 128K (16 query / 8 key-value heads: the same useful FLOPs as 32 heads at 128)
    "long_128k_d256": _single("long_128k_d256", 131072, 16, 8, 256, 16, "zigzag", 8),
}


def workload(name: str) -> Workload:
    if name.endswith("_contiguous") or name.endswith("_zigzag"):
        base, layout = name.rsplit("_", 1)
        return CONFIGS[base].with_layout(layout)
    return CONFIGS[name]


def custom(T_or_lengths, Hq, Hkv, d, cp, layout="zigzag", causal=True, seed=0,
           scale=0.0, name="custom") -> Workload:
    """A workload from a list of document lengths (or one length) and a ring size.

    ``cp`` is one int for every document or a list with one entry per document.
    """
    lens = [T_or_lengths] if isinstance(T_or_lengths, int) else list(T_or_lengths)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + int(L))
    cps = tuple(cp) if isinstance(cp, (list, tuple)) else tuple([cp] * len(lens))
    return Workload(name, cu[-1], Hq, Hkv, d, tuple(cu), cps, layout, causal, seed, scale)


def _draw_bf16(rng, shape, chunk_rows=8192):
    """Draw float32 N(0,1) row-chunk by row-chunk, rounding each chunk to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    T = shape[0]
    for t0 in range(0, T, chunk_rows):
        t1 = min(T, t0 + chunk_rows)
        x = rng.standard_normal(size=(t1 - t0,) + tuple(shape[1:]), dtype=np.float32)
        out[t0:t1] = torch.from_numpy(x).to(torch.bfloat16)
    return out


def draw_qkvdo(wl: Workload, seed: int | None = None):
    """q [T,Hq,d], k [T,Hkv,d], v [T,Hkv,d], dO [T,Hq,d]: bf16 CPU tensors."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    q = _draw_bf16(rng, (wl.T, wl.Hq, wl.d))
    k = _draw_bf16(rng, (wl.T, wl.Hkv, wl.d))
    v = _draw_bf16(rng, (wl.T, wl.Hkv, wl.d))
    do = _draw_bf16(rng, (wl.T, wl.Hq, wl.d))
    return q, k, v, do
