"""Dynamic context-parallel sizing in plain Python.  TEST INFRASTRUCTURE ONLY.

Follows the Dynamic-CP page ("Modelado del programador de datos", "Necesidad
de un enfoque dinamico", "Construccion de multiples grupos de contexto
paralelo por rango"):

* cost model: a sample's time grows with the square of its length (attention)
  plus a linear part.  Written here as
      time(L) = sec_per_pair * pairs(L) + sec_per_token * L,
  pairs(L) = L (L + 1) / 2 causal, L * L without a mask (the visible (q, k)
  pairs, i.e. the attention work);
* CP group sizes are powers of two from 1 to the number of ranks;
* a static CP size is set by the longest sequence of the batch (so shorter
  sequences are split too); the dynamic choice gives each sequence the
  smallest group that fits the per-rank memory limit and does not leave any
  one rank of the group more than the balanced share of the batch's time
  (sum of time(L) over the ranks): the page wants both the compute balance
  across data-parallel groups and no needless CP communication;
* the page's solver is "a heuristic" without further detail.  Reading taken:
  longest-processing-time-first placement of each sequence on an aligned
  group of its size (ranks [g * cp, (g + 1) * cp)), choosing the group whose
  busiest rank ends least loaded, within the per-rank token limit; a sequence
  that fits no group moves to the next larger group size.

Each rank's load is the sum of time(L) / cp over the sequences it holds
(zigzag sharding splits a causal sequence's work evenly over its group);
its tokens are the sum of ceil(L / cp).
"""

from __future__ import annotations

import math


def pairs(L: int, causal: bool = True) -> int:
    """Visible (query, key) pairs of one sequence of length L."""
    return L * (L + 1) // 2 if causal else L * L


def seq_time(L: int, causal: bool, sec_per_pair: float, sec_per_token: float) -> float:
    return sec_per_pair * pairs(L, causal) + sec_per_token * L


def min_pow2_cp(L: int, max_tokens_per_rank: int, num_ranks: int) -> int:
    """Smallest power-of-two group size whose shard of L fits the limit (0 if none)."""
    c = 1
    while c <= num_ranks:
        if -(-L // c) <= max_tokens_per_rank:
            return c
        c *= 2
    return 0


def place(lengths, num_ranks, max_tokens_per_rank, causal=True, sec_per_pair=1.0, sec_per_token=0.0,
          mode="dynamic"):
    """Group size and first rank per sequence, and each rank's load and tokens.

    mode "dynamic": each sequence starts at its smallest fitting group size.
    mode "static": every sequence gets the group size of the longest one.
    Returns (cp, first, load, tokens); raises ValueError if a sequence fits nowhere.
    """
    if num_ranks < 1 or num_ranks & (num_ranks - 1):
        raise ValueError("num_ranks must be a power of two")
    n = len(lengths)
    base = [min_pow2_cp(L, max_tokens_per_rank, num_ranks) if L > 0 else 1 for L in lengths]
    if any(c == 0 for c in base):
        raise ValueError("a sequence exceeds the memory of all ranks")
    times = [seq_time(L, causal, sec_per_pair, sec_per_token) for L in lengths]
    if mode == "static":
        top = max(base) if base else 1
        base = [top] * n
    else:
        share = sum(times) / num_ranks  # balanced time per rank
        for i in range(n):
            while base[i] < num_ranks and times[i] / base[i] > share:
                base[i] *= 2
    order = sorted(range(n), key=lambda i: (-times[i], i))
    load = [0.0] * num_ranks
    tokens = [0] * num_ranks
    cp = [0] * n
    first = [0] * n
    for i in order:
        c = base[i]
        while True:
            share = -(-lengths[i] // c)
            best = None
            for g in range(num_ranks // c):
                ranks = range(g * c, (g + 1) * c)
                if any(tokens[r] + share > max_tokens_per_rank for r in ranks):
                    continue
                end = max(load[r] for r in ranks) + times[i] / c
                if best is None or end < best[0]:
                    best = (end, g)
            if best is not None:
                break
            c *= 2
            if c > num_ranks:
                raise ValueError("the batch does not fit the ranks' memory")
        g = best[1]
        cp[i], first[i] = c, g * c
        for r in range(g * c, (g + 1) * c):
            load[r] += times[i] / c
            tokens[r] += -(-lengths[i] // c)
    return cp, first, load, tokens


def imbalance(load) -> float:
    """Busiest rank over the mean (1.0 = perfectly balanced)."""
    mean = sum(load) / len(load)
    return max(load) / mean if mean > 0 else 1.0


def exchanged_tokens(lengths, cp) -> int:
    """Key/value tokens a ring moves per pass: every rank of a group of size c
    receives the other c - 1 shards, L (c - 1) / c tokens per rank."""
    return sum(L * (c - 1) for L, c in zip(lengths, cp))


def log2_int(c: int) -> int:
    return int(math.log2(c))
