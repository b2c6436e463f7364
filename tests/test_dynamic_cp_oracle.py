"""Pins of the Dynamic-CP sizing oracle (oracle/dynamic_cp.py) against brute
force and the page's statements (Dynamic-CP page: quadratic cost model,
power-of-two CP groups, static size set by the longest sequence)."""

import itertools

import pytest

from oracle import dynamic_cp as DC


@pytest.mark.parametrize("L", [1, 2, 5, 17, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_pairs_is_the_count_of_visible_pairs(L, causal):
    brute = sum(1 for q in range(L) for k in range(L) if not causal or k <= q)
    assert DC.pairs(L, causal) == brute


def test_cost_is_quadratic_plus_linear():
    t = [DC.seq_time(L, True, 2.0, 3.0) for L in (10, 20, 40)]
    assert t[0] == 2.0 * 55 + 30 and t[1] == 2.0 * 210 + 60 and t[2] == 2.0 * 820 + 120


@pytest.mark.parametrize("L,cap,n", [(1, 1, 1), (100, 30, 8), (100, 100, 8), (129, 64, 4), (4096, 1000, 4)])
def test_min_pow2_cp_is_the_smallest_fitting_power_of_two(L, cap, n):
    c = DC.min_pow2_cp(L, cap, n)
    fits = [x for x in (1, 2, 4, 8, 16) if x <= n and -(-L // x) <= cap]
    assert c == (min(fits) if fits else 0)


def _dynamic_sizes(lengths, num_ranks, cap, causal):
    """The dynamic group sizes restated: smallest power of two that fits memory
    and leaves no rank above the balanced share."""
    t = [DC.seq_time(L, causal, 1.0, 0.0) for L in lengths]
    share = sum(t) / num_ranks
    out = []
    for L, ti in zip(lengths, t):
        ok = [c for c in (1, 2, 4, 8, 16, 32) if c <= num_ranks and -(-L // c) <= cap and
              (ti / c <= share or c == num_ranks)]
        out.append(min(ok))
    return out


def _brute_best(lengths, num_ranks, cap, causal):
    """Optimal busiest-rank load over every placement with the dynamic group sizes."""
    base = _dynamic_sizes(lengths, num_ranks, cap, causal)
    times = [DC.seq_time(L, causal, 1.0, 0.0) for L in lengths]
    choices = [list(range(num_ranks // c)) for c in base]
    best = None
    for gs in itertools.product(*choices):
        load, tok = [0.0] * num_ranks, [0] * num_ranks
        for L, c, g, t in zip(lengths, base, gs, times):
            for r in range(g * c, (g + 1) * c):
                load[r] += t / c
                tok[r] += -(-L // c)
        if max(tok) <= cap and (best is None or max(load) < best):
            best = max(load)
    return best


@pytest.mark.parametrize("lengths,n", [([7, 5, 4, 4, 3, 3, 2], 2), ([6, 6, 5, 5, 5, 4, 4, 3, 3], 4),
                                       ([12, 12, 11, 10, 9, 9, 2], 4), ([8, 8, 7, 6, 5, 1], 2)])
def test_greedy_is_within_the_lpt_bound_of_brute_force(lengths, n):
    """Every sequence fits one rank (group size 1): the placement is
    longest-processing-time-first on identical ranks, at most
    (4/3 - 1/(3 m)) of the optimum (Graham's bound), checked by brute force."""
    cap = 1000
    cp, first, load, tok = DC.place(lengths, n, cap, True)
    assert cp == _dynamic_sizes(lengths, n, cap, True)
    if cp != [1] * len(lengths):
        pytest.skip("not a group-size-1 case")
    opt = _brute_best(lengths, n, cap, True)
    assert max(load) <= (4.0 / 3.0 - 1.0 / (3 * n)) * opt + 1e-9


@pytest.mark.parametrize("lengths,n,cap", [([40, 12, 12, 11, 10, 9], 4, 30), ([30, 8, 8, 7, 6, 5, 1], 4, 20)])
def test_greedy_with_groups_respects_memory_and_stays_near_brute_force(lengths, n, cap):
    cp, first, load, tok = DC.place(lengths, n, cap, True)
    opt = _brute_best(lengths, n, cap, True)
    assert opt is not None and max(tok) <= cap
    assert max(load) <= 1.5 * opt + 1e-9


def test_placement_invariants():
    lengths = [5000, 300, 1200, 64, 64, 9000, 2048, 1, 700]
    cp, first, load, tok = DC.place(lengths, 8, 3000, True, 1.0, 0.5)
    for L, c, f in zip(lengths, cp, first):
        assert c & (c - 1) == 0 and f % c == 0 and f + c <= 8
        assert -(-L // c) <= 3000
    # loads and tokens are the sums they claim to be
    want_load, want_tok = [0.0] * 8, [0] * 8
    for L, c, f in zip(lengths, cp, first):
        for r in range(f, f + c):
            want_load[r] += DC.seq_time(L, True, 1.0, 0.5) / c
            want_tok[r] += -(-L // c)
    assert all(abs(a - b) <= 1e-9 * max(1.0, b) for a, b in zip(load, want_load))
    assert tok == want_tok
    assert abs(sum(load) - sum(DC.seq_time(L, True, 1.0, 0.5) for L in lengths)) < 1e-6


def test_static_size_is_set_by_the_longest_sequence():
    lengths = [16000, 500, 400, 300, 200]
    cp_s, _, load_s, _ = DC.place(lengths, 8, 4096, mode="static")
    cp_d, _, load_d, _ = DC.place(lengths, 8, 4096, mode="dynamic")
    assert cp_s == [4] * 5            # ceil(16000 / 4) = 4000 <= 4096: every sequence split 4 ways
    # dynamic: the long one carries almost all the work and spreads over all 8
    # ranks; the short ones stay whole (no ring traffic for them)
    assert cp_d == [8, 1, 1, 1, 1]
    assert DC.imbalance(load_d) < DC.imbalance(load_s)
    assert DC.exchanged_tokens(lengths[1:], cp_d[1:]) == 0 < DC.exchanged_tokens(lengths[1:], cp_s[1:])


def test_a_sequence_that_fits_no_rank_is_refused():
    with pytest.raises(ValueError):
        DC.place([10000], 2, 4000)
    with pytest.raises(ValueError):
        DC.place([10], 3, 100)   # not a power of two


def test_planted_mistake_in_the_load_sum_is_caught():
    """A load that forgot to divide by the group size breaks the invariants test."""
    lengths = [400, 100]
    cp, first, load, tok = DC.place(lengths, 4, 150, True)
    bad = [0.0] * 4
    for L, c, f in zip(lengths, cp, first):
        for r in range(f, f + c):
            bad[r] += DC.seq_time(L, True, 1.0, 0.0)   # missing / c
    assert any(abs(a - b) > 1e-6 for a, b in zip(load, bad))



def test_dynamic_sizes_bound_each_sequence_by_the_balanced_share():
    lengths = [30000, 12000, 3000, 2500, 800, 600, 100]
    n = 8
    cp, first, load, tok = DC.place(lengths, n, 40000, True)
    t = [DC.seq_time(L, True, 1.0, 0.0) for L in lengths]
    share = sum(t) / n
    assert cp == _dynamic_sizes(lengths, n, 40000, True)
    for ti, c in zip(t, cp):
        assert ti / c <= share or c == n
        assert c == 1 or ti / (c // 2) > share   # and no larger than needed
    assert DC.imbalance(load) < 1.5
