"""ra_dynamic_cp (C ABI, host only) against the oracle's Dynamic-CP sizing,
and its result used as a ring plan's per-document cp sizes."""

import numpy as np
import pytest

from oracle import dynamic_cp as DC
from workloads.synth import varlen_doc_lengths


@pytest.fixture(scope="module")
def ra(lib_path):
    import context_ring_attention_step_gb300 as m
    m.load_library(lib_path)
    return m


CASES = [
    ([5000, 300, 1200, 64, 64, 9000, 2048, 1, 700], 8, 3000, True, 1.0, 0.5),
    ([5000, 300, 1200, 64, 64, 9000, 2048, 1, 700], 8, 4000, True, 1.0, 0.5),
    ([16000, 500, 400, 300, 200], 8, 4096, True, 1e-12, 0.0),
    ([7, 5, 4, 4, 3, 3, 2], 2, 100, False, 1.0, 0.0),
    ([1], 1, 1, True, 1.0, 0.0),
    ([0, 10, 0], 4, 5, True, 1.0, 1.0),
    (varlen_doc_lengths(), 8, 8192, True, 7e-13, 2e-9),
    (varlen_doc_lengths(), 8, 12288, True, 7e-13, 2e-9),
    (varlen_doc_lengths(), 16, 4096, True, 7e-13, 0.0),
    (list(np.random.default_rng(3).integers(1, 20000, 200)), 64, 12000, True, 1e-12, 1e-9),
]


@pytest.mark.parametrize("mode", ["dynamic", "static"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_matches_oracle(ra, case, mode):
    lengths, n, cap, causal, a, b = CASES[case]
    lengths = [int(x) for x in lengths]
    try:
        cp, first, load, tok = DC.place(lengths, n, cap, causal, a, b, mode)
    except ValueError:
        with pytest.raises(ra.RingAttnError):
            ra.dynamic_cp(lengths, n, cap, causal, a, b, mode)
        return
    got = ra.dynamic_cp(lengths, n, cap, causal, a, b, mode)
    assert got["cp_per_doc"] == cp
    assert got["first_rank"] == first
    assert got["rank_tokens"] == tok
    assert np.allclose(got["rank_load"], load, rtol=1e-12, atol=0)


def test_refusals(ra):
    with pytest.raises(ra.RingAttnError) as e:
        ra.dynamic_cp([10000], 2, 4000)
    assert e.value.status == 1 and "memory" in str(e.value)
    with pytest.raises(ra.RingAttnError):
        ra.dynamic_cp([10], 3, 100)
    with pytest.raises(ra.RingAttnError):
        ra.dynamic_cp([10], 2, 0)
    with pytest.raises(ra.RingAttnError):
        ra.dynamic_cp([-1], 2, 10)


def test_dynamic_sizes_drive_a_ring_plan(ra):
    """The sizes are valid per-document cp for ra_plan_create; the plan covers
    every visible pair, and the dynamic choice balances the modelled work
    better than the static one, within the memory limit, splitting only the
    sequences that need it."""
    lengths = varlen_doc_lengths()
    got = ra.dynamic_cp(lengths, 8, 12288)
    st = ra.dynamic_cp(lengths, 8, 12288, mode="static")
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    plan = ra.Plan(cu, got["cp_per_doc"], "zigzag", True, 32, 8, 128)
    assert plan.stats()["visible_pairs"] == sum(L * (L + 1) // 2 for L in lengths)
    assert max(got["rank_tokens"]) <= 12288
    assert DC.imbalance(got["rank_load"]) <= DC.imbalance(st["rank_load"])
    assert sum(c == 1 for c in got["cp_per_doc"]) > len(lengths) // 2
