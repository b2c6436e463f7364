"""Host-side checks of the C-ABI library (no GPU): exports, planner, errors.

The planner is checked against the oracle's own restatement of the layouts
(``oracle.ring``), and its work items are expanded pair by pair to show that
every visible (query, key) pair is covered exactly once, at the ring step the
pairing rule assigns to it.
"""

import ctypes
import re

import pytest

from oracle import ring as R
from workloads import custom, workload

HEADER = "include/ring_attn.h"


def _declared():
    import os
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(here, HEADER)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


@pytest.fixture(scope="module")
def ra(lib_path):
    import context_ring_attention_step_gb300 as m
    m.load_library(lib_path)
    return m


def test_abi_version(ra):
    assert ra.load_library().ra_abi_version() == 2


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("lengths,cp", [([512], 4), ([10], 3), ([37, 3, 100], 5), ([1, 2, 7], 8)])
def test_shard_ranges_match_oracle_layout(ra, layout, lengths, cp):
    wl = custom(lengths, 2, 1, 64, cp, layout)
    plan = ra.Plan(wl.cu_seqlens, cp, layout, True, 2, 1, 64)
    for d, L in enumerate(lengths):
        base = wl.cu_seqlens[d]
        for r in range(cp):
            want = [(base + a, base + b) for a, b in R.shard_ranges(L, cp, layout, r)]
            assert plan.shard_token_ranges(d, r) == want


def _expand_fwd(items, off, causal):
    """{step: set of (q, k)} covered by forward items, with the causal mask applied."""
    cover = {}
    for s in range(len(off) - 1):
        pairs = []
        for it in items[off[s]:off[s + 1]]:
            q0, q1, kb0, ke0, kb1, ke1, flags, tiles = it
            assert q1 - q0 <= 256 and q1 > q0
            assert (flags == 1) == (s == 0)
            assert kb0 < ke0 and (kb1 == ke1 == 0 or ke0 <= kb1 < ke1)
            for q in range(q0, q1):
                for kb, ke in ((kb0, ke0), (kb1, ke1)):
                    for k in range(kb, ke):
                        if not causal or k <= q:
                            pairs.append((q, k))
        cover[s] = pairs
    return cover


def _expand_bwd(items, off, causal, head=0, pairs=False):
    """Pairs covered by the backward items of one key/value head.  With
    `pairs` (head_dim 128: CTA pairs over two key tiles) items come two by two,
    neighbouring key tiles with the same query ranges, the second possibly
    empty."""
    cover = {}
    for s in range(len(off) - 1):
        step = items[off[s]:off[s + 1]]
        if pairs:
            assert len(step) % 2 == 0
            for a, b in zip(step[0::2], step[1::2]):
                assert a[2:] == b[2:] and b[0] == a[1] and b[1] - b[0] <= 128
                assert a[1] - a[0] == 128 or b[1] == b[0]
        pairs_ = []
        for n, it in enumerate(step):
            k0, k1, qb0, qe0, qb1, qe1, flags, tiles = it
            assert (flags & 1) == (s == 0)
            if flags >> 8 != head:
                continue
            assert k1 - k0 <= 128 and (k1 > k0 or (pairs and n % 2 == 1))
            for k in range(k0, k1):
                for qb, qe in ((qb0, qe0), (qb1, qe1)):
                    for q in range(qb, qe):
                        if not causal or k <= q:
                            pairs_.append((q, k))
        cover[s] = pairs_
    return cover


def _expected(wl, causal):
    """{step: set of visible (q, k)} from the oracle's layout and ring rule."""
    want = {}
    for d in range(wl.num_docs):
        base, L, cp = wl.cu_seqlens[d], wl.doc_lengths[d], wl.cp_per_doc[d]
        for s in range(cp):
            for r in range(cp):
                j = R.ring_source(r, s, cp)
                qs = [base + x for a, b in R.shard_ranges(L, cp, wl.layout, r) for x in range(a, b)]
                ks = [base + x for a, b in R.shard_ranges(L, cp, wl.layout, j) for x in range(a, b)]
                want.setdefault(s, set()).update((q, k) for q in qs for k in ks if not causal or k <= q)
    return want


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lengths,cp", [([512], 4), ([700, 3, 1, 260], [4, 2, 1, 3]), ([130, 9], 8),
                                        ([600, 300], [1, 1])])
@pytest.mark.parametrize("head_dim", [64, 128])  # 128: with the CTA-pair backward
def test_work_items_cover_each_visible_pair_once(ra, layout, causal, lengths, cp, head_dim):
    wl = custom(lengths, 2, 2, head_dim, cp, layout, causal)
    paired = head_dim == 128
    plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), layout, causal, 2, 2, head_dim, bwd_cta_pairs=paired)
    want = _expected(wl, causal)
    expanders = [("fwd", _expand_fwd)] + [("bwd", lambda i, o, c, h=h: _expand_bwd(i, o, c, h, paired))
                                          for h in range(2)]
    for which, expand in expanders:
        items, off = plan.work_items(which)
        got = expand(items, off, causal)
        total = 0
        for s, pairs in got.items():
            assert len(pairs) == len(set(pairs)), (which, s)
            assert set(pairs) == want.get(s, set()), (which, s)
            total += len(pairs)
        assert total == plan.stats()["visible_pairs"]


def test_first_step_writes_every_row(ra):
    wl = custom([700, 3, 1, 260], 2, 2, 64, [4, 2, 1, 3], "zigzag")
    plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), "zigzag", True, 2, 2, 64)
    items, off = plan.work_items("fwd")
    rows = set()
    for it in items[off[0]:off[1]]:
        rows.update(range(it[0], it[1]))
    assert rows == set(range(wl.T))


def test_visible_pairs_of_workloads(ra):
    for name in ("tiny", "llama3_8b_32k", "varlen_65k"):
        wl = workload(name)
        plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), wl.layout, wl.causal, wl.Hq, wl.Hkv, wl.d)
        want = sum(L * (L + 1) // 2 for L in wl.doc_lengths)
        st = plan.stats()
        assert st["visible_pairs"] == want
        assert st["steps"] == max(wl.cp_per_doc)


def test_workspace_bytes_grow_with_outputs(ra):
    plan = ra.Plan([0, 4096], 4, "zigzag", True, 8, 2, 128)
    f_bf16, b_bf16 = plan.workspace_bytes(False, False)
    f_fp32, b_fp32 = plan.workspace_bytes(True, True)
    # the single-launch forward writes O once, in its final dtype
    assert f_bf16 == f_fp32 == plan.fused_workspace_bytes()
    # the ring-step forward merges into an fp32 running output when O is bf16
    assert plan.ring_step_workspace_bytes(False) - plan.ring_step_workspace_bytes(True) >= 4096 * 8 * 128 * 4
    assert b_bf16 - b_fp32 >= 4096 * (8 + 2 + 2) * 128 * 4


@pytest.mark.parametrize("kwargs,status", [
    (dict(cu=[0, 10], cp=0), 1),
    (dict(cu=[0, 10], cp=2, hq=3, hkv=2), 1),
    (dict(cu=[0, 10], cp=2, d=96), 2),
    (dict(cu=[1, 10], cp=2), 1),
    (dict(cu=[0, 10, 5], cp=2), 1),
    (dict(cu=[0, 0], cp=2), 1),
    (dict(cu=[0, 10], cp=2, layout=7), 1),
])
def test_plan_rejects_bad_arguments(ra, kwargs, status):
    with pytest.raises(ra.RingAttnError) as e:
        ra.Plan(kwargs["cu"], kwargs["cp"], kwargs.get("layout", "zigzag"), True, kwargs.get("hq", 2),
                kwargs.get("hkv", 1), kwargs.get("d", 64))
    assert e.value.status == status
    assert len(str(e.value)) > 20


def test_fwd_rejects_bad_pointers_before_touching_the_gpu(ra):
    lib = ra.load_library()
    plan = ra.Plan([0, 256], 2, "zigzag", True, 2, 1, 64)
    p = ctypes.c_void_p
    # NULL tensor
    st = lib.ra_fwd(plan.handle, p(0), p(16), p(32), p(48), 0, p(64), p(128), 1 << 30, p(0))
    assert st == 1
    # misaligned pointer
    st = lib.ra_fwd(plan.handle, p(8), p(16), p(32), p(48), 0, p(64), p(128), 1 << 30, p(0))
    assert st == 1
    # workspace too small
    st = lib.ra_fwd(plan.handle, p(16), p(32), p(48), p(64), 0, p(80), p(96), 16, p(0))
    assert st == 4
    assert b"workspace too small" in lib.ra_last_error()
    st = lib.ra_bwd(plan.handle, p(16), p(32), p(48), p(64), 0, p(80), p(96), p(112), p(128), p(144), 0,
                    p(160), 16, p(0))
    assert st == 4


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lengths,cp", [([512], 4), ([700, 3, 1, 260], [4, 2, 1, 3]), ([130, 9], 8), ([1000], 1)])
def test_fused_forward_tiles_cover_each_visible_pair_once(ra, layout, causal, lengths, cp):
    """The single-launch forward visits, per query chunk, every visible key once,
    shard by shard in ring order, and its active-tile counts match the mask."""
    wl = custom(lengths, 2, 2, 64, cp, layout, causal)
    plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), layout, causal, 2, 2, 64)
    items, tiles = plan.fused_items()
    want = set()
    for pairs in _expected(wl, causal).values():
        want |= pairs
    got = []
    rows = set()
    for q0, q1, t0, nt, na0, na1, flags, work in items:
        assert 0 < q1 - q0 <= 256 and nt == work and flags == 1
        rows.update(range(q0, q1))
        last = [min(q0 + 128, q1) - 1, q1 - 1]
        seen = [0, 0]
        for kst, kend in tiles[t0:t0 + nt]:
            assert kst < kend and kend - kst > 0
            for qt in range(2):
                if q0 + 128 * qt < q1 and (not causal or kst <= last[qt]):
                    seen[qt] += 1
            for q in range(q0, q1):
                for k in range(kst, min(kst + 128, kend)):
                    if not causal or k <= q:
                        got.append((q, k))
        assert seen == [na0, na1]
        # ring order: the shards the chunk meets come as (r - s) mod cp, s = 0, 1, ...
        d = max(i for i in range(wl.num_docs) if wl.cu_seqlens[i] <= q0)
        base, L, c = wl.cu_seqlens[d], wl.doc_lengths[d], wl.cp_per_doc[d]
        r = next(r for r in range(c) for a, b in R.shard_ranges(L, c, layout, r) if a <= q0 - base < b)
        order = []
        for kst, _ in tiles[t0:t0 + nt]:
            j = next(j for j in range(c) for a, b in R.shard_ranges(L, c, layout, j) if a <= kst - base < b)
            if not order or order[-1] != j:
                order.append(j)
        steps = [(r - j) % c for j in order]
        assert steps == sorted(steps) and len(set(steps)) == len(steps)
    assert len(got) == len(set(got))
    assert set(got) == want
    assert rows == set(range(wl.T))
    assert plan.fused_workspace_bytes() >= 256 + 32 * len(items) + 8 * len(tiles)


def test_python_api_has_no_cpu_path(ra):
    """The binding computes nothing itself: CPU tensors are refused (no silent
    fallback), for the forward, the backward and the autograd wrapper."""
    import torch
    T, H, D = 256, 2, 64
    q = torch.zeros((T, H, D), dtype=torch.bfloat16)
    lse = torch.zeros((H, T), dtype=torch.float32)
    args = ([0, T], 2, "zigzag", True)
    with pytest.raises(ValueError, match="CUDA"):
        ra.ring_attn_fwd(q, q, q, *args)
    with pytest.raises(ValueError, match="CUDA"):
        ra.ring_attn_bwd(q, q, q, q, q, lse, *args)
    with pytest.raises(ValueError, match="CUDA"):
        ra.ring_attention(q, q, q, *args)


def test_missing_library_fails_loudly(tmp_path):
    """A missing shared library is an error, not a fallback."""
    import context_ring_attention_step_gb300.ring_attn as m
    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(RuntimeError, match="not found"):
            m.load_library(str(tmp_path / "absent.so"))
    finally:
        m._lib = saved


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("lengths,cp", [([512], 4), ([700, 3, 1, 260], [4, 2, 1, 3]), ([1000], 1)])
def test_rank_work_lists_partition_each_step(ra, layout, lengths, cp):
    """The per-rank lists of a step hold exactly the step's items, and rank r's
    items are those of query shard r (forward: query rows in shard r;
    backward: key rows in shard (r - s) mod cp, queries in shard r)."""
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    plan = ra.Plan(cu, cp, layout, True, 4, 2, 64)
    cps = plan.cp_per_doc
    steps = plan.stats()["steps"]

    def shard_rows(r):
        rows = set()
        for d in range(len(lengths)):
            if r < cps[d]:
                for b, e in plan.shard_token_ranges(d, r):
                    rows.update(range(b, e))
        return rows

    for which in ("fwd", "bwd"):
        items, off = plan.work_items(which)
        per_rank = plan.rank_work_items(which)
        for s in range(steps):
            got = sorted(it for r in range(steps) for it in per_rank[(s, r)])
            assert got == sorted(items[off[s]:off[s + 1]])
            for r in range(steps):
                rows_r = shard_rows(r)
                for it in per_rank[(s, r)]:
                    if which == "fwd":
                        assert set(range(it[0], it[1])) <= rows_r
                    else:
                        qs = set(range(it[2], it[3])) | set(range(it[4], it[5]))
                        assert qs <= rows_r
                        d = next(i for i in range(len(lengths)) if cu[i] <= it[0] < cu[i + 1])
                        assert set(range(it[0], it[1])) <= shard_rows((r - s) % cps[d]) or cps[d] <= s


def test_bwd_cta_pairs_option(ra):
    """The CTA-pair backward: head_dim 128 only; switching it rebuilds the
    backward items (pairs of neighbouring key tiles) and back again."""
    wl = custom([700, 300], 4, 2, 128, [2, 1], "zigzag")
    plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), "zigzag", True, 4, 2, 128)
    single, off1 = plan.work_items("bwd")
    plan.set_bwd_cta_pairs(True)
    paired, off2 = plan.work_items("bwd")
    assert len(paired) % 2 == 0 and len(paired) >= len(single) and paired != single
    assert all(b[1] - b[0] <= 128 for b in paired)
    plan.set_bwd_cta_pairs(False)
    assert plan.work_items("bwd") == (single, off1)
    p64 = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), "zigzag", True, 4, 2, 64)
    with pytest.raises(ra.RingAttnError):
        p64.set_bwd_cta_pairs(True)


def test_kernel_source_hash_ignores_comments_only():
    """The recorded DRAM traffic is tied to the kernel's code: comments and
    blank lines do not change the hash, code does."""
    import bench
    a = "// header\nint f(int x) {  // add one\n  /* block\n     comment */ return x + 1;\n}\n"
    b = "int f(int x) {\n\n  return x + 1;   // other words\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    assert len(bench.kernel_source_hash("ring_bwd_step_kernel")) == 16
