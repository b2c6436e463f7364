"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped scale,
a wrong mask edge, a transposed operand, a wrong GQA head map, a missing
term in the backward) fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import ring as R

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _cu(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    return cu


# ---------------------------------------------------------------- brute force

def _brute_fwd(q, k, v, cu, causal, scale):
    """Pure-Python loops with math.fsum: the definition, element by element."""
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    o = [[[0.0] * v.shape[2] for _ in range(Hq)] for _ in range(T)]
    lse = [[0.0] * T for _ in range(Hq)]
    for doc in range(len(cu) - 1):
        b, e = cu[doc], cu[doc + 1]
        for h in range(Hq):
            g = h // G
            for i in range(b, e):
                keys = [j for j in range(b, e) if (not causal or j <= i)]
                s = [scale * math.fsum(q[i, h, t] * k[j, g, t] for t in range(d)) for j in keys]
                m = max(s)
                l = m + math.log(math.fsum(math.exp(x - m) for x in s))
                lse[h][i] = l
                for t in range(v.shape[2]):
                    o[i][h][t] = math.fsum(math.exp(s[n] - l) * v[keys[n], g, t]
                                           for n in range(len(keys)))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [True, False])
def test_fwd_matches_brute_force(causal):
    lengths = [5, 1, 13, 9]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 6
    q, k, v = _rand((T, Hq, d), 1), _rand((T, Hkv, d), 2), _rand((T, Hkv, d), 3)
    cu = _cu(lengths)
    scale = 0.37
    o, lse = A.attention_fwd(q, k, v, cu, causal=causal, scale=scale, row_block=4)
    bo, blse = _brute_fwd(q, k, v, cu, causal, scale)
    assert np.abs(o - bo).max() < 1e-12
    assert np.abs(lse - blse).max() < 1e-12


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [True, False])
def test_zero_queries_give_uniform_attention(causal):
    """q = 0: P is uniform over visible keys, LSE_i = ln(n_i), O_i = mean of visible v."""
    lengths = [7, 1, 3, 12]
    T, Hq, Hkv, d = sum(lengths), 2, 1, 5
    q = np.zeros((T, Hq, d))
    k, v = _rand((T, Hkv, d), 4), _rand((T, Hkv, d), 5)
    cu = _cu(lengths)
    o, lse = A.attention_fwd(q, k, v, cu, causal=causal, scale=0.5, row_block=3)
    for doc in range(len(lengths)):
        b, e = cu[doc], cu[doc + 1]
        for i in range(b, e):
            n = (i - b + 1) if causal else (e - b)
            last = i + 1 if causal else e
            for h in range(Hq):
                assert abs(lse[h, i] - math.log(n)) < 1e-13
                assert np.abs(o[i, h] - v[b:last, 0].mean(axis=0)).max() < 1e-13


def test_first_row_of_each_doc_copies_its_value():
    lengths = [4, 6, 2]
    T, Hq, Hkv, d = sum(lengths), 2, 2, 3
    q, k, v = _rand((T, Hq, d), 6), _rand((T, Hkv, d), 7), _rand((T, Hkv, d), 8)
    cu = _cu(lengths)
    o, lse = A.attention_fwd(q, k, v, cu, causal=True, scale=1.0)
    for doc in range(len(lengths)):
        b = cu[doc]
        for h in range(Hq):
            assert np.array_equal(o[b, h], v[b, h])
            assert abs(lse[h, b] - q[b, h] @ k[b, h]) < 1e-14


@pytest.mark.parametrize("causal", [True, False])
def test_one_hot_values_expose_probabilities(causal):
    """v_j = e_j makes O_i the probability row: non-negative, sums to 1, zero where masked."""
    lengths = [6, 10]
    T, d = sum(lengths), 16
    q, k = _rand((T, 1, d), 9), _rand((T, 1, d), 10)
    v = np.eye(T)[:, None, :]
    cu = _cu(lengths)
    o, lse = A.attention_fwd(q, k, v, cu, causal=causal, scale=0.3, row_block=5)
    p = o[:, 0, :]
    assert np.abs(p.sum(axis=1) - 1.0).max() < 1e-12
    assert p.min() >= 0.0
    for doc in range(len(lengths)):
        b, e = cu[doc], cu[doc + 1]
        for i in range(b, e):
            for j in range(T):
                visible = b <= j < e and (not causal or j <= i)
                if not visible:
                    assert p[i, j] == 0.0
                else:
                    s = 0.3 * q[i, 0] @ k[j, 0]
                    assert abs(math.log(p[i, j]) - (s - lse[0, i])) < 1e-12


def test_key_shift_invariance():
    """k_j + c for all j: O unchanged, LSE_i shifted by scale <q_i, c>, dv unchanged."""
    lengths = [9, 4]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 5
    q, k, v, do = (_rand((T, Hq, d), 11), _rand((T, Hkv, d), 12),
                   _rand((T, Hkv, d), 13), _rand((T, Hq, d), 14))
    c = _rand((d,), 15)
    cu = _cu(lengths)
    o1, l1 = A.attention_fwd(q, k, v, cu, scale=0.7)
    o2, l2 = A.attention_fwd(q, k + c, v, cu, scale=0.7)
    assert np.abs(o1 - o2).max() < 1e-12
    G = Hq // Hkv
    for h in range(Hq):
        assert np.abs(l2[h] - l1[h] - 0.7 * q[:, h] @ c).max() < 1e-12
    g1 = A.attention_bwd(q, k, v, do, cu, scale=0.7)
    g2 = A.attention_bwd(q, k + c, v, do, cu, scale=0.7)
    assert np.abs(g1[2] - g2[2]).max() < 1e-12
    assert G == 2


def test_gqa_head_map_is_contiguous_groups():
    """Query head h reads kv head h // G: equals MHA with the kv heads repeated."""
    T, Hq, Hkv, d = 11, 6, 2, 4
    q, k, v = _rand((T, Hq, d), 16), _rand((T, Hkv, d), 17), _rand((T, Hkv, d), 18)
    cu = [0, 5, 11]
    o, lse = A.attention_fwd(q, k, v, cu, scale=0.4)
    krep = np.repeat(k, Hq // Hkv, axis=1)
    vrep = np.repeat(v, Hq // Hkv, axis=1)
    o2, lse2 = A.attention_fwd(q, krep, vrep, cu, scale=0.4)
    assert np.abs(o - o2).max() < 1e-14 and np.abs(lse - lse2).max() < 1e-14


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal", [True, False])
def test_single_doc_matches_torch_sdpa_and_autograd(causal):
    T, Hq, d = 37, 3, 8
    q, k, v, do = (_rand((T, Hq, d), 19), _rand((T, Hq, d), 20),
                   _rand((T, Hq, d), 21), _rand((T, Hq, d), 22))
    scale = 0.45
    o, lse = A.attention_fwd(q, k, v, [0, T], causal=causal, scale=scale, row_block=8)
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    assert np.abs(o - to.detach().numpy().transpose(1, 0, 2)).max() < 1e-12
    to.backward(torch.tensor(do.transpose(1, 0, 2)))
    dq, dk, dv, _, _ = A.attention_bwd(q, k, v, do, [0, T], causal=causal, scale=scale, row_block=8)
    assert np.abs(dq - tq.grad.numpy().transpose(1, 0, 2)).max() < 1e-11
    assert np.abs(dk - tk.grad.numpy().transpose(1, 0, 2)).max() < 1e-11
    assert np.abs(dv - tv.grad.numpy().transpose(1, 0, 2)).max() < 1e-11


# ---------------------------------------------------------------- backward

def test_backward_central_finite_differences():
    lengths = [5, 7]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 3
    rng = np.random.default_rng(23)
    q, k, v, do = (rng.standard_normal(s) for s in
                   ((T, Hq, d), (T, Hkv, d), (T, Hkv, d), (T, Hq, d)))
    cu = _cu(lengths)
    scale = 0.6
    dq, dk, dv, _, _ = A.attention_bwd(q, k, v, do, cu, scale=scale, row_block=4)

    def f(q_, k_, v_):
        o, _ = A.attention_fwd(q_, k_, v_, cu, scale=scale, row_block=4)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        idx = [tuple(rng.integers(0, s) for s in x.shape) for _ in range(12)]
        for ix in idx:
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            assert abs(fd - g[ix]) <= 1e-6 * max(1.0, abs(g[ix])), (name, ix, fd, g[ix])


def test_gradient_sum_identities():
    """sum_j dv_j = sum over group heads of sum_i dO_i;  sum_j dk_j = 0 (per document)."""
    lengths = [8, 3, 6]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 5
    q, k, v, do = (_rand((T, Hq, d), 24), _rand((T, Hkv, d), 25),
                   _rand((T, Hkv, d), 26), _rand((T, Hq, d), 27))
    cu = _cu(lengths)
    dq, dk, dv, _, _ = A.attention_bwd(q, k, v, do, cu, scale=0.8)
    G = Hq // Hkv
    for doc in range(len(lengths)):
        b, e = cu[doc], cu[doc + 1]
        for g in range(Hkv):
            want = do[b:e, g * G:(g + 1) * G].sum(axis=(0, 1))
            assert np.abs(dv[b:e, g].sum(axis=0) - want).max() < 1e-12
            assert np.abs(dk[b:e, g].sum(axis=0)).max() < 1e-12


# ---------------------------------------------------------------- layouts

def _read_golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = line.split(":", 1)
        rows[key.strip()] = [tuple(int(x) for x in rng.split("-")) for rng in val.split()]
    return rows


def test_zigzag_layout_golden():
    gold = _read_golden("zigzag_L512_cp4.txt")
    for r in range(4):
        assert R.shard_ranges(512, 4, "zigzag", r) == gold["shard%d" % r]


def test_uneven_layout_golden():
    gold = _read_golden("layouts_L10_cp3.txt")
    for r in range(3):
        assert R.shard_ranges(10, 3, "zigzag", r) == gold["zigzag%d" % r]
        assert R.shard_ranges(10, 3, "contiguous", r) == gold["contiguous%d" % r]


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("L,cp", [(512, 4), (37, 5), (3, 4), (1, 8), (100, 8)])
def test_shards_partition_the_document(layout, L, cp):
    seen = []
    for r in range(cp):
        for a, b in R.shard_ranges(L, cp, layout, r):
            assert 0 <= a <= b <= L
            seen.extend(range(a, b))
    assert sorted(seen) == list(range(L))


def test_ring_visits_every_shard_once():
    for cp in range(1, 9):
        for r in range(cp):
            assert sorted(R.ring_source(r, s, cp) for s in range(cp)) == list(range(cp))
            assert R.ring_source(r, 0, cp) == r


def test_attention_matrix_memory_figure():
    """Accelerate guide, "Por que paralelismo de contexto?": 128k x 128k x 2 B is ~32 GB per head."""
    assert 131072 * 131072 * 2 == 32 * 2 ** 30


# ---------------------------------------------------------------- ring == monolithic

@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_equals_monolithic_all_cp(layout, causal):
    lengths = [29, 1, 6, 17]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 4
    q, k, v, do = (_rand((T, Hq, d), 30), _rand((T, Hkv, d), 31),
                   _rand((T, Hkv, d), 32), _rand((T, Hq, d), 33))
    cu = _cu(lengths)
    dq0, dk0, dv0, o0, l0 = A.attention_bwd(q, k, v, do, cu, causal=causal, scale=0.55)
    for cp in range(1, 9):
        cps = [cp, min(cp, 3), cp, max(1, cp - 2)]
        o, lse = R.ring_attention_fwd(q, k, v, cu, cps, layout, causal=causal, scale=0.55)
        assert np.abs(o - o0).max() < 1e-12, cp
        assert np.abs(lse - l0).max() < 1e-12, cp
        dq, dk, dv = R.ring_attention_bwd(q, k, v, do, o, lse, cu, cps, layout,
                                          causal=causal, scale=0.55)
        assert np.abs(dq - dq0).max() < 1e-12
        assert np.abs(dk - dk0).max() < 1e-12
        assert np.abs(dv - dv0).max() < 1e-12


def test_merge_handles_empty_sides():
    oa, la = np.ones((3, 2)), np.array([-np.inf, 0.5, -np.inf])
    ob, lb = 2 * np.ones((3, 2)), np.array([1.0, -np.inf, -np.inf])
    o, lse = R.merge(oa, la, ob, lb)
    assert lse[0] == 1.0 and np.all(o[0] == 2.0)
    assert lse[1] == 0.5 and np.all(o[1] == 1.0)
    assert np.isneginf(lse[2])


def test_rows_sampler_matches_full_oracle():
    lengths = [40, 25]
    T, Hq, Hkv, d = sum(lengths), 4, 1, 8
    q, k, v = _rand((T, Hq, d), 34), _rand((T, Hkv, d), 35), _rand((T, Hkv, d), 36)
    cu = _cu(lengths)
    o, lse = A.attention_fwd(q, k, v, cu, scale=0.3)
    rows = [0, 1, 39, 40, 41, 64]
    for h in range(Hq):
        ro, rl = A.attention_rows(q, k, v, cu, rows, h, scale=0.3)
        assert np.abs(ro - o[rows, h]).max() < 1e-13
        assert np.abs(rl - lse[h, rows]).max() < 1e-13


def test_rows_dq_matches_full_oracle():
    lengths = [33, 20]
    T, Hq, Hkv, d = sum(lengths), 4, 2, 8
    q, k, v, do = (_rand((T, Hq, d), 37), _rand((T, Hkv, d), 38),
                   _rand((T, Hkv, d), 39), _rand((T, Hq, d), 40))
    cu = _cu(lengths)
    for causal in (True, False):
        dq, _, _, _, _ = A.attention_bwd(q, k, v, do, cu, causal=causal, scale=0.3)
        rows = [0, 5, 32, 33, 52]
        for h in range(Hq):
            rdq = A.attention_rows_dq(q, k, v, do, cu, rows, h, causal=causal, scale=0.3)
            assert np.abs(rdq - dq[rows, h]).max() < 1e-12


# ---------------------------------------------------------------- planted mistakes

def test_pins_catch_a_planted_mask_slip(monkeypatch):
    """An off-by-one causal edge planted in the oracle must fail the closed form."""
    orig = A._block_scores

    def slipped(q, k, h, g, r0, r1, b, e, causal, scale):
        s, kend = orig(q, k, h, g, r0, r1, b, e, False, scale)
        if causal:
            qpos = np.arange(r0, r1)[:, None]
            kpos = np.arange(b, kend)[None, :]
            s = np.where(kpos < qpos, s, -np.inf)   # drops the diagonal
        return s, kend

    monkeypatch.setattr(A, "_block_scores", slipped)
    with pytest.raises(AssertionError):
        test_zero_queries_give_uniform_attention(True)


def test_pins_catch_a_planted_backward_slip(monkeypatch):
    """Halving dv in the oracle must fail the finite-difference pin."""
    orig_bwd = A.attention_bwd

    def slipped(q, k, v, do, cu, causal=True, scale=None, heads=None, row_block=256):
        dq, dk, dv, o, lse = orig_bwd(q, k, v, do, cu, causal, scale, heads, row_block)
        return dq * 1.0, dk, dv * 0.5, o, lse

    monkeypatch.setattr(A, "attention_bwd", slipped)
    with pytest.raises(AssertionError):
        test_backward_central_finite_differences()


# ---------------------------------------------------------------- gradients of chosen key rows

def _torch_masked_grads(q, k, v, do, cu, causal, scale):
    """dk, dv through torch float64 autograd of an explicitly masked softmax
    attention (a mask matrix built from cu_seqlens, GQA by repeating heads)."""
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    tq = torch.tensor(q)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    doc = torch.zeros(T, dtype=torch.long)
    for n in range(len(cu) - 1):
        doc[cu[n]:cu[n + 1]] = n
    pos = torch.arange(T)
    vis = doc[:, None] == doc[None, :]
    if causal:
        vis &= pos[None, :] <= pos[:, None]
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    s = scale * torch.einsum("ihd,jhd->hij", tq, kk)
    s = s.masked_fill(~vis[None], float("-inf"))
    o = torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), vv)
    (o * torch.tensor(do)).sum().backward()
    return tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_keys_dkdv_matches_torch_autograd(causal):
    lengths = [37, 1, 300, 22]
    T, Hq, Hkv, d = sum(lengths), 6, 2, 8
    q, k, v, do = (_rand((T, Hq, d), 61), _rand((T, Hkv, d), 62),
                   _rand((T, Hkv, d), 63), _rand((T, Hq, d), 64))
    cu = _cu(lengths)
    rk, rv = _torch_masked_grads(q, k, v, do, cu, causal, 0.4)
    keys = [0, 5, 36, 37, 38, 100, 290, 337, 338, 359]
    for g in range(Hkv):
        dk, dv = A.attention_keys_dkdv(q, k, v, do, cu, keys, g, causal=causal, scale=0.4)
        assert np.abs(dk - rk[keys, g]).max() < 1e-12
        assert np.abs(dv - rv[keys, g]).max() < 1e-12


def test_keys_dkdv_matches_full_oracle():
    lengths = [600, 45]
    T, Hq, Hkv, d = sum(lengths), 4, 1, 16
    q, k, v, do = (_rand((T, Hq, d), 65), _rand((T, Hkv, d), 66),
                   _rand((T, Hkv, d), 67), _rand((T, Hq, d), 68))
    cu = _cu(lengths)
    _, rk, rv, _, _ = A.attention_bwd(q, k, v, do, cu, scale=0.25)
    keys = list(range(440, 600)) + [600, 644]
    dk, dv = A.attention_keys_dkdv(q, k, v, do, cu, keys, 0, scale=0.25)
    assert np.abs(dk - rk[keys, 0]).max() < 1e-12
    assert np.abs(dv - rv[keys, 0]).max() < 1e-12


def test_pins_catch_a_planted_keys_slip(monkeypatch):
    """An LSE off by a constant (P rows no longer summing to 1) must fail the autograd pin."""
    orig = A._softmax_lse

    def slipped(s):
        lse, p = orig(s)
        return lse + 1e-3, p   # an LSE off by a constant: P no longer sums to 1

    monkeypatch.setattr(A, "_softmax_lse", slipped)
    with pytest.raises(AssertionError):
        test_keys_dkdv_matches_torch_autograd(True)
