"""GPU parity of the ring-attention backward against the fp64 oracle.

Tolerance: bf16 inputs, fp32 accumulation: max |dX - dX_ref| <= 2e-2 for dQ,
dK, dV read from the fp32 accumulators (grads_fp32).  The bf16 gradients add
their own round-to-nearest of at most half a bf16 ulp (2^-9 |x|), so they are
held to 2e-2 + 2^-9 |dX_ref|.  The ring result on the GPU equals the GPU's own
cp_size = 1 result within 1e-3 with fp32 gradients.  The backward is fed the GPU forward's own O and LSE
(Delta = rowsum(dO * O) from the returned O).
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import custom, draw_qkvdo, workload

pytestmark = pytest.mark.gpu

G_TOL, RING_TOL = 2e-2, 1e-3


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


def _run(ra, wl, q, k, v, do, grads_fp32=False, cp=None, layout=None, o_fp32=False, pairs=False):
    cps = list(wl.cp_per_doc) if cp is None else cp
    lay = layout or wl.layout
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    plan = ra.Plan(wl.cu_seqlens, cps, lay, wl.causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale, bwd_cta_pairs=pairs)
    o, lse = ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, lay, wl.causal, wl.softmax_scale,
                              o_fp32=o_fp32, plan=plan, check=True)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, o, dod, lse, wl.cu_seqlens, cps, lay, wl.causal,
                                  wl.softmax_scale, grads_fp32=grads_fp32, plan=plan, check=True)
    torch.cuda.synchronize()
    return tuple(x.float().cpu().numpy() for x in (dq, dk, dv))


def _check_vs_oracle(ra, wl, pairs=False):
    q, k, v, do = draw_qkvdo(wl)
    rq, rk, rv, _, _ = A.attention_bwd(q, k, v, do, wl.cu_seqlens, wl.causal, wl.softmax_scale)
    for fp32 in (True, False):
        grads = _run(ra, wl, q, k, v, do, grads_fp32=fp32, pairs=pairs)
        for name, x, ref in zip(("dq", "dk", "dv"), grads, (rq, rk, rv)):
            assert np.isfinite(x).all(), name
            bound = G_TOL if fp32 else G_TOL + np.abs(ref) * 2.0 ** -9
            excess = (np.abs(x - ref) - bound).max()
            assert excess <= 0, (wl.name, name, fp32, np.abs(x - ref).max())


def test_tiny_workload_matches_oracle(ra):
    _check_vs_oracle(ra, workload("tiny"))


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_multi_tile_ragged_gqa(ra, layout, causal):
    wl = custom([1500], 4, 2, 128, 3, layout, causal, seed=21, name="ragged_gqa")
    _check_vs_oracle(ra, wl)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_varlen_docs_per_doc_cp(ra, d):
    wl = custom([300, 1, 5, 777, 129, 64], 4, 1, d, [3, 1, 2, 5, 8, 1], "zigzag", True, seed=22, name="varlen")
    _check_vs_oracle(ra, wl)


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_cta_pair_backward_ragged_gqa(ra, layout, causal):
    """The CTA-pair backward (head_dim 128): key tiles in pairs, one of them
    ragged or empty at every range end, GQA, multi-document."""
    wl = custom([1500, 77, 300], 4, 2, 128, [3, 1, 2], layout, causal, seed=26, name="pairs_bwd")
    _check_vs_oracle(ra, wl, pairs=True)


def test_cta_pair_backward_tiny_documents(ra):
    """CTA pairs where most ranges hold one key tile or less (the second
    tile of the pair empty), no GQA grouping (Hq = Hkv)."""
    wl = custom([1, 5, 130, 129, 257, 3, 64], 2, 2, 128, [1, 1, 2, 1, 3, 1, 2], "zigzag", True, seed=28,
                name="pairs_tiny_docs")
    _check_vs_oracle(ra, wl, pairs=True)


def test_cta_pair_backward_equals_single_cta(ra):
    """Same gradients from the CTA-pair backward as from the one-CTA kernel,
    within fp32 accumulation-order differences (fp32 gradients)."""
    wl = custom([2500], 8, 2, 128, 4, "zigzag", True, seed=27, name="pairs_vs_single")
    q, k, v, do = draw_qkvdo(wl)
    one = _run(ra, wl, q, k, v, do, grads_fp32=True)
    two = _run(ra, wl, q, k, v, do, grads_fp32=True, pairs=True)
    for name, a, b in zip(("dq", "dk", "dv"), one, two):
        assert np.abs(a - b).max() <= RING_TOL, (name, np.abs(a - b).max())


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_256_ragged_gqa(ra, layout, causal):
    """head_dim 256: two CTAs per key tile (column halves), 64-row query tiles."""
    wl = custom([1500, 77], 4, 2, 256, [3, 2], layout, causal, seed=25, name="d256_bwd")
    _check_vs_oracle(ra, wl)


def test_ring_equals_gpu_cp1_fp32(ra):
    """Backward ring invariance: from the same saved (O, LSE), every ring layout equals cp_size = 1.

    The forward of each layout reaches O and LSE equal only up to fp32 rounding
    (its own invariance is tested in test_gpu_fwd); feeding the backward those
    last-bit differences flips ties in the bf16 rounding of P and dS.  So the
    layouts are compared on one shared (O, LSE), with fp32 gradients, at 1e-3.
    """
    wl = custom([2048, 700], 8, 2, 128, 4, "zigzag", True, seed=23, name="ring_vs_cp1")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    plan1 = ra.Plan(wl.cu_seqlens, [1, 1], "zigzag", True, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale)
    o, lse = ra.ring_attn_fwd(q, k, v, wl.cu_seqlens, [1, 1], "zigzag", True, wl.softmax_scale, o_fp32=True,
                              plan=plan1, check=True)
    g1 = ra.ring_attn_bwd(q, k, v, o, do, lse, wl.cu_seqlens, [1, 1], "zigzag", True, wl.softmax_scale,
                          grads_fp32=True, plan=plan1, check=True)
    g1 = [x.cpu().numpy() for x in g1]
    for layout in ("zigzag", "contiguous"):
        for cp in ([4, 4], [8, 3], [2, 7]):
            plan = ra.Plan(wl.cu_seqlens, cp, layout, True, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale)
            g = ra.ring_attn_bwd(q, k, v, o, do, lse, wl.cu_seqlens, cp, layout, True, wl.softmax_scale,
                                 grads_fp32=True, plan=plan, check=True)
            for name, x, ref in zip(("dq", "dk", "dv"), g, g1):
                err = np.abs(x.cpu().numpy() - ref).max()
                assert err <= RING_TOL, (layout, cp, name, err)


def test_llama_32k_sampled_rows_and_sum_identities(ra):
    """Full-size 32K workload: dq on sampled rows, dk/dv through identities that hold at any size."""
    wl = workload("llama3_8b_32k")
    q, k, v, do = draw_qkvdo(wl)
    dq, dk, dv = _run(ra, wl, q, k, v, do, grads_fp32=True)
    rng = np.random.default_rng(1)
    for h in (0, 13, 31):
        rows = sorted(set(rng.integers(0, wl.T, 24).tolist()) | {0, 1, 2047, 2048, wl.T - 1})
        ref = A.attention_rows_dq(q, k, v, do, wl.cu_seqlens, rows, h, True, wl.softmax_scale)
        assert np.abs(dq[rows, h] - ref).max() <= G_TOL
    # sum_j dv_j = sum over the group's query heads of sum_i dO_i ; sum_j dk_j = 0
    G = wl.Hq // wl.Hkv
    dof = do.float().numpy().astype(np.float64)
    for g in range(wl.Hkv):
        want = dof[:, g * G:(g + 1) * G].sum(axis=(0, 1))
        e_dv = np.abs(dv[:, g].astype(np.float64).sum(axis=0) - want).max()
        e_dk = np.abs(dk[:, g].astype(np.float64).sum(axis=0)).max()
        print("sum identities g=%d: dv %.4g dk %.4g" % (g, e_dv, e_dk))
        assert e_dv <= 2.0
        assert e_dk <= 2.0
