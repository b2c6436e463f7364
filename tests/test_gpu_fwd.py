"""GPU parity of the ring-attention forward against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation): max |O - O_ref| <= 2e-2 for the
fp32 output and 2e-2 + 2^-9 |O_ref| for the bf16 output (which adds its own
round-to-nearest of at most half a bf16 ulp), max |LSE - LSE_ref| <= 1e-3, and
the ring result on the GPU equals the GPU's own cp_size = 1 result within 1e-3
when the output is fp32.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import custom, draw_qkvdo, workload

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, RING_TOL = 2e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


def _run_fwd(ra, wl, q, k, v, o_fp32=False, cp=None, layout=None, fused=False):
    cps = list(wl.cp_per_doc) if cp is None else cp
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, layout or wl.layout, wl.causal,
                              wl.softmax_scale, o_fp32=o_fp32, check=True, fused=fused)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check_vs_oracle(ra, wl, fused=False):
    q, k, v, _ = draw_qkvdo(wl)
    o_ref, lse_ref = A.attention_fwd(q, k, v, wl.cu_seqlens, wl.causal, wl.softmax_scale)
    for fp32 in (True, False):
        o, lse = _run_fwd(ra, wl, q, k, v, o_fp32=fp32, fused=fused)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        bound = O_TOL if fp32 else O_TOL + np.abs(o_ref) * 2.0 ** -9
        assert (np.abs(o - o_ref) - bound).max() <= 0, (wl.name, fp32, np.abs(o - o_ref).max())
        err_l = np.abs(lse - lse_ref).max()
        assert err_l <= LSE_TOL, (wl.name, err_l)
    return q, k, v


def test_tiny_workload_matches_oracle(ra):
    _check_vs_oracle(ra, workload("tiny"))


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_multi_tile_ragged_gqa(ra, layout, causal):
    # 1500 tokens over cp 3: zigzag chunks of 250 (ragged vs the 128-row tiles)
    wl = custom([1500], 4, 2, 128, 3, layout, causal, seed=11, name="ragged_gqa")
    _check_vs_oracle(ra, wl)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_varlen_docs_per_doc_cp(ra, d):
    wl = custom([300, 1, 5, 777, 129, 64], 4, 1, d, [3, 1, 2, 5, 8, 1], "zigzag", True, seed=12, name="varlen")
    _check_vs_oracle(ra, wl)


# ---- head_dim 256: one 128-row query tile per CTA, S double-buffered

@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_256_ragged_gqa(ra, fused, layout, causal):
    wl = custom([1500, 77], 4, 2, 256, [3, 2], layout, causal, seed=15, name="d256")
    _check_vs_oracle(ra, wl, fused=fused)


def test_head_dim_256_ring_equals_cp1_fp32(ra):
    wl = custom([2048, 700], 4, 2, 256, 4, "zigzag", True, seed=16, name="d256_ring_vs_cp1")
    q, k, v, _ = draw_qkvdo(wl)
    o1, l1 = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=[1, 1])
    for layout in ("zigzag", "contiguous"):
        for cp in ([4, 4], [8, 3]):
            for fused in (False, True):
                o, l = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=cp, layout=layout, fused=fused)
                assert np.abs(o - o1).max() <= RING_TOL, (layout, cp, fused, np.abs(o - o1).max())
                assert np.abs(l - l1).max() <= RING_TOL


def test_ring_equals_gpu_cp1_fp32(ra):
    wl = custom([2048, 700], 8, 2, 128, 4, "zigzag", True, seed=13, name="ring_vs_cp1")
    q, k, v, _ = draw_qkvdo(wl)
    o1, l1 = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=[1, 1])
    for layout in ("zigzag", "contiguous"):
        for cp in ([4, 4], [8, 3], [2, 7]):
            o, l = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=cp, layout=layout)
            assert np.abs(o - o1).max() <= RING_TOL, (layout, cp, np.abs(o - o1).max())
            assert np.abs(l - l1).max() <= RING_TOL


def test_zero_queries_give_uniform_average(ra):
    """q = 0 on the GPU: LSE = ln(#visible keys), O = running mean of v."""
    wl = custom([640, 200], 2, 2, 64, 4, "zigzag", True, seed=14, name="zero_q")
    _, k, v, _ = draw_qkvdo(wl)
    q = torch.zeros((wl.T, 2, 64), dtype=torch.bfloat16)
    o, lse = _run_fwd(ra, wl, q, k, v, o_fp32=True)
    vf = v.float().numpy()
    for d, (b, e) in enumerate(zip(wl.cu_seqlens[:-1], wl.cu_seqlens[1:])):
        n = np.arange(1, e - b + 1)
        assert np.abs(lse[:, b:e] - np.log(n)[None, :]).max() < 1e-4
        mean = np.cumsum(vf[b:e], axis=0) / n[:, None, None]
        assert np.abs(o[b:e] - mean).max() < 1e-2


def test_llama_32k_sampled_rows(ra):
    """Full-size 32K workload in the bench's launch configuration, checked on sampled rows."""
    wl = workload("llama3_8b_32k")
    q, k, v, _ = draw_qkvdo(wl)
    o, lse = _run_fwd(ra, wl, q, k, v, o_fp32=True)
    rng = np.random.default_rng(0)
    for h in (0, 5, 31):
        rows = sorted(set(rng.integers(0, wl.T, 48).tolist()) | {0, 1, 2047, 2048, wl.T - 1})
        ro, rl = A.attention_rows(q, k, v, wl.cu_seqlens, rows, h, True, wl.softmax_scale)
        assert np.abs(o[rows, h] - ro).max() <= O_TOL
        assert np.abs(lse[h, rows] - rl).max() <= LSE_TOL


# ---- the whole ring in one launch (ra_fwd_fused)

@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_fused_multi_tile_ragged_gqa(ra, layout, causal):
    wl = custom([1500], 4, 2, 128, 3, layout, causal, seed=11, name="ragged_gqa")
    _check_vs_oracle(ra, wl, fused=True)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fused_varlen_docs_per_doc_cp(ra, d):
    wl = custom([300, 1, 5, 777, 129, 64], 4, 1, d, [3, 1, 2, 5, 8, 1], "zigzag", True, seed=12, name="varlen")
    _check_vs_oracle(ra, wl, fused=True)


def test_fused_tiny_matches_oracle(ra):
    _check_vs_oracle(ra, workload("tiny"), fused=True)


def test_fused_equals_ring_steps_fp32(ra):
    """One launch over the ring and one launch per ring step agree within 1e-3 (fp32 outputs)."""
    wl = custom([2048, 700], 8, 2, 128, 4, "zigzag", True, seed=13, name="fused_vs_steps")
    q, k, v, _ = draw_qkvdo(wl)
    for layout in ("zigzag", "contiguous"):
        for cp in ([4, 4], [8, 3]):
            o1, l1 = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=cp, layout=layout)
            o2, l2 = _run_fwd(ra, wl, q, k, v, o_fp32=True, cp=cp, layout=layout, fused=True)
            assert np.abs(o1 - o2).max() <= RING_TOL, (layout, cp, np.abs(o1 - o2).max())
            assert np.abs(l1 - l2).max() <= RING_TOL


def test_fused_llama_32k_sampled_rows(ra):
    wl = workload("llama3_8b_32k")
    q, k, v, _ = draw_qkvdo(wl)
    o, lse = _run_fwd(ra, wl, q, k, v, o_fp32=False, fused=True)
    rng = np.random.default_rng(1)
    for h in (0, 7, 30):
        rows = sorted(set(rng.integers(0, wl.T, 48).tolist()) | {0, 1, 2047, 2048, wl.T - 1})
        ro, rl = A.attention_rows(q, k, v, wl.cu_seqlens, rows, h, True, wl.softmax_scale)
        assert (np.abs(o[rows, h] - ro) - (O_TOL + np.abs(ro) * 2.0 ** -9)).max() <= 0
        assert np.abs(lse[h, rows] - rl).max() <= LSE_TOL


def test_caller_owned_outputs(ra):
    """out= writes the same values into caller tensors (forward and backward),
    and a mis-shaped or mis-typed output is refused before any launch."""
    wl = custom([700, 300], 4, 2, 128, 2, "zigzag", True, seed=31, name="out_param")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    cps = list(wl.cp_per_doc)
    args = (wl.cu_seqlens, cps, wl.layout, wl.causal, wl.softmax_scale)
    o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, *args)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    r = ra.ring_attn_fwd(q, k, v, *args, out=(o, lse))
    assert r[0] is o and r[1] is lse
    g_ref = ra.ring_attn_bwd(q, k, v, o_ref, do, lse_ref, *args)
    g = tuple(torch.full_like(x, float("nan")) for x in g_ref)
    r = ra.ring_attn_bwd(q, k, v, o, do, lse, *args, out=g)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)  # the forward has no atomics
    for a, b in zip(g, g_ref):  # dQ is summed with atomic adds: equal up to bf16 rounding
        assert torch.allclose(a.float(), b.float(), rtol=2 ** -7, atol=1e-5)
    with pytest.raises(ValueError):
        ra.ring_attn_fwd(q, k, v, *args, out=(o.float(), lse))
    with pytest.raises(ValueError):
        ra.ring_attn_bwd(q, k, v, o, do, lse, *args, out=(g[0], g[1], g[2][:-1]))


def test_autograd_wrapper_matches_explicit_calls(ra):
    """ring_attention under autograd gives the forward's (o, lse) and, from
    o.backward(dO), the explicit backward's dq, dk, dv."""
    wl = custom([640, 200], 4, 2, 128, 2, "zigzag", True, seed=33, name="autograd")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    cps = list(wl.cp_per_doc)
    args = (wl.cu_seqlens, cps, wl.layout, wl.causal, wl.softmax_scale)
    o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, *args)
    g_ref = ra.ring_attn_bwd(q, k, v, o_ref, do, lse_ref, *args)
    qa, ka, va = (x.clone().requires_grad_(True) for x in (q, k, v))
    o, lse = ra.ring_attention(qa, ka, va, *args)
    o.backward(do)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o_ref) and torch.equal(lse, lse_ref)
    for a, b in zip((qa.grad, ka.grad, va.grad), g_ref):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert torch.allclose(a.float(), b.float(), rtol=2 ** -7, atol=1e-5)


def test_work_list_copy_fallback_matches(ra, monkeypatch):
    """A plan built without pinned work lists (the calls then copy them with
    cudaMemcpyAsync) gives the same forward and backward as the default plan,
    whose calls set up the workspace with a kernel."""
    wl = custom([900, 333], 4, 2, 128, 3, "zigzag", True, seed=35, name="ws_setup")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    cps = list(wl.cp_per_doc)
    args = (wl.cu_seqlens, cps, wl.layout, wl.causal, wl.softmax_scale)
    mk = lambda: ra.Plan(wl.cu_seqlens, cps, wl.layout, wl.causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale)
    staged = mk()
    monkeypatch.setenv("RA_NO_PINNED_WORK_LISTS", "1")
    copied = mk()
    monkeypatch.delenv("RA_NO_PINNED_WORK_LISTS")
    outs = []
    for plan in (staged, copied):
        o, lse = ra.ring_attn_fwd(q, k, v, *args, o_fp32=True, plan=plan, check=True)
        o_f, lse_f = ra.ring_attn_fwd(q, k, v, *args, plan=plan, check=True, fused=True)
        g = ra.ring_attn_bwd(q, k, v, o, do, lse, *args, grads_fp32=True, plan=plan, check=True)
        outs.append((o, lse, o_f, lse_f) + tuple(g))
    torch.cuda.synchronize()
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert torch.equal(a, b)  # the forward has no atomics
    for a, b in zip(outs[0][4:], outs[1][4:]):
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-5)  # dQ is summed with atomic adds
