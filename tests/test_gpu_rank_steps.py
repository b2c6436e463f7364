"""The per-rank ring-step calls on the GPU, with the ring's exchange emulated.

Every rank gets its own full-length buffers, zero except for its own shard's
rows.  The test runs the multi-GPU schedule (ring_driver's order) rank after
rank on the one GPU, and moves the key/value shards and the travelling dK/dV
partials between the ranks' buffers with plain copies where the driver would
send and receive.  No kernel waits on another: each launch completes on its
own.  Each rank's own rows must equal the all-ranks result: bit for bit for
the forward (the same work items in the same order per row), within 1e-5 for
the gradients (summed in another order), and the oracle within the usual
tolerances.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import custom, draw_qkvdo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


def _rows(ranges):
    idx = [torch.arange(b, e) for b, e in ranges]
    return torch.cat(idx).cuda() if idx else torch.zeros(0, dtype=torch.long, device="cuda")


@pytest.mark.parametrize("layout,causal,pairs", [("zigzag", True, False), ("contiguous", True, False),
                                                ("zigzag", False, False), ("zigzag", True, True)])
def test_rank_steps_emulated_ring(ra, layout, causal, pairs):
    """pairs: the backward on CTA pairs, so each rank's work list must keep
    its key tiles two by two."""
    from context_ring_attention_step_gb300.ring_driver import RankCompute, RingDriver
    W = 4
    wl = custom([1500, 300, 77], 4, 2, 128, W, layout, causal, seed=81, name="rank_steps")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    args = (wl.cu_seqlens, [W] * wl.num_docs, layout, causal, wl.softmax_scale)
    plan = ra.Plan(wl.cu_seqlens, [W] * wl.num_docs, layout, causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale,
                   bwd_cta_pairs=pairs)
    o_ref, l_ref = ra.ring_attn_fwd(q, k, v, *args, plan=plan, check=True, fused=False)
    g_ref = ra.ring_attn_bwd(q, k, v, o_ref, do, l_ref, *args, plan=plan, grads_fp32=True, check=True)
    drv = [RingDriver(plan, r, W) for r in range(W)]
    own = [_rows(drv[r].ranges[r]) for r in range(W)]

    def local(x, r):
        y = torch.zeros_like(x)
        y[own[r]] = x[own[r]]
        return y

    comp = [RankCompute(plan, r, local(q, r), local(k, r), local(v, r)) for r in range(W)]

    def move(tensors_of, shard_of, s):
        # rank r passes shard_of(r, s) to rank r + 1
        for r in range(W):
            rows = _rows(drv[r].ranges[shard_of(r, s)])
            for src, dst in zip(tensors_of(r), tensors_of((r + 1) % W)):
                dst[rows] = src[rows]

    for c in comp:
        c.fwd_begin()
    for s in range(W):
        for c in comp:
            c.fwd_step(s)
        if s + 1 < W:
            move(lambda r: (comp[r].k, comp[r].v), lambda r, s: drv[r].source(s), s)
    for c in comp:
        c.fwd_end()
    for r, c in enumerate(comp):
        c.do = local(do, r)
        c.bwd_begin()
    for s in range(W):
        for c in comp:
            c.bwd_step(s)
        move(lambda r: (comp[r].dk, comp[r].dv), lambda r, s: drv[r].source(s), s)
        if s + 1 < W:
            move(lambda r: (comp[r].k, comp[r].v), lambda r, s: drv[r].source(s), s)
    torch.cuda.synchronize()
    for c in comp:
        assert ra.workspace_status(c.ws_f) == 0 and ra.workspace_status(c.ws_b) == 0
    for r, c in enumerate(comp):
        rows = own[r]
        assert torch.equal(c.o[rows], o_ref[rows]), r
        assert torch.equal(c.lse[:, rows], l_ref[:, rows]), r
        for name, x, ref in zip(("dq", "dk", "dv"), (c.dq, c.dk, c.dv), g_ref):
            err = (x[rows] - ref[rows]).abs().max().item()
            assert err <= 1e-5, (r, name, err)
    # and the assembled result against the oracle
    qh, kh, vh, doh = draw_qkvdo(wl)
    rq, rk, rv, ro, rl = A.attention_bwd(qh, kh, vh, doh, wl.cu_seqlens, causal, wl.softmax_scale)
    o = torch.zeros_like(o_ref, dtype=torch.float32)
    lse = torch.zeros_like(l_ref)
    grads = [torch.zeros_like(x) for x in g_ref]
    for r, c in enumerate(comp):
        o[own[r]] = c.o[own[r]].float()
        lse[:, own[r]] = c.lse[:, own[r]]
        for g, x in zip(grads, (c.dq, c.dk, c.dv)):
            g[own[r]] = x[own[r]]
    o = o.cpu().numpy()
    assert (np.abs(o - ro) - (2e-2 + np.abs(ro) * 2.0 ** -9)).max() <= 0
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
    for x, ref in zip(grads, (rq, rk, rv)):
        assert np.abs(x.cpu().numpy() - ref).max() <= 2e-2


def test_rank_steps_emulated_allgather(ra):
    """The all-gather variant's order (ring_driver.AllGatherDriver): every rank
    holds all key/value rows before its first step, runs its steps with no
    exchange, and each key/value shard's dK/dV partials are summed over the
    ranks onto the shard's owner at the end."""
    from context_ring_attention_step_gb300.ring_driver import AllGatherDriver, RankCompute
    W = 4
    layout, causal = "zigzag", True
    wl = custom([1500, 300, 77], 4, 2, 128, W, layout, causal, seed=82, name="rank_steps_allgather")
    q, k, v, do = (x.cuda() for x in draw_qkvdo(wl))
    args = (wl.cu_seqlens, [W] * wl.num_docs, layout, causal, wl.softmax_scale)
    plan = ra.Plan(wl.cu_seqlens, [W] * wl.num_docs, layout, causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale)
    o_ref, l_ref = ra.ring_attn_fwd(q, k, v, *args, plan=plan, check=True, fused=False)
    g_ref = ra.ring_attn_bwd(q, k, v, o_ref, do, l_ref, *args, plan=plan, grads_fp32=True, check=True)
    drv = [AllGatherDriver(plan, r, W) for r in range(W)]
    own = [_rows(drv[r].ranges[r]) for r in range(W)]

    def local(x, r):
        y = torch.zeros_like(x)
        y[own[r]] = x[own[r]]
        return y

    comp = [RankCompute(plan, r, local(q, r), k.clone(), v.clone()) for r in range(W)]  # K, V gathered
    for c in comp:
        c.fwd_begin()
        for s in range(W):
            c.fwd_step(s)
        c.fwd_end()
    for r, c in enumerate(comp):
        c.do = local(do, r)
        c.bwd_begin()
        for s in range(W):
            c.bwd_step(s)
    for j in range(W):  # the per-shard reduction onto the owner
        for name in ("dk", "dv"):
            total = sum(getattr(c, name)[own[j]] for c in comp)
            getattr(comp[j], name)[own[j]] = total
    torch.cuda.synchronize()
    for c in comp:
        assert ra.workspace_status(c.ws_f) == 0 and ra.workspace_status(c.ws_b) == 0
    for r, c in enumerate(comp):
        rows = own[r]
        assert torch.equal(c.o[rows], o_ref[rows]), r
        assert torch.equal(c.lse[:, rows], l_ref[:, rows]), r
        for name, x, ref in zip(("dq", "dk", "dv"), (c.dq, c.dk, c.dv), g_ref):
            err = (x[rows] - ref[rows]).abs().max().item()
            assert err <= 1e-5, (r, name, err)
