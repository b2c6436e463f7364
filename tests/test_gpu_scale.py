"""GPU parity at full size, element by element against the fp64 oracle.

The ring must equal standard attention (NVSHMEM/XLA page, "Paralelismo de
contexto y atencion en anillo"), so every output is compared with the plain
monolithic definition:

* the Llama-3-8B shape at 32K tokens (cp 8 zigzag) and the packed varlen
  batch (65536 tokens, 40 documents, per-document cp): one whole key/value
  head group, kv head 0 with query heads 0..3, i.e. complete O, LSE and dQ of
  those query heads and complete dK, dV of kv head 0 (all four heads
  contribute to them).  The GPU runs the whole workload (all 32 heads) in the
  launch configuration the bench times (single-launch forward, ring-step
  backward, bf16 outputs), then with fp32 outputs, then with the ring-step
  forward;
* a cp = 1 case whose first key tiles meet more than 256 (query head, query
  tile) pairs, so the backward flushes its dK/dV chain from tensor memory into
  the accumulators mid-CTA (twice per CTA, with a chain boundary inside a
  query head), checked in full.

Tolerances: bf16 inputs with fp32 accumulation, max abs error <= 2e-2 on
O/dQ/dK/dV from fp32 outputs and <= 1e-3 on LSE; bf16 outputs add their own
round-to-nearest of at most half a bf16 ulp, so they are held to
2e-2 + 2^-9 |ref|.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import custom, draw_qkvdo, workload

pytestmark = pytest.mark.gpu

TOL, LSE_TOL = 2e-2, 1e-3


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


def _group_reference(wl, q, k, v, do, g):
    """Oracle O, LSE, dQ of query heads [gG, (g+1)G) and dK, dV of kv head g."""
    G = wl.Hq // wl.Hkv
    hs = slice(g * G, (g + 1) * G)
    dq, dk, dv, o, lse = A.attention_bwd(q[:, hs].contiguous(), k[:, g:g + 1].contiguous(),
                                         v[:, g:g + 1].contiguous(), do[:, hs].contiguous(),
                                         wl.cu_seqlens, wl.causal, wl.softmax_scale)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk[:, 0], "dv": dv[:, 0]}


def _gpu_group(ra, wl, qd, kd, vd, dod, g, o_fp32, grads_fp32, fused, pairs=False):
    G = wl.Hq // wl.Hkv
    cps = list(wl.cp_per_doc)
    plan = ra.Plan(wl.cu_seqlens, cps, wl.layout, wl.causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale,
                   bwd_cta_pairs=pairs)
    o, lse = ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, wl.layout, wl.causal, wl.softmax_scale,
                              o_fp32=o_fp32, plan=plan, check=True, fused=fused)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, o, dod, lse, wl.cu_seqlens, cps, wl.layout, wl.causal,
                                  wl.softmax_scale, grads_fp32=grads_fp32, plan=plan, check=True)
    torch.cuda.synchronize()
    hs = slice(g * G, (g + 1) * G)
    out = {"o": o[:, hs], "lse": lse[hs], "dq": dq[:, hs], "dk": dk[:, g], "dv": dv[:, g]}
    return {n: x.float().cpu().numpy() for n, x in out.items()}


def _compare(tag, got, ref, bf16_out, bf16_grads):
    errs = {}
    for name in ("o", "lse", "dq", "dk", "dv"):
        x, r = got[name], ref[name]
        assert x.shape == r.shape, (tag, name, x.shape, r.shape)
        assert np.isfinite(x).all(), (tag, name)
        err = np.abs(x - r)
        errs[name] = float(err.max())
        if name == "lse":
            bound = LSE_TOL
        else:
            rounded = bf16_out if name == "o" else bf16_grads
            bound = TOL + (np.abs(r) * 2.0 ** -9 if rounded else 0.0)
        assert (err - bound).max() <= 0, (tag, name, errs[name])
    print("parity %s: max abs errors %s" % (tag, {n: "%.3g" % e for n, e in errs.items()}))
    return errs


def _full_group_check(ra, wl, g=0):
    q, k, v, do = draw_qkvdo(wl)
    ref = _group_reference(wl, q, k, v, do, g)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    # the bench's configuration: single-launch forward, ring-step backward, bf16 outputs
    _compare(wl.name + " bf16", _gpu_group(ra, wl, qd, kd, vd, dod, g, False, False, None), ref, True, True)
    _compare(wl.name + " fp32", _gpu_group(ra, wl, qd, kd, vd, dod, g, True, True, None), ref, False, False)
    # the ring-step forward (one launch per ring step, merge in the epilogue)
    _compare(wl.name + " ring-step fwd fp32", _gpu_group(ra, wl, qd, kd, vd, dod, g, True, True, False), ref,
             False, False)


def test_llama_32k_full_kv_group(ra):
    _full_group_check(ra, workload("llama3_8b_32k"))


@pytest.mark.parametrize("name", ["llama3_8b_32k", "varlen_65k"])
def test_cta_pair_backward_full_kv_group(ra, name):
    """The CTA-pair backward in the bench's launch configuration (bf16 outputs)
    and with fp32 gradients, one whole KV-head group element by element."""
    wl = workload(name)
    q, k, v, do = draw_qkvdo(wl)
    ref = _group_reference(wl, q, k, v, do, 0)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    _compare(wl.name + " pairs bf16", _gpu_group(ra, wl, qd, kd, vd, dod, 0, False, False, None, True), ref, True,
             True)
    _compare(wl.name + " pairs fp32", _gpu_group(ra, wl, qd, kd, vd, dod, 0, True, True, None, True), ref, False,
             False)


def test_varlen_65k_full_kv_group(ra):
    _full_group_check(ra, workload("varlen_65k"))


@pytest.mark.parametrize("d,causal,L", [(128, True, 24000), (128, False, 9000), (64, True, 24000),
                                         (256, True, 9000)])
def test_dkdv_chain_flush_cp1(ra, d, causal, L):
    """cp = 1, 4 query heads on one kv head (the GQA ratio of the workloads):
    the first key tiles of a 24000-token causal document meet 188 query tiles
    x 4 heads = 752 pairs, i.e. two chain flushes mid-CTA (at pairs 256 and
    512, inside query heads 1 and 2) before the final one; without a mask a
    9000-token document gives 71 x 4 = 284 pairs, one flush.  At head_dim 256
    the query tiles are 64 rows: 141 x 4 = 564 pairs, two flushes."""
    wl = custom([L, 1500], 4, 1, d, [1, 1], "zigzag", causal, seed=51, name="chain_flush")
    q, k, v, do = draw_qkvdo(wl)
    ref = _group_reference(wl, q, k, v, do, 0)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    _compare("chain flush d=%d causal=%s fp32" % (d, causal),
             _gpu_group(ra, wl, qd, kd, vd, dod, 0, True, True, None), ref, False, False)
    _compare("chain flush d=%d causal=%s bf16" % (d, causal),
             _gpu_group(ra, wl, qd, kd, vd, dod, 0, False, False, None), ref, True, True)
    if d == 128:  # the CTA-pair backward flushes its own chains
        _compare("chain flush d=%d causal=%s pairs fp32" % (d, causal),
                 _gpu_group(ra, wl, qd, kd, vd, dod, 0, True, True, None, True), ref, False, False)
