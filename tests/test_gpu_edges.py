"""GPU edge cases against the fp64 oracle: empty documents inside cu_seqlens,
a single token, more ring shards than tokens (empty shards), a token count
that is not a multiple of 4 (the padded LSE/Delta rows), for the ring-step
forward, the single-launch forward and the backward, at head_dim 64, 128
(with the one-CTA and the CTA-pair backward) and 256.  Tolerances as in the
other parity tests: 2e-2 on fp32 outputs, 1e-3 on LSE."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import custom, draw_qkvdo

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL = 2e-2, 1e-3

CASES = [
    ("empty_docs", [0, 300, 0, 0, 129, 1, 0], [2, 3, 1, 4, 8, 1, 5]),
    ("one_token", [1], [1]),
    ("one_token_cp4", [1], [4]),
    ("more_shards_than_tokens", [3, 5, 2], [8, 8, 4]),
    ("t_not_multiple_of_4", [1001, 2], [3, 2]),
]


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


VARIANTS = [("d64", 64, False), ("d128", 128, False), ("d128_pairs", 128, True), ("d256", 256, False)]


@pytest.mark.parametrize("variant", VARIANTS, ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_edge_case(ra, case, layout, causal, variant):
    name, lengths, cps = case
    _, d, pairs = variant
    wl = custom(lengths, 4, 2, d, cps, layout, causal, seed=31, name=name)
    q, k, v, do = draw_qkvdo(wl)
    rq, rk, rv, ro, rl = A.attention_bwd(q, k, v, do, wl.cu_seqlens, causal, wl.softmax_scale)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    plan = ra.Plan(wl.cu_seqlens, cps, layout, causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale, bwd_cta_pairs=pairs)
    for fused in (False, True):
        o, lse = ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, layout, causal, wl.softmax_scale, o_fp32=True,
                                  plan=plan, check=True, fused=fused)
        o, lse_h = o.cpu().numpy(), lse.cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(lse_h).all()
        assert np.abs(o - ro).max() <= O_TOL, (name, fused)
        assert np.abs(lse_h - rl).max() <= LSE_TOL, (name, fused)
    o, lse = ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, layout, causal, wl.softmax_scale, o_fp32=True,
                              plan=plan, check=True)
    dq, dk, dv = ra.ring_attn_bwd(qd, kd, vd, o, dod, lse, wl.cu_seqlens, cps, layout, causal, wl.softmax_scale,
                                  grads_fp32=True, plan=plan, check=True)
    for nm, a, b in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        a = a.cpu().numpy()
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= O_TOL, (name, nm, np.abs(a - b).max())
