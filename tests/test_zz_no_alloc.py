"""ra_fwd_noalloc: the forward for callers that cannot allocate device memory.

Callers inside a host framework that owns every device allocation, or in a
loop that must not allocate, get the forward without handing over a
workspace: the library uses a fixed 32 MiB device array of its own instead.
These tests call it through the C ABI and compare it with ra_fwd on two calls
in a row with different problems (every call reuses the same array, so a
stale work list or status word from the previous call would show).  The
forward has no atomics and ra_fwd_noalloc runs the same kernel as ra_fwd, so
the outputs must be bit-identical; ra_noalloc_status must read RA_OK.

This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from workloads import custom, draw_qkvdo


@pytest.fixture(scope="module")
def ra():
    import context_ring_attention_step_gb300 as m
    m.load_library()
    return m


def _noalloc(ra, plan, q, k, v, o_fp32):
    lib = ra.load_library()
    T, Hq, D = q.shape
    o = torch.full((T, Hq, D), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=q.device)
    lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device=q.device)
    p = ra.ring_attn._ptr
    stream = ra.ring_attn._stream(q.device)
    st = lib.ra_fwd_noalloc(plan.handle, p(q), p(k), p(v), p(o), int(o_fp32), p(lse), stream)
    assert st == 0, lib.ra_last_error()
    assert lib.ra_noalloc_status(stream) == 0, lib.ra_last_error()
    return o, lse


@pytest.mark.gpu
def test_noalloc_forward_equals_ra_fwd_twice_in_a_row(ra):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cases = [
        (custom([1500, 300], 4, 2, 128, [3, 2], "zigzag", True, seed=41, name="na1"), False),
        (custom([700, 1, 90], 2, 1, 64, [4, 1, 2], "contiguous", True, seed=42, name="na2"), True),
    ]
    for wl, o_fp32 in cases:
        q, k, v, _ = (x.cuda() for x in draw_qkvdo(wl))
        plan = ra.Plan(wl.cu_seqlens, list(wl.cp_per_doc), wl.layout, wl.causal, wl.Hq, wl.Hkv, wl.d,
                       wl.softmax_scale)
        o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, wl.cu_seqlens, list(wl.cp_per_doc), wl.layout, wl.causal,
                                          wl.softmax_scale, o_fp32=o_fp32, plan=plan, check=True)
        o, lse = _noalloc(ra, plan, q, k, v, o_fp32)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert torch.equal(o, o_ref), (wl.name, (o.float() - o_ref.float()).abs().max().item())
        assert torch.equal(lse, lse_ref), wl.name


def test_noalloc_rejects_plans_above_the_scratch_limit(ra):
    """A plan needing more than 32 MiB of scratch is refused before any GPU work.

    512K tokens without a mask, cp 1: 2048 query chunks each meeting 4096 key
    tiles, 8 bytes per tile in the key-tile table (64 MiB)."""
    lib = ra.load_library()
    plan = ra.Plan([0, 524288], 1, "zigzag", False, 1, 1, 64)
    assert plan.workspace_bytes(o_fp32=False)[0] > 32 << 20
    p = ctypes.c_void_p
    st = lib.ra_fwd_noalloc(plan.handle, p(256), p(512), p(768), p(1024), 0, p(1280), p(0))
    assert st == 4
    assert b"fixed maximum" in lib.ra_last_error()
