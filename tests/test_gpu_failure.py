"""Failure detection on the GPU without a fault: a bounded pipeline wait that
nothing completes gives up after its limit, records its site in the workspace
status word (read back as RA_ERR_TIMEOUT) and returns; the CUDA context stays
usable (a forward run afterwards still matches the oracle)."""

import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import draw_qkvdo, workload


@pytest.fixture(scope="module")
def ra(lib_path):
    import context_ring_attention_step_gb300 as m
    m.load_library(lib_path)
    return m


def test_selftest_rejects_bad_arguments_on_the_host(ra):
    lib = ra.load_library()
    p = ctypes.c_void_p
    assert lib.ra_selftest_wait_timeout(p(0), 1000, p(0)) == 1
    assert lib.ra_selftest_wait_timeout(p(256), 0, p(0)) == 1
    assert lib.ra_selftest_wait_timeout(p(256), 5000000, p(0)) == 1
    assert lib.ra_selftest_wait_timeout(p(8), 1000, p(0)) == 1   # misaligned


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_survives(ra):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = ra.load_library()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sp = ra.ring_attn._stream(ws.device)
    torch.cuda.synchronize()
    t0 = time.time()
    assert lib.ra_selftest_wait_timeout(ra.ring_attn._ptr(ws), 100000, sp) == 0   # 0.1 s limit
    st = lib.ra_workspace_status(ra.ring_attn._ptr(ws), sp)
    dt = time.time() - t0
    assert st == 5, lib.ra_last_error()
    assert b"site 900" in lib.ra_last_error()
    assert 0.09 <= dt < 5.0
    # the context is usable afterwards
    wl = workload("tiny")
    q, k, v, _ = draw_qkvdo(wl)
    o, lse = ra.ring_attn_fwd(q.cuda(), k.cuda(), v.cuda(), wl.cu_seqlens, list(wl.cp_per_doc), wl.layout, True,
                              wl.softmax_scale, o_fp32=True, check=True)
    ro, rl = A.attention_fwd(q, k, v, wl.cu_seqlens, True, wl.softmax_scale)
    assert np.abs(o.cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
