"""Python binding of the ring-attention C ABI (``include/ring_attn.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libring_attn.so``.  PyTorch supplies device memory and the
current CUDA stream.  If the library is missing the calls raise; there is no
fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LAYOUTS = {"contiguous": 0, "zigzag": 1}

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_WORKSPACE, RA_ERR_TIMEOUT = range(6)

_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("ring_attn status %d: %s" % (status, msg))
        self.status = status


def load_library(path: str | None = None):
    """Load libring_attn.so (building it first when the sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.LIB
        if not _build.up_to_date():
            _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libring_attn.so not found at %s: run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    c = ctypes
    P = c.c_void_p
    i32, i64, sz = c.c_int32, c.c_int64, c.c_size_t
    lib.ra_abi_version.restype = i32
    lib.ra_last_error.restype = c.c_char_p
    lib.ra_plan_create.argtypes = [c.POINTER(P), c.POINTER(i32), i32, c.POINTER(i32), i32, i32, i32,
                                   i32, i32, i32, c.c_float]
    lib.ra_plan_create.restype = i32
    lib.ra_plan_destroy.argtypes = [P]
    lib.ra_plan_destroy.restype = None
    lib.ra_plan_workspace_bytes.argtypes = [P, i32, i32, c.POINTER(sz), c.POINTER(sz)]
    lib.ra_plan_workspace_bytes.restype = i32
    lib.ra_plan_stats.argtypes = [P, c.POINTER(i32), c.POINTER(i64), c.POINTER(i64), c.POINTER(i64)]
    lib.ra_plan_stats.restype = i32
    lib.ra_plan_set_bwd_cta_pairs.argtypes = [P, i32]
    lib.ra_plan_set_bwd_cta_pairs.restype = i32
    lib.ra_shard_token_ranges.argtypes = [P, i32, i32, c.POINTER(i32), c.POINTER(i32), c.POINTER(i32)]
    lib.ra_shard_token_ranges.restype = i32
    lib.ra_plan_work_items.argtypes = [P, i32, c.POINTER(i32), i64, c.POINTER(i64), c.POINTER(i64)]
    lib.ra_plan_work_items.restype = i32
    lib.ra_fwd.argtypes = [P, P, P, P, P, i32, P, P, sz, P]
    lib.ra_fwd.restype = i32
    lib.ra_fwd_ring_steps.argtypes = [P, P, P, P, P, i32, P, P, sz, P]
    lib.ra_fwd_ring_steps.restype = i32
    lib.ra_plan_ring_step_workspace_bytes.argtypes = [P, i32, c.POINTER(sz)]
    lib.ra_plan_ring_step_workspace_bytes.restype = i32
    lib.ra_fwd_noalloc.argtypes = [P, P, P, P, P, i32, P, P]
    lib.ra_fwd_noalloc.restype = i32
    lib.ra_noalloc_status.argtypes = [P]
    lib.ra_noalloc_status.restype = i32
    lib.ra_bwd.argtypes = [P, P, P, P, P, i32, P, P, P, P, P, i32, P, sz, P]
    lib.ra_bwd.restype = i32
    lib.ra_fwd_prepare.argtypes = [P, i32, P, sz, P]
    lib.ra_fwd_ring_step.argtypes = [P, i32, P, P, P, P, i32, P, P, sz, P]
    lib.ra_fwd_finish.argtypes = [P, P, i32, P, sz, P]
    lib.ra_bwd_prepare.argtypes = [P, P, i32, P, P, P, P, P, i32, P, sz, P]
    lib.ra_bwd_ring_step.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, sz, P]
    lib.ra_bwd_finish.argtypes = [P, P, P, P, i32, P, sz, P]
    for name in ("ra_fwd_prepare", "ra_fwd_ring_step", "ra_fwd_finish", "ra_bwd_prepare", "ra_bwd_ring_step",
                 "ra_bwd_finish"):
        getattr(lib, name).restype = i32
    lib.ra_fwd_ring_step_rank.argtypes = [P, i32, i32, P, P, P, P, i32, P, P, sz, P]
    lib.ra_fwd_ring_step_rank.restype = i32
    lib.ra_bwd_ring_step_rank.argtypes = [P, i32, i32, P, P, P, P, P, P, P, i32, P, sz, P]
    lib.ra_bwd_ring_step_rank.restype = i32
    lib.ra_plan_rank_work_items.argtypes = [P, i32, c.POINTER(i32), i64, c.POINTER(i64), c.POINTER(i64)]
    lib.ra_plan_rank_work_items.restype = i32
    lib.ra_fwd_fused.argtypes = [P, P, P, P, P, i32, P, P, sz, P]
    lib.ra_fwd_fused.restype = i32
    lib.ra_plan_fused_workspace_bytes.argtypes = [P, c.POINTER(sz)]
    lib.ra_plan_fused_workspace_bytes.restype = i32
    lib.ra_plan_fused_items.argtypes = [P, c.POINTER(i32), i64, c.POINTER(i32), i64, c.POINTER(i64), c.POINTER(i64)]
    lib.ra_plan_fused_items.restype = i32
    lib.ra_dynamic_cp.argtypes = [c.POINTER(i32), i32, i32, i64, i32, c.c_double, c.c_double, i32,
                                  c.POINTER(i32), c.POINTER(i32), c.POINTER(c.c_double), c.POINTER(i64)]
    lib.ra_dynamic_cp.restype = i32
    lib.ra_selftest_wait_timeout.argtypes = [P, c.c_uint32, P]
    lib.ra_selftest_wait_timeout.restype = i32
    lib.ra_workspace_status.argtypes = [P, P]
    lib.ra_workspace_status.restype = i32
    _lib = lib
    return lib


def _check(status):
    if status != RA_OK:
        raise RingAttnError(status, _lib.ra_last_error().decode())


def _i32_array(values):
    values = [int(x) for x in values]
    return (ctypes.c_int32 * max(1, len(values)))(*values)


class Plan:
    """Host-side ring plan: shards, ring pairing and GPU work items."""

    def __init__(self, cu_seqlens, cp_size, layout="zigzag", causal=True, num_q_heads=1,
                 num_kv_heads=1, head_dim=128, scale=None, bwd_cta_pairs=False):
        """``bwd_cta_pairs=True`` (head_dim 128) runs the backward on CTA pairs
        (ra_plan_set_bwd_cta_pairs)."""
        lib = load_library()
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        self.num_docs = len(cu) - 1
        per_doc = None
        cp_all = 0
        if isinstance(cp_size, (list, tuple)):
            per_doc = _i32_array(cp_size)
        else:
            cp_all = int(cp_size)
        self.cp_per_doc = [int(x) for x in cp_size] if per_doc is not None else [cp_all] * self.num_docs
        self._handle = ctypes.c_void_p()
        self.layout = layout
        self.causal = bool(causal)
        self.Hq, self.Hkv, self.D = int(num_q_heads), int(num_kv_heads), int(head_dim)
        self.T = cu[-1]
        _check(lib.ra_plan_create(ctypes.byref(self._handle), _i32_array(cu), self.num_docs, per_doc,
                                  cp_all, LAYOUTS[layout] if isinstance(layout, str) else int(layout),
                                  1 if causal else 0, self.Hq, self.Hkv, self.D,
                                  float(scale) if scale else 0.0))
        self.bwd_cta_pairs = False
        if bwd_cta_pairs:
            self.set_bwd_cta_pairs(True)

    def set_bwd_cta_pairs(self, on=True):
        """Backward on CTA pairs (head_dim 128) or on single CTAs; rebuilds the
        plan's backward work lists."""
        _check(_lib.ra_plan_set_bwd_cta_pairs(self._handle, 1 if on else 0))
        self.bwd_cta_pairs = bool(on)

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h and _lib is not None:
            _lib.ra_plan_destroy(h)
            self._handle = None

    @property
    def handle(self):
        return self._handle

    def workspace_bytes(self, o_fp32=False, grads_fp32=False):
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.ra_plan_workspace_bytes(self._handle, int(o_fp32), int(grads_fp32),
                                            ctypes.byref(f), ctypes.byref(b)))
        return f.value, b.value

    def stats(self):
        s, vp, fi, bi = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.ra_plan_stats(self._handle, ctypes.byref(s), ctypes.byref(vp), ctypes.byref(fi),
                                  ctypes.byref(bi)))
        return {"steps": s.value, "visible_pairs": vp.value, "fwd_items": fi.value, "bwd_items": bi.value}

    def work_items(self, which="fwd"):
        """(items as a list of 8-int tuples, step offsets) of the forward or backward pass."""
        w = 0 if which == "fwd" else 1
        n = ctypes.c_int64()
        _check(_lib.ra_plan_work_items(self._handle, w, None, 0, None, ctypes.byref(n)))
        steps = self.stats()["steps"]
        buf = (ctypes.c_int32 * max(1, 8 * n.value))()
        off = (ctypes.c_int64 * (steps + 1))()
        _check(_lib.ra_plan_work_items(self._handle, w, buf, n.value, off, ctypes.byref(n)))
        items = [tuple(buf[8 * i:8 * i + 8]) for i in range(n.value)]
        return items, list(off)

    def ring_step_workspace_bytes(self, o_fp32=False):
        """Workspace bytes of the ring-step forward (one launch per ring step)."""
        f = ctypes.c_size_t()
        _check(_lib.ra_plan_ring_step_workspace_bytes(self._handle, int(o_fp32), ctypes.byref(f)))
        return f.value

    def rank_work_items(self, which="fwd"):
        """Per-rank work lists: {(step, rank): [items as 8-int tuples]}."""
        w = 0 if which == "fwd" else 1
        n = ctypes.c_int64()
        _check(_lib.ra_plan_rank_work_items(self._handle, w, None, 0, None, ctypes.byref(n)))
        steps = self.stats()["steps"]
        buf = (ctypes.c_int32 * max(1, 8 * n.value))()
        off = (ctypes.c_int64 * (steps * steps + 1))()
        _check(_lib.ra_plan_rank_work_items(self._handle, w, buf, n.value, off, ctypes.byref(n)))
        out = {}
        for s in range(steps):
            for r in range(steps):
                c = s * steps + r
                out[(s, r)] = [tuple(buf[8 * i:8 * i + 8]) for i in range(off[c], off[c + 1])]
        return out

    def fused_workspace_bytes(self):
        """Workspace bytes of the single-launch forward."""
        f = ctypes.c_size_t()
        _check(_lib.ra_plan_fused_workspace_bytes(self._handle, ctypes.byref(f)))
        return f.value

    def fused_items(self):
        """(items as 8-int tuples, tiles as (start, range end) pairs) of the single-launch forward."""
        ni, nt = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.ra_plan_fused_items(self._handle, None, 0, None, 0, ctypes.byref(ni), ctypes.byref(nt)))
        ib = (ctypes.c_int32 * max(1, 8 * ni.value))()
        tb = (ctypes.c_int32 * max(1, 2 * nt.value))()
        _check(_lib.ra_plan_fused_items(self._handle, ib, ni.value, tb, nt.value, ctypes.byref(ni),
                                        ctypes.byref(nt)))
        return [tuple(ib[8 * i:8 * i + 8]) for i in range(ni.value)], [tuple(tb[2 * i:2 * i + 2])
                                                                      for i in range(nt.value)]

    def shard_token_ranges(self, doc, rank):
        b, e, n = (ctypes.c_int32 * 2)(), (ctypes.c_int32 * 2)(), ctypes.c_int32()
        _check(_lib.ra_shard_token_ranges(self._handle, int(doc), int(rank), b, e, ctypes.byref(n)))
        return [(b[i], e[i]) for i in range(n.value)]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_tensor(name, t, shape, dtype):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.dtype != dtype:
        raise ValueError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))


def ring_attn_fwd(q, k, v, cu_seqlens, cp_size, layout="zigzag", causal=True, scale=None,
                  o_fp32=False, plan=None, workspace=None, check=False, fused=None, out=None):
    """Ring attention forward: returns (o [T,Hq,d], lse [Hq,T] fp32).

    By default (``fused=None`` or ``True``) the whole ring runs in one launch
    (ra_fwd); ``fused=False`` runs one launch per ring step
    (ra_fwd_ring_steps).  ``out=(o, lse)`` writes into caller-owned tensors
    instead of allocating them.  ``check=True`` synchronises and raises if a
    kernel reported a timeout.
    """
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if plan is None:
        plan = Plan(cu_seqlens, cp_size, layout, causal, Hq, Hkv, D, scale)
    _check_tensor("q", q, (T, Hq, D), torch.bfloat16)
    _check_tensor("k", k, (T, Hkv, D), torch.bfloat16)
    _check_tensor("v", v, (T, Hkv, D), torch.bfloat16)
    dev = q.device
    ot = torch.float32 if o_fp32 else torch.bfloat16
    if out is None:
        o = torch.empty((T, Hq, D), dtype=ot, device=dev)
        lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    else:
        o, lse = out
        _check_tensor("o", o, (T, Hq, D), ot)
        _check_tensor("lse", lse, (Hq, T), torch.float32)
    steps = fused is False
    ws_bytes = plan.ring_step_workspace_bytes(o_fp32) if steps else plan.workspace_bytes(o_fp32=o_fp32)[0]
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    call = _lib.ra_fwd_ring_steps if steps else _lib.ra_fwd
    _check(call(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), int(o_fp32), _ptr(lse),
                _ptr(workspace), workspace.numel(), _stream(dev)))
    if check:
        _check(workspace_status(workspace, dev))
    return o, lse


def ring_attn_bwd(q, k, v, o, do, lse, cu_seqlens, cp_size, layout="zigzag", causal=True, scale=None,
                  grads_fp32=False, plan=None, workspace=None, check=False, out=None):
    """Ring attention backward from the saved LSE: returns (dq, dk, dv).

    ``out=(dq, dk, dv)`` writes into caller-owned tensors instead of
    allocating them.  ``check=True`` synchronises and raises if a kernel
    reported a timeout.
    """
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if plan is None:
        plan = Plan(cu_seqlens, cp_size, layout, causal, Hq, Hkv, D, scale)
    _check_tensor("q", q, (T, Hq, D), torch.bfloat16)
    _check_tensor("k", k, (T, Hkv, D), torch.bfloat16)
    _check_tensor("v", v, (T, Hkv, D), torch.bfloat16)
    _check_tensor("do", do, (T, Hq, D), torch.bfloat16)
    _check_tensor("lse", lse, (Hq, T), torch.float32)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("o must be bf16 or fp32")
    _check_tensor("o", o, (T, Hq, D), o.dtype)
    dev = q.device
    gt = torch.float32 if grads_fp32 else torch.bfloat16
    if out is None:
        dq = torch.empty((T, Hq, D), dtype=gt, device=dev)
        dk = torch.empty((T, Hkv, D), dtype=gt, device=dev)
        dv = torch.empty((T, Hkv, D), dtype=gt, device=dev)
    else:
        dq, dk, dv = out
        _check_tensor("dq", dq, (T, Hq, D), gt)
        _check_tensor("dk", dk, (T, Hkv, D), gt)
        _check_tensor("dv", dv, (T, Hkv, D), gt)
    ws_bytes = plan.workspace_bytes(grads_fp32=grads_fp32)[1]
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _check(_lib.ra_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), int(o.dtype == torch.float32),
                       _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), int(grads_fp32),
                       _ptr(workspace), workspace.numel(), _stream(dev)))
    if check:
        _check(workspace_status(workspace, dev))
    return dq, dk, dv


class RingAttention(torch.autograd.Function):
    """Autograd wrapper: the forward runs ring_attn_fwd and saves (q, k, v, o,
    lse); the backward runs ring_attn_bwd from the saved LSE.  Gradients flow
    to q, k and v only.  Use ``ring_attention(...)``."""

    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, cp_size, layout, causal, scale, plan):
        o, lse = ring_attn_fwd(q, k, v, cu_seqlens, cp_size, layout, causal, scale, plan=plan)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.args = (cu_seqlens, cp_size, layout, causal, scale, plan)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        cu_seqlens, cp_size, layout, causal, scale, plan = ctx.args
        dq, dk, dv = ring_attn_bwd(q, k, v, o, do.contiguous().to(torch.bfloat16), lse, cu_seqlens, cp_size,
                                   layout, causal, scale, plan=plan)
        return dq, dk, dv, None, None, None, None, None, None


def ring_attention(q, k, v, cu_seqlens, cp_size, layout="zigzag", causal=True, scale=None, plan=None):
    """Differentiable ring attention: returns (o, lse); o.backward(dO) fills
    q.grad, k.grad and v.grad through the ring backward."""
    if plan is None:
        plan = Plan(cu_seqlens, cp_size, layout, causal, q.shape[1], k.shape[1], q.shape[2], scale)
    return RingAttention.apply(q, k, v, cu_seqlens, cp_size, layout, causal, scale, plan)


def workspace_status(workspace, device=None):
    """Synchronise and return the status word of the last call on this workspace."""
    dev = workspace.device if device is None else device
    return _lib.ra_workspace_status(_ptr(workspace), _stream(dev))


def dynamic_cp(doc_lengths, num_ranks, max_tokens_per_rank, causal=True, sec_per_pair=1.0, sec_per_token=0.0,
               mode="dynamic"):
    """Dynamic-CP sizing (ra_dynamic_cp): per-sequence group sizes and placement.

    Returns a dict with ``cp_per_doc``, ``first_rank``, ``rank_load`` (modelled
    seconds) and ``rank_tokens``.
    """
    lib = load_library()
    n = len(doc_lengths)
    lens = _i32_array(doc_lengths)
    cp = (ctypes.c_int32 * max(1, n))()
    first = (ctypes.c_int32 * max(1, n))()
    load = (ctypes.c_double * num_ranks)()
    tok = (ctypes.c_int64 * num_ranks)()
    m = {"dynamic": 0, "static": 1}[mode]
    _check(lib.ra_dynamic_cp(lens, n, int(num_ranks), int(max_tokens_per_rank), int(bool(causal)),
                             float(sec_per_pair), float(sec_per_token), m, cp, first, load, tok))
    return {"cp_per_doc": list(cp[:n]), "first_rank": list(first[:n]), "rank_load": list(load),
            "rank_tokens": list(tok)}
