#!/usr/bin/env python3
"""Ring-attention fwd+bwd throughput on GB300 (useful causal TFLOP/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = the whole hot path on one batch: ring forward (every ring step in
one launch, the merge of each step into the running state kept on chip, bf16
output; ra_fwd) then ring backward (Delta preprocess, one launch per ring
step, bf16 gradients; ra_bwd's calls), on seeded synthetic bf16 inputs
resident in HBM.  The forward with one launch per ring step (merge through
HBM) is timed beside it and reported as ring_step_forward.  Useful FLOPs count visible (query, key) pairs only: forward 4 d Hq P,
backward 10 d Hq P (P = sum over documents of L(L+1)/2 when causal).

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica of the same workload ("replicas only": on one GPU per box the ring has
no inter-GPU exchange); value = all ranks' FLOPs / max-over-ranks time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attn fwd+bwd TFLOP/s (useful, causal) on 1 GB300; % of BF16 dense peak"


def visible_pairs(wl):
    return sum(L * (L + 1) // 2 if wl.causal else L * L for L in wl.doc_lengths)


def useful_flops(wl, pairs=None):
    P = visible_pairs(wl) if pairs is None else pairs
    return 4.0 * wl.d * wl.Hq * P, 10.0 * wl.d * wl.Hq * P


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["bf16_tflops_sustained"]), float(m["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


KERNEL_SOURCES = {
    "ring_fwd_step_kernel": ("fwd.cu", "tc.cuh", "ring_attn_internal.h"),
    "ring_bwd_step_kernel": ("bwd.cu", "bwd_tiles.cuh", "tc.cuh", "ring_attn_internal.h"),
}


def strip_comments(src):
    """C++ source without comments, blank lines and runs of whitespace (an
    edit to a comment or to spacing does not change the kernel)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(" ".join(line.split()) for line in src.splitlines() if line.strip())


def kernel_source_hash(kernel):
    """sha256 (first 16 hex digits) of the code a kernel is built from
    (comments, blank lines and spacing removed)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "context_ring_attention_step_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload_name):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of this
    workload, or None when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_%s.md" % workload_name)
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    want = kernel_source_hash(kernel)
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel:
            try:
                return float(cells[2]) if cells[3] == want else None
            except ValueError:
                return None
    return None


def max_over_ranks(ms, dist=None, device=None):
    """Max of a per-rank time over all ranks (identity on one process)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_step, steps, ms_total):
    """Whole-job throughput: every replica's useful FLOPs over the slowest rank's time."""
    return world * flops_per_step * steps / (ms_total * 1e-3) / 1e12


def step_pairs_bwd(items, off, causal):
    """Visible (query, key) pairs processed by each backward ring-step launch."""
    import numpy as np
    out = []
    for s in range(len(off) - 1):
        tot = 0
        for k0, k1, qb0, qe0, qb1, qe1, flags, _ in items[off[s]:off[s + 1]]:
            if flags >> 8:  # backward items are per key/value head: count head 0 only
                continue
            keys = np.arange(k0, k1)
            for qb, qe in ((qb0, qe0), (qb1, qe1)):
                if qe <= qb:
                    continue
                if causal:  # queries q in [qb, qe) with q >= k
                    tot += int(np.clip(qe - np.maximum(qb, keys), 0, None).sum())
                else:
                    tot += (k1 - k0) * (qe - qb)
        out.append(tot)
    return out


def step_pairs_fwd(items, off, causal):
    """Visible (query, key) pairs processed by each forward ring-step launch."""
    import numpy as np
    out = []
    for s in range(len(off) - 1):
        tot = 0
        for q0, q1, kb0, ke0, kb1, ke1, _, _ in items[off[s]:off[s + 1]]:
            rows = np.arange(q0, q1)
            for kb, ke in ((kb0, ke0), (kb1, ke1)):
                if ke <= kb:
                    continue
                if causal:  # keys k in [kb, ke) with k <= q
                    tot += int(np.clip(np.minimum(rows + 1, ke) - kb, 0, None).sum())
                else:
                    tot += (q1 - q0) * (ke - kb)
        out.append(tot)
    return out


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(wl, q, k, v, do, tokens):
    """fp64 oracle fwd+bwd on a causal prefix of `tokens` tokens of query head 0."""
    from oracle import attention as A
    import torch
    Tn = min(tokens, wl.doc_lengths[0])
    qs, ks, vs, dos = (x[:Tn] for x in (q, k, v, do))
    qs = qs[:, :1].contiguous()
    dos = dos[:, :1].contiguous()
    ks = ks[:, :1].contiguous()
    vs = vs[:, :1].contiguous()
    t0 = time.perf_counter()
    A.attention_bwd(qs, ks, vs, dos, [0, Tn], wl.causal, wl.softmax_scale)
    dt = time.perf_counter() - t0
    P = Tn * (Tn + 1) // 2 if wl.causal else Tn * Tn
    flops = 14.0 * wl.d * 1 * P
    del torch
    return flops, dt, "causal prefix of %d tokens of document 0, query head 0 / kv head 0, fwd+bwd in float64" % Tn


def cpu_parity_sample(wl, q, k, v, do, o, lse, dq, dk, dv, nrows=16):
    """Max abs errors of the bench's own outputs (bf16 O, dQ, dK, dV; fp32 LSE)
    against the fp64 oracle on a sample that the oracle computes exactly one
    output at a time: O, LSE and dQ of sampled query rows (random rows plus
    every document's first and last row) of the first and last query heads,
    and, under a causal mask, dK and dV of the last 128 keys of the longest
    document for the first and last key/value heads."""
    import numpy as np
    from oracle import attention as A
    G = wl.Hq // wl.Hkv
    cu = wl.cu_seqlens
    rng = np.random.default_rng(wl.seed)
    rows = set(rng.integers(0, wl.T, nrows).tolist())
    for d in range(wl.num_docs):
        if cu[d + 1] > cu[d]:
            rows.update({cu[d], cu[d + 1] - 1})
    rows = sorted(rows)
    err = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    excess = -1.0  # max over outputs of |err| - bound (<= 0: within the bounds)
    ridx = torch_index(rows)
    for h in (0, wl.Hq - 1):
        g = h // G
        qh, dh = q[:, h:h + 1].contiguous(), do[:, h:h + 1].contiguous()
        kh, vh = k[:, g:g + 1].contiguous(), v[:, g:g + 1].contiguous()
        ro, rl = A.attention_rows(qh, kh, vh, cu, rows, 0, wl.causal, wl.softmax_scale)
        rdq = A.attention_rows_dq(qh, kh, vh, dh, cu, rows, 0, wl.causal, wl.softmax_scale)
        go = o[ridx, h].float().cpu().numpy()
        gl = lse[h, ridx].cpu().numpy()
        gq = dq[ridx, h].float().cpu().numpy()
        for name, x, r in (("o", go, ro), ("dq", gq, rdq)):
            e = np.abs(x - r)
            err[name] = max(err[name], float(e.max()))
            excess = max(excess, float((e - (2e-2 + np.abs(r) * 2.0 ** -9)).max()))
        err["lse"] = max(err["lse"], float(np.abs(gl - rl).max()))
        excess = max(excess, err["lse"] - 1e-3)
    what = "O, LSE, dQ of %d query rows of query heads 0 and %d" % (len(rows), wl.Hq - 1)
    if wl.causal:
        longest = max(range(wl.num_docs), key=lambda d: cu[d + 1] - cu[d])
        keys = list(range(max(cu[longest], cu[longest + 1] - 128), cu[longest + 1]))
        kidx = torch_index(keys)
        for g in (0, wl.Hkv - 1):
            hs = slice(g * G, (g + 1) * G)
            rk, rv = A.attention_keys_dkdv(q[:, hs].contiguous(), k[:, g:g + 1].contiguous(),
                                           v[:, g:g + 1].contiguous(), do[:, hs].contiguous(), cu, keys, 0,
                                           True, wl.softmax_scale)
            for name, x, r in (("dk", dk[kidx, g], rk), ("dv", dv[kidx, g], rv)):
                e = np.abs(x.float().cpu().numpy() - r)
                err[name] = max(err[name], float(e.max()))
                excess = max(excess, float((e - (2e-2 + np.abs(r) * 2.0 ** -9)).max()))
        what += "; dK, dV of the last %d keys of document %d, kv heads 0 and %d" % (len(keys), longest,
                                                                                   wl.Hkv - 1)
    else:
        err["dk"] = err["dv"] = None
    return {"max_abs_err": err, "within_bounds": excess <= 0, "sample": what,
            "bounds": "2e-2 + 2^-9 |ref| on the bf16 outputs O, dQ, dK, dV; 1e-3 on LSE",
            "outputs": "the bench's last timed step (bf16 O and gradients)"}


def torch_index(idx):
    import torch
    return torch.tensor(idx, dtype=torch.long)


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from workloads import draw_qkvdo
    q, k, v, do = draw_qkvdo(wl)
    tokens = args.cpu_tokens
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, q, k, v, do, min(tokens, 2048))
    times, flops, sample = [], 0.0, ""
    for _ in range(args.steps):
        flops, dt, sample = cpu_oracle_sample(wl, q, k, v, do, tokens)
        times.append(dt)
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_of(wl):
    return {"workload": wl.name, "T": wl.T, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.d,
            "cp_size": max(wl.cp_per_doc), "layout": wl.layout, "causal": wl.causal,
            "docs": wl.num_docs, "seed": wl.seed,
            "l2": "inputs larger than L2 (q, dO 1 GiB each at 128K), no flush"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_128k")
    ap.add_argument("--layout", default=None, choices=["zigzag", "contiguous"],
                    help="override the workload's shard layout (same inputs)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="a shorter single-document workload of the same shape (profiling small cases)")
    # the first upload and the last download are not overlapped with compute:
    # over 16 steps that pipeline fill is a smaller share of the timed region
    ap.add_argument("--e2e-steps", type=int, default=16)
    # ~12 s of fp64 oracle work per sample on a 16-core host at the 128K shape
    ap.add_argument("--cpu-tokens", type=int, default=40960)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from workloads import workload
    wl = workload(args.workload)
    if args.layout and args.layout != wl.layout:
        wl = dataclasses.replace(wl, layout=args.layout, name="%s_%s" % (wl.name, args.layout))
    if args.tokens:
        if wl.num_docs != 1:
            raise SystemExit("--tokens applies to single-document workloads")
        wl = dataclasses.replace(wl, T=args.tokens, cu_seqlens=(0, args.tokens), name="%s_T%d" % (wl.name, args.tokens))
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist
    import context_ring_attention_step_gb300 as ra
    from workloads import draw_qkvdo

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = ra.load_library()

    q_h, k_h, v_h, do_h = draw_qkvdo(wl)
    cps = list(wl.cp_per_doc)
    t_plan = time.perf_counter()
    plan = ra.Plan(wl.cu_seqlens, cps, wl.layout, wl.causal, wl.Hq, wl.Hkv, wl.d, wl.softmax_scale)
    plan_ms = (time.perf_counter() - t_plan) * 1e3  # host, once per batch layout; not in the timed region
    steps = plan.stats()["steps"]
    q, k, v, do = (x.to(dev) for x in (q_h, k_h, v_h, do_h))
    T, Hq, Hkv, D = wl.T, wl.Hq, wl.Hkv, wl.d
    o = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    dq = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    wf, wb = plan.workspace_bytes(False, False)
    ws_f = torch.empty(wf, dtype=torch.uint8, device=dev)
    ws_b = torch.empty(wb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ra.ring_attn._stream(dev)
    P_ = ra.ring_attn._ptr
    H = plan.handle
    fitems, foff = plan.work_items("fwd")
    bitems, boff = plan.work_items("bwd")
    fpairs = step_pairs_fwd(fitems, foff, wl.causal)
    bpairs = step_pairs_bwd(bitems, boff, wl.causal)
    fwd_launches = sum(1 for s in range(steps) if foff[s + 1] > foff[s])
    bwd_launches = sum(1 for s in range(steps) if boff[s + 1] > boff[s])

    def chk(st):
        if st != 0:
            raise RuntimeError("ring_attn status %d: %s" % (st, lib.ra_last_error().decode()))

    def new_event():
        return torch.cuda.Event(enable_timing=True)

    # One step: the forward (the whole ring in one launch, ra_fwd), then the
    # backward (Delta preprocess, one launch per ring step, gradient casts).
    # Events mark the start of the step, the end of the forward and the span
    # of the backward ring-step launches (an event between two ring-step
    # launches would stop the next one from starting on the SMs the previous
    # one frees, so the backward's launches are bracketed as a whole).
    def one_step(ev=None):
        if ev:
            ev["start"].record(stream)
        chk(lib.ra_fwd(H, P_(q), P_(k), P_(v), P_(o), 0, P_(lse), P_(ws_f), wf, sp))
        if ev:
            ev["fwd"].record(stream)
        chk(lib.ra_bwd_prepare(H, P_(o), 0, P_(do), P_(lse), P_(dq), P_(dk), P_(dv), 0, P_(ws_b), wb, sp))
        if ev:
            ev["bwd0"].record(stream)
        for s in range(steps):
            chk(lib.ra_bwd_ring_step(H, s, P_(q), P_(k), P_(v), P_(do), P_(dq), P_(dk), P_(dv), 0, P_(ws_b), wb,
                                     sp))
        if ev:
            ev["bwd1"].record(stream)
        chk(lib.ra_bwd_finish(H, P_(dq), P_(dk), P_(dv), 0, P_(ws_b), wb, sp))

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    chk(lib.ra_workspace_status(P_(ws_f), sp))
    chk(lib.ra_workspace_status(P_(ws_b), sp))

    # ---------------------------------------------------------------- timed region
    e0, e1 = new_event(), new_event()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [{n: new_event() for n in ("start", "fwd", "bwd0", "bwd1")} for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        e0.record(stream)
        for it in range(args.steps):
            one_step(evs[it])
        e1.record(stream)
        torch.cuda.synchronize()
    ms_total = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    if world > 1:
        dist.barrier()
    chk(lib.ra_workspace_status(P_(ws_f), sp))
    chk(lib.ra_workspace_status(P_(ws_b), sp))
    step_ms = [evs[i]["start"].elapsed_time(evs[i + 1]["start"] if i + 1 < args.steps else e1)
               for i in range(args.steps)]
    t_f = [ev["start"].elapsed_time(ev["fwd"]) for ev in evs]
    t_b = [ev["bwd0"].elapsed_time(ev["bwd1"]) for ev in evs]

    # ---------------------------------------------------------------- ring-step forward
    # The same forward with one launch per ring step and the merge into a
    # running (O, LSE) in HBM (ra_fwd_ring_steps, the per-step unit a
    # multi-GPU driver would interleave with its KV exchanges): timed after the
    # main region, on its own output buffers.
    wrs = plan.ring_step_workspace_bytes(False)
    ws_r = torch.empty(wrs, dtype=torch.uint8, device=dev)
    o_r = torch.empty_like(o)
    lse_r = torch.empty_like(lse)

    def ring_step_fwd(ev=None):
        chk(lib.ra_fwd_prepare(H, 0, P_(ws_r), wrs, sp))
        if ev:
            ev[0].record(stream)
        for s in range(steps):
            chk(lib.ra_fwd_ring_step(H, s, P_(q), P_(k), P_(v), P_(o_r), 0, P_(lse_r), P_(ws_r), wrs, sp))
        if ev:
            ev[1].record(stream)
        chk(lib.ra_fwd_finish(H, P_(o_r), 0, P_(ws_r), wrs, sp))

    for _ in range(max(1, args.warmup)):
        ring_step_fwd()
    torch.cuda.synchronize()
    rev = [(new_event(), new_event()) for _ in range(args.steps)]
    for it in range(args.steps):
        ring_step_fwd(rev[it])
    torch.cuda.synchronize()
    chk(lib.ra_workspace_status(P_(ws_r), sp))
    rs_kernel_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in rev), dist, dev) / args.steps

    # ---------------------------------------------------------------- CTA-pair backward
    # head_dim 128: the same backward on CTA pairs (cta_group::2), timed like
    # the headline's backward over its ring-step launches, on its own buffers.
    pairs_ms = None
    if D == 128:
        plan.set_bwd_cta_pairs(True)
        _, wbp = plan.workspace_bytes(False, False)
        ws_p = torch.empty(wbp, dtype=torch.uint8, device=dev)
        dq_p, dk_p, dv_p = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)

        def pair_bwd(ev=None):
            chk(lib.ra_bwd_prepare(H, P_(o), 0, P_(do), P_(lse), P_(dq_p), P_(dk_p), P_(dv_p), 0, P_(ws_p), wbp, sp))
            if ev:
                ev[0].record(stream)
            for s in range(steps):
                chk(lib.ra_bwd_ring_step(H, s, P_(q), P_(k), P_(v), P_(do), P_(dq_p), P_(dk_p), P_(dv_p), 0,
                                         P_(ws_p), wbp, sp))
            if ev:
                ev[1].record(stream)
            chk(lib.ra_bwd_finish(H, P_(dq_p), P_(dk_p), P_(dv_p), 0, P_(ws_p), wbp, sp))

        for _ in range(max(1, args.warmup)):
            pair_bwd()
        torch.cuda.synchronize()
        pev = [(new_event(), new_event()) for _ in range(args.steps)]
        for it in range(args.steps):
            pair_bwd(pev[it])
        torch.cuda.synchronize()
        chk(lib.ra_workspace_status(P_(ws_p), sp))
        pairs_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in pev), dist, dev) / args.steps
        plan.set_bwd_cta_pairs(False)
        del ws_p, dq_p, dk_p, dv_p

    ff, fb = useful_flops(wl)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(world, ff + fb, args.steps, ms_total)
    peak_b, peak_s, hbm, peak_kind = peaks()
    fwd_ms = sum(t_f) / args.steps
    bwd_ms = sum(t_b) / args.steps
    cta_pairs = None if pairs_ms is None else {
        "bwd_kernels_ms": pairs_ms, "bwd_tflops": fb / (pairs_ms * 1e-3) / 1e12,
        "note": "the backward on CTA pairs (ra_plan_set_bwd_cta_pairs: cta_group::2 over two key tiles), timed "
                "separately over its ring-step launches; not part of value"}
    ring_steps = {"fwd_kernels_ms": rs_kernel_ms, "fwd_tflops": ff / (rs_kernel_ms * 1e-3) / 1e12,
                  "launches": fwd_launches,
                  "note": "forward with one launch per ring step (ra_fwd_ring_steps), timed separately over "
                          "its ring-step launches; not part of value"}

    # roofline of the dominant kernel (events on the launching stream)
    bwd_alg = 10.0 * wl.d * wl.Hq * sum(bpairs) / max(1, bwd_launches)
    bwd_launch_s = sum(t_b) * 1e-3 / (args.steps * max(1, bwd_launches))
    fwd_alg = ff  # the single-launch forward: one launch per step does the whole forward
    fwd_launch_s = sum(t_f) * 1e-3 / args.steps
    kernels = {
        "ring_bwd_step_kernel": (bwd_alg, bwd_launch_s, sum(t_b),
                                 "CUDA events on the launching stream around each step's backward ring-step "
                                 "launches (one kernel per ring step); average = span / launches"),
        "ring_fwd_step_kernel (single launch)": (fwd_alg, fwd_launch_s, sum(t_f),
                                                 "CUDA events on the launching stream around ra_fwd "
                                                 "(work-list set-up kernel + the forward kernel)"),
    }
    roofs = {}
    for name, (alg, launch_s, _, how) in kernels.items():
        achieved = alg / launch_s / 1e12
        roofs[name] = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peak_s,
                       "unit": "TFLOP/s", "frac": achieved / peak_s,
                       "peak_kind": peak_kind + " bf16 sustained (kernel timed inside a long step)",
                       "frac_of_burst_peak": achieved / peak_b,
                       "traffic": recorded_traffic(name.split(" ")[0], wl.name) if name.startswith("ring_bwd")
                       else None,
                       "traffic_unit": "bytes per launch (dram read + write, ncu)",
                       "per_launch_flops": alg, "avg_launch_ms": launch_s * 1e3, "timing": how}
    dominant = max(kernels, key=lambda n: kernels[n][2])
    roof = roofs[dominant]
    roof_other = {n: r for n, r in roofs.items() if n != dominant}

    # ---------------------------------------------------------------- end to end (host buffers)
    # Every step copies its inputs from pinned host memory and its results back
    # (o, lse, dq, dk, dv), through the public Python API.  Uploads and
    # downloads run on two streams of their own (both directions of the host
    # link at once), double-buffered in device inputs and outputs (passed as
    # out=, so nothing is allocated in the timed loop): step i+1's inputs go up
    # while step i computes, and step i's results come down while step i+1
    # computes.  Two untimed steps first (first use of the pinned buffers and
    # the copy streams); the timed region then runs from the first copy to the
    # end of the last one.
    e2e = None
    if args.e2e_steps > 0:
        pin = [x.pin_memory() for x in (q_h, k_h, v_h, do_h)]
        outs_h = [[torch.empty((T, Hq, D), dtype=torch.bfloat16).pin_memory(),
                   torch.empty((Hq, T), dtype=torch.float32).pin_memory(),
                   torch.empty((T, Hq, D), dtype=torch.bfloat16).pin_memory(),
                   torch.empty((T, Hkv, D), dtype=torch.bfloat16).pin_memory(),
                   torch.empty((T, Hkv, D), dtype=torch.bfloat16).pin_memory()] for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in pin)
        d2h = sum(x.numel() * x.element_size() for x in outs_h[0])
        ins = [[torch.empty_like(x, device=dev) for x in pin] for _ in range(2)]
        outs_d = [[torch.empty(x.shape, dtype=x.dtype, device=dev) for x in outs_h[0]] for _ in range(2)]
        up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)  # both link directions at once

        def run_e2e(n_steps):
            """n_steps end-to-end steps; returns their device time (ms) from the
            first upload to the end of the last download."""
            ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of a buffer landed
            ev_used = [torch.cuda.Event() for _ in range(2)]   # compute done with a buffer
            ev_down = [torch.cuda.Event() for _ in range(2)]   # a device output buffer has been copied out
            ev_out = torch.cuda.Event()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            up_stream.wait_stream(stream)
            down_stream.wait_stream(stream)

            def upload(i):
                b = i % 2
                with torch.cuda.stream(up_stream):
                    if i >= 2:
                        up_stream.wait_event(ev_used[b])
                    for dst, src in zip(ins[b], pin):
                        dst.copy_(src, non_blocking=True)
                    ev_in[b].record(up_stream)

            upload(0)
            for i in range(n_steps):
                b = i % 2
                if i + 1 < n_steps:
                    upload(i + 1)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_down[b])
                qd, kd, vd, dod = ins[b]
                oo, ll, gq, gk, gv = outs_d[b]
                ra.ring_attn_fwd(qd, kd, vd, wl.cu_seqlens, cps, wl.layout, wl.causal, wl.softmax_scale,
                                 plan=plan, workspace=ws_f, out=(oo, ll))
                ra.ring_attn_bwd(qd, kd, vd, oo, dod, ll, wl.cu_seqlens, cps, wl.layout, wl.causal,
                                 wl.softmax_scale, plan=plan, workspace=ws_b, out=(gq, gk, gv))
                ev_used[b].record(stream)
                ev_out.record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(ev_out)
                    for dst, src in zip(outs_h[b], outs_d[b]):
                        dst.copy_(src, non_blocking=True)
                    ev_down[b].record(down_stream)
            stream.wait_stream(up_stream)
            stream.wait_stream(down_stream)
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1)

        run_e2e(2)  # untimed: first use of the pinned buffers and copy streams
        e_ms = max_over_ranks(run_e2e(args.e2e_steps), dist, dev)
        e2e = {"value": whole_job_tflops(world, ff + fb, args.e2e_steps, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "ms_per_step": e_ms / args.e2e_steps, "warmup": 2,
               "copies": "pinned host <-> device, uploads and downloads on two streams, double-buffered device inputs and outputs (no allocation in the timed loop), overlapping compute; the first upload and the last download are inside the timed region and not overlapped"}

    # CPU leg (rank 0, one GPU): the oracle timed on a bounded sample, and the
    # bench's own outputs checked against it on sampled rows and keys
    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops, dt, sample = cpu_oracle_sample(wl, q_h, k_h, v_h, do_h, args.cpu_tokens)
        cpu = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": sample, "seconds": dt}
        parity = cpu_parity_sample(wl, q_h, k_h, v_h, do_h, o, lse, dq, dk, dv)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(wl),
            "pct_of_bf16_peak": 100.0 * value / world / peak_b, "pct_of_bf16_peak_sustained":
                100.0 * value / world / peak_s,
            "ms_per_step_median": statistics.median(step_ms), "ms_per_step_mean": statistics.mean(step_ms),
            "ms_per_step_all": step_ms,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "bwd_with_preprocess_and_casts_ms": ms_step - fwd_ms,
            "fwd_tflops": ff / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None,
            "bwd_tflops": fb / (bwd_ms * 1e-3) / 1e12 if bwd_ms else None,
            "useful_flops_per_step": ff + fb, "strict_bwd_flops_per_step": 0.8 * fb,
            "roofline": roof, "roofline_other_kernels": roof_other, "cpu_baseline": cpu,
            "parity_vs_oracle": parity, "e2e": e2e, "ring_step_forward": ring_steps, "bwd_cta_pairs": cta_pairs,
            # per step: the forward's work-list set-up and forward kernel, the
            # backward's work-list set-up and Delta preprocess, its ring steps
            # and the three gradient casts (a plan without pinned work lists
            # copies its work lists instead of running the set-up kernels)
            "gpu_launches": args.steps * (2 + 2 + bwd_launches + 3),
            "plan_ms": plan_ms,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
