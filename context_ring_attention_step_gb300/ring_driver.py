"""Multi-GPU ring: the per-rank ring-step calls interleaved with the key/value
exchange between ring neighbours.

One process per GPU; rank r of a ring of cp ranks keeps query shard r of
every document (Accelerate guide, "Detalhes tecnicos": Q, K, V sharded along
the sequence) and, at ring step s, holds key/value shard (r - s) mod cp: every
step it passes the shard it holds to rank r + 1 and receives the next one from
rank r - 1, while it computes attention against the one it holds
(NVSHMEM/XLA page, "Patrones de comunicacion en la atencion en anillo":
compute on the current KV block while the next one is fetched, point-to-point
sends between ring neighbours).

Schedule, for step s = 0 .. cp-1 (j = (r - s) mod cp):
  forward   post send(K_j, V_j -> r+1) and recv(K_{j-1}, V_{j-1} <- r-1)
            [not at the last step]; run step s (queries of shard r against
            K_j, V_j, merged into the running O, LSE of shard r); wait.
  backward  the same key/value rotation.  dQ stays with its query shard.
            The partial dK_j, dV_j travel with K_j, V_j: before step s the
            rank waits for the partial of shard j from r-1 (which added its
            contribution at step s-1), adds its own contribution in step s,
            then sends it on to r+1 and posts the receive of shard j-1's
            partial.  After cp steps every shard's accumulator has visited
            every rank and is back with its owner, complete.

Buffers keep the global THD layout [T, H, d]: a rank's q, o, dout and dq
hold valid rows of its own shard only, its k, v (and dk, dv) the rows of the
shards it has received so far.  Every other row must hold finite values
(zeros, say): 128-row tiles overhang the edges of a shard's ranges, and
although the overhanging rows are masked (probability 0), 0 times a NaN or
an infinity is not 0.  Every transfer is a contiguous row range (one
per chunk of a shard per document) copied into the receiving rank's own
memory: no kernel reads another GPU's memory.  The ring needs one ring size
for every document, equal to the number of ranks.

`AllGatherDriver` is the other variant the Accelerate guide describes ("all-to-all
vs all-gather"): all key/value shards gathered once up front, the steps run
without exchange, and the dK/dV partials summed onto their owners at the end.

The exchange uses torch.distributed point-to-point calls (NCCL between GPUs,
gloo on CPU for the tests); the compute of each step is an object with
fwd_begin / fwd_step(s) / fwd_end and bwd_begin / bwd_step(s) / bwd_end.
`RankCompute` is the library's: it calls ra_fwd_ring_step_rank /
ra_bwd_ring_step_rank, so each step is one kernel launch of this rank's work
items.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import ring_attn as _ra


class RingDriver:
    """The ring schedule of one rank (see the module docstring)."""

    def __init__(self, plan, rank, world, group=None):
        if not 0 <= rank < world:
            raise ValueError("rank %d outside [0, %d)" % (rank, world))
        cps = list(plan.cp_per_doc)
        if any(c != world for c in cps):
            raise ValueError("the ring needs cp_size == number of ranks (%d) for every document, got %s"
                             % (world, sorted(set(cps))))
        self.plan, self.rank, self.world, self.group = plan, rank, world, group
        self.next, self.prev = (rank + 1) % world, (rank - 1) % world
        # global row ranges of every shard (one per chunk per document), empty ones dropped
        self.ranges = {j: [(b, e) for d in range(plan.num_docs) for b, e in plan.shard_token_ranges(d, j)
                           if e > b] for j in range(world)}

    def source(self, s):
        """Key/value shard this rank holds at ring step s."""
        return (self.rank - s) % self.world

    def _post(self, tensors, shard, send, tag):
        ops = []
        for ti, t in enumerate(tensors):
            for ri, (b, e) in enumerate(self.ranges[shard]):
                tg = (tag * len(tensors) + ti) * 1024 + ri % 1024
                if send:
                    ops.append(dist.isend(t[b:e], self.next, group=self.group, tag=tg))
                else:
                    ops.append(dist.irecv(t[b:e], self.prev, group=self.group, tag=tg))
        return ops

    @staticmethod
    def _wait(ops):
        for w in ops:
            w.wait()

    def forward(self, compute, k, v):
        """Run the forward ring.  k, v: this rank's full-length buffers holding
        its own shard's rows; the other shards' rows are filled as they arrive."""
        compute.fwd_begin()
        for s in range(self.world):
            j = self.source(s)
            kv = []
            if s + 1 < self.world:
                kv = self._post((k, v), j, True, 2 * s) + self._post((k, v), self.source(s + 1), False, 2 * s)
            compute.fwd_step(s)
            self._wait(kv)
        compute.fwd_end()

    def backward(self, compute, k, v, dk, dv):
        """Run the backward ring.  dk, dv: this rank's fp32 accumulators,
        zeroed by compute.bwd_begin(); on return the rows of the rank's own
        shard hold the complete gradients."""
        compute.bwd_begin()
        acc = []
        for s in range(self.world):
            j = self.source(s)
            kv = []
            if s + 1 < self.world:
                kv = self._post((k, v), j, True, 4 * s) + self._post((k, v), self.source(s + 1), False, 4 * s)
            self._wait(acc)  # the partial dK_j, dV_j from rank r-1 has landed (s > 0)
            compute.bwd_step(s)
            if self.world > 1:
                # pass the partial on; the last one goes back to its owner, r+1
                acc = self._post((dk, dv), j, True, 4 * s + 2) + \
                    self._post((dk, dv), self.source(s + 1), False, 4 * s + 2)
            self._wait(kv)
        self._wait(acc)  # this rank's own shard, complete
        compute.bwd_end()


class AllGatherDriver(RingDriver):
    """The all-gather variant of the same schedule (Accelerate guide,
    "all-to-all vs all-gather"): every rank gathers every key/value shard once,
    before its first step, and then runs its cp ring steps with no exchange in
    between; in the backward each key/value shard's partial dK, dV are summed
    onto the shard's owner after the last step (one reduction per shard).  It
    hides no transfer behind compute and holds all of K and V on every rank,
    against the ring's one shard in flight; it needs no step-by-step
    choreography.  Same compute interface, same results as RingDriver."""

    def _sizes(self):
        return [sum(e - b for b, e in self.ranges[j]) for j in range(self.world)]

    def _pack(self, t, shard):
        """The rows of `shard` (all its ranges, in order) as one contiguous copy."""
        rows = [t[b:e] for b, e in self.ranges[shard]]
        return torch.cat(rows) if rows else t[:0].clone()

    def _unpack(self, t, shard, buf):
        o = 0
        for b, e in self.ranges[shard]:
            t[b:e].copy_(buf[o:o + e - b])
            o += e - b

    def gather(self, tensors):
        """Every shard's rows of each tensor onto every rank: one all_gather
        per tensor of the packed shard rows, padded to the largest shard."""
        n = self._sizes()
        m = max(n)
        for t in tensors:
            mine = t.new_zeros((m,) + tuple(t.shape[1:]))
            mine[:n[self.rank]] = self._pack(t, self.rank)
            parts = [t.new_empty((m,) + tuple(t.shape[1:])) for _ in range(self.world)]
            dist.all_gather(parts, mine, group=self.group)
            for j in range(self.world):
                if j != self.rank:
                    self._unpack(t, j, parts[j][:n[j]])

    def forward(self, compute, k, v):
        """Run the forward: gather K, V, then every ring step locally."""
        self.gather((k, v))
        compute.fwd_begin()
        for s in range(self.world):
            compute.fwd_step(s)
        compute.fwd_end()

    def backward(self, compute, k, v, dk, dv):
        """Run the backward: gather K, V, every ring step locally (the partial
        dK, dV of every shard accumulate in this rank's full-length dk, dv),
        then sum each shard's partials onto its owner."""
        self.gather((k, v))
        compute.bwd_begin()
        for s in range(self.world):
            compute.bwd_step(s)
        for t in (dk, dv):
            for j in range(self.world):
                part = self._pack(t, j)
                dist.reduce(part, dst=j, group=self.group)
                if j == self.rank:
                    self._unpack(t, j, part)
        compute.bwd_end()


DRIVERS = {"ring": RingDriver, "allgather": AllGatherDriver}


class RankCompute:
    """One rank's ring steps through the library's per-rank calls: every step
    is one kernel launch over the work items of query shard `rank`.  Outputs:
    o (bf16, or fp32 with o_fp32) and lse after the forward; fp32 dq, dk, dv
    (the accumulators the backward's partials travel in) after the backward."""

    def __init__(self, plan, rank, q, k, v, o_fp32=False):
        self.lib = _ra.load_library()
        self.plan, self.rank = plan, rank
        self.q, self.k, self.v = q, k, v
        T, Hq, D = q.shape
        Hkv = k.shape[1]
        dev = q.device
        self.o_fp32 = bool(o_fp32)
        # zeros: rows of other shards stay finite (the backward's Delta reads
        # every row of o, and tiles overhang the shard's ranges)
        self.o = torch.zeros((T, Hq, D), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=dev)
        self.lse = torch.zeros((Hq, T), dtype=torch.float32, device=dev)
        self.dq = torch.empty((T, Hq, D), dtype=torch.float32, device=dev)
        self.dk = torch.empty((T, Hkv, D), dtype=torch.float32, device=dev)
        self.dv = torch.empty((T, Hkv, D), dtype=torch.float32, device=dev)
        self.wf = plan.ring_step_workspace_bytes(o_fp32)
        self.wb = plan.workspace_bytes(o_fp32, True)[1]
        self.ws_f = torch.zeros(self.wf, dtype=torch.uint8, device=dev)  # its fp32 running output too
        self.ws_b = torch.empty(self.wb, dtype=torch.uint8, device=dev)
        self.do = None

    def _s(self):
        return _ra._stream(self.q.device)

    def fwd_begin(self):
        _ra._check(self.lib.ra_fwd_prepare(self.plan.handle, int(self.o_fp32), _ra._ptr(self.ws_f), self.wf,
                                           self._s()))

    def fwd_step(self, s):
        p = _ra._ptr
        _ra._check(self.lib.ra_fwd_ring_step_rank(self.plan.handle, s, self.rank, p(self.q), p(self.k), p(self.v),
                                                  p(self.o), int(self.o_fp32), p(self.lse), p(self.ws_f), self.wf,
                                                  self._s()))

    def fwd_end(self):
        _ra._check(self.lib.ra_fwd_finish(self.plan.handle, _ra._ptr(self.o), int(self.o_fp32), _ra._ptr(self.ws_f),
                                          self.wf, self._s()))

    def bwd_begin(self):
        p = _ra._ptr
        _ra._check(self.lib.ra_bwd_prepare(self.plan.handle, p(self.o), int(self.o.dtype == torch.float32),
                                           p(self.do), p(self.lse), p(self.dq), p(self.dk), p(self.dv), 1,
                                           p(self.ws_b), self.wb, self._s()))

    def bwd_step(self, s):
        p = _ra._ptr
        _ra._check(self.lib.ra_bwd_ring_step_rank(self.plan.handle, s, self.rank, p(self.q), p(self.k), p(self.v),
                                                  p(self.do), p(self.dq), p(self.dk), p(self.dv), 1, p(self.ws_b),
                                                  self.wb, self._s()))

    def bwd_end(self):
        pass  # the gradients are the fp32 accumulators


def ring_attn_fwd_rank(q, k, v, plan, rank, world, group=None, o_fp32=False, check=False, variant="ring"):
    """Forward of one rank of a multi-GPU ring: returns (o, lse, compute),
    with the rows of shard `rank` valid in o and lse.  q, k, v: full-length
    [T, H, d] bf16 buffers on this rank's GPU holding its own shard's rows and
    finite values (zeros) elsewhere (k and v receive the other shards' rows).
    variant: "ring" (neighbour exchange overlapped with each step) or
    "allgather" (all shards gathered first).  Keep `compute` for the backward."""
    comp = RankCompute(plan, rank, q, k, v, o_fp32)
    DRIVERS[variant](plan, rank, world, group).forward(comp, k, v)
    if check:
        _ra._check(_ra.workspace_status(comp.ws_f))
    return comp.o, comp.lse, comp


def ring_attn_bwd_rank(compute, do, plan, rank, world, group=None, check=False, variant="ring"):
    """Backward of one rank after ring_attn_fwd_rank: returns fp32 (dq, dk, dv)
    with the rows of shard `rank` complete.  do: full-length [T, Hq, d] bf16
    with this rank's rows and finite values (zeros) elsewhere."""
    compute.do = do
    DRIVERS[variant](plan, rank, world, group).backward(compute, compute.k, compute.v, compute.dk, compute.dv)
    if check:
        _ra._check(_ra.workspace_status(compute.ws_b))
    return compute.dq, compute.dk, compute.dv
