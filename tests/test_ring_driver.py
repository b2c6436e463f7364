"""The multi-GPU ring schedules (ring_driver.RingDriver, and its all-gather
variant AllGatherDriver) on CPU: gloo ranks,
world size 2 and 4, each rank computing its ring steps with the fp64 oracle's
per-shard-pair partials (oracle/ring.py) on its own full-length buffers.

Rows a rank has not received are NaN, so a step that reads a key/value shard
before it arrived (or the wrong one) poisons the result; the gradients of a
shard must travel the whole ring and come back to their owner complete.  The
assembled O, LSE, dQ, dK, dV of all ranks must equal the monolithic oracle
(NVSHMEM/XLA page, "Paralelismo de contexto y atencion en anillo": the ring
keeps mathematical equivalence with standard attention).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class _OracleCompute:
    """Ring steps of one rank in fp64 with the oracle's partial attention and merge."""

    def __init__(self, drv, plan, q, k, v, do, causal, scale):
        self.drv, self.plan = drv, plan
        self.q, self.k, self.v, self.do = q, k, v, do   # k, v: the rank's torch buffers (exchanged)
        self.causal, self.scale = causal, scale
        T, Hq, d = q.shape
        self.G = Hq // k.shape[1]
        self.o = np.zeros((T, Hq, d))
        self.lse = np.full((Hq, T), -np.inf)
        self.dq = np.zeros((T, Hq, d))
        self.dk = torch.zeros(k.shape, dtype=torch.float64)
        self.dv = torch.zeros(v.shape, dtype=torch.float64)

    def _pairs(self, s):
        """(query positions, key positions) per document at step s."""
        from oracle import ring as R
        r, j = self.drv.rank, self.drv.source(s)
        for d in range(self.plan.num_docs):
            qpos = R._positions(self.plan.shard_token_ranges(d, r), 0)
            kpos = R._positions(self.plan.shard_token_ranges(d, j), 0)
            if len(qpos) and len(kpos):
                yield qpos, kpos

    def fwd_begin(self):
        self.o[:] = 0.0
        self.lse[:] = -np.inf

    def fwd_step(self, s):
        from oracle import ring as R
        k, v = self.k.numpy(), self.v.numpy()
        for qpos, kpos in self._pairs(s):
            for h in range(self.q.shape[1]):
                g = h // self.G
                po, pl = R.partial_attention(self.q[qpos, h], k[kpos, g], v[kpos, g], qpos, kpos, self.causal,
                                             self.scale)
                self.o[qpos, h], self.lse[h, qpos] = R.merge(self.o[qpos, h], self.lse[h, qpos], po, pl)

    def fwd_end(self):
        pass

    def bwd_begin(self):
        self.dq[:] = 0.0
        self.dk.zero_()
        self.dv.zero_()

    def bwd_step(self, s):
        k, v, dk, dv = self.k.numpy(), self.v.numpy(), self.dk.numpy(), self.dv.numpy()
        for qpos, kpos in self._pairs(s):
            for h in range(self.q.shape[1]):
                g = h // self.G
                sc = self.scale * (self.q[qpos, h] @ k[kpos, g].T)
                if self.causal:
                    sc = np.where(kpos[None, :] <= qpos[:, None], sc, -np.inf)
                p = np.exp(sc - self.lse[h, qpos][:, None])
                delta = (self.do[qpos, h] * self.o[qpos, h]).sum(axis=1)
                ds = p * (self.do[qpos, h] @ v[kpos, g].T - delta[:, None])
                self.dq[qpos, h] += self.scale * (ds @ k[kpos, g])
                dk[kpos, g] += self.scale * (ds.T @ self.q[qpos, h])
                dv[kpos, g] += p.T @ self.do[qpos, h]

    def bwd_end(self):
        pass


def _worker(rank, world, port, case, out, kind="ring"):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import datetime
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        import context_ring_attention_step_gb300 as ra
        from context_ring_attention_step_gb300.ring_driver import DRIVERS, RingDriver
        from workloads import custom, draw_qkvdo
        lengths, Hq, Hkv, d, layout, causal, planted = case
        if planted and kind == "ring":  # a ring turning the wrong way must be caught
            RingDriver.source = lambda self, s: (self.rank + s) % self.world
        if planted and kind == "allgather":  # gradients left unsummed must be caught
            from context_ring_attention_step_gb300.ring_driver import AllGatherDriver

            def no_reduce(self, c, kk, vv, dk, dv):
                self.gather((kk, vv))
                c.bwd_begin()
                for st in range(self.world):
                    c.bwd_step(st)
                c.bwd_end()
            AllGatherDriver.backward = no_reduce
        wl = custom(lengths, Hq, Hkv, d, world, layout, causal, seed=71)
        q, k, v, do = (x.double().numpy() for x in draw_qkvdo(wl))
        plan = ra.Plan(wl.cu_seqlens, [world] * wl.num_docs, layout, causal, Hq, Hkv, d)
        drv = DRIVERS[kind](plan, rank, world)
        own = np.concatenate([np.arange(b, e) for b, e in drv.ranges[rank]]).astype(np.int64) \
            if drv.ranges[rank] else np.zeros(0, np.int64)
        # this rank's buffers: its own shard's rows, NaN elsewhere until they arrive
        k_loc = torch.full(k.shape, float("nan"), dtype=torch.float64)
        v_loc = torch.full(v.shape, float("nan"), dtype=torch.float64)
        k_loc[own] = torch.from_numpy(k[own])
        v_loc[own] = torch.from_numpy(v[own])
        q_loc = np.full(q.shape, np.nan)
        do_loc = np.full(do.shape, np.nan)
        q_loc[own], do_loc[own] = q[own], do[own]
        comp = _OracleCompute(drv, plan, q_loc, k_loc, v_loc, do_loc, causal, wl.softmax_scale)
        drv.forward(comp, k_loc, v_loc)
        drv.backward(comp, k_loc, v_loc, comp.dk, comp.dv)
        out[rank] = (own, comp.o[own], comp.lse[:, own], comp.dq[own], comp.dk.numpy()[own], comp.dv.numpy()[own])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, case, kind="ring"):
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), case, out, kind), nprocs=world, join=True)
    return dict(out)


CASES = [
    (2, ([300], 4, 2, 64, "zigzag", True)),
    (4, ([200, 37, 5, 130], 4, 2, 64, "zigzag", True)),
    (4, ([97, 160], 2, 1, 64, "contiguous", False)),
]


@pytest.mark.parametrize("kind", ["ring", "allgather"])
@pytest.mark.parametrize("world,case", CASES)
def test_ring_driver_matches_oracle(world, case, kind):
    """Both schedules: the neighbour ring and the all-gather variant."""
    from oracle import attention as A
    from workloads import custom, draw_qkvdo
    lengths, Hq, Hkv, d, layout, causal = case
    res = _run(world, case + (False,), kind)
    wl = custom(lengths, Hq, Hkv, d, world, layout, causal, seed=71)
    q, k, v, do = draw_qkvdo(wl)
    rdq, rdk, rdv, ro, rl = A.attention_bwd(q, k, v, do, wl.cu_seqlens, causal, wl.softmax_scale)
    seen = np.zeros(wl.T, bool)
    for rank in range(world):
        own, o, lse, dq, dk, dv = res[rank]
        assert not seen[own].any()
        seen[own] = True
        assert np.abs(o - ro[own]).max() < 1e-12
        assert np.abs(lse - rl[:, own]).max() < 1e-12
        assert np.abs(dq - rdq[own]).max() < 1e-12
        assert np.abs(dk - rdk[own]).max() < 1e-12
        assert np.abs(dv - rdv[own]).max() < 1e-12
    assert seen.all()  # the shards partition the tokens


def test_ring_driver_catches_a_ring_turning_the_wrong_way():
    """Receiving from the wrong neighbour's shard either breaks the exchange
    (mismatched transfers end the ranks with an error) or poisons the outputs."""
    world, case = CASES[1]
    try:
        res = _run(world, case + (True,))
    except (mp.ProcessRaisedException, mp.ProcessExitedException):
        return
    from oracle import attention as A
    from workloads import custom, draw_qkvdo
    lengths, Hq, Hkv, d, layout, causal = case
    wl = custom(lengths, Hq, Hkv, d, world, layout, causal, seed=71)
    q, k, v, do = draw_qkvdo(wl)
    _, _, _, ro, _ = A.attention_bwd(q, k, v, do, wl.cu_seqlens, causal, wl.softmax_scale)
    bad = [not (np.isfinite(res[r][1]).all() and np.abs(res[r][1] - ro[res[r][0]]).max() < 1e-12)
           for r in range(world)]
    assert any(bad)


def test_ring_driver_requires_cp_equal_to_world():
    import context_ring_attention_step_gb300 as ra
    from context_ring_attention_step_gb300.ring_driver import RingDriver
    plan = ra.Plan([0, 100, 300], [2, 4], "zigzag", True, 2, 1, 64)
    with pytest.raises(ValueError):
        RingDriver(plan, 0, 4)
    with pytest.raises(ValueError):
        RingDriver(ra.Plan([0, 100], 4, "zigzag", True, 2, 1, 64), 4, 4)


def test_allgather_driver_catches_unsummed_gradients():
    """Without the per-shard reduction each owner keeps only its own query
    shard's contribution to dK, dV: the comparison must fail."""
    world, case = CASES[1]
    res = _run(world, case + (True,), "allgather")
    from oracle import attention as A
    from workloads import custom, draw_qkvdo
    lengths, Hq, Hkv, d, layout, causal = case
    wl = custom(lengths, Hq, Hkv, d, world, layout, causal, seed=71)
    q, k, v, do = draw_qkvdo(wl)
    _, rdk, _, _, _ = A.attention_bwd(q, k, v, do, wl.cu_seqlens, causal, wl.softmax_scale)
    bad = [np.abs(res[r][4] - rdk[res[r][0]]).max() > 1e-9 for r in range(world)]
    assert any(bad)
