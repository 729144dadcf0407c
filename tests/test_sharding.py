"""Sharding by prompt group across 2 ranks (gloo, CPU): per-rank loss partials
with the global normaliser sum to the whole batch's loss, and each rank's
gradient rows equal the whole batch's rows.  Uses the float64 oracle."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from vocab_wide_logprob_gb300 import sharding
from vocab_wide_logprob_gb300 import workloads as wl


def test_group_ranges_cover_the_batch():
    for B in (1, 2, 7, 8):
        for world in (1, 2, 3, 4):
            rs = [sharding.group_range(B, world, r) for r in range(world)]
            assert [g for r in rs for g in r] == list(range(B))
            assert max(len(r) for r in rs) - min(len(r) for r in rs) <= 1
    with pytest.raises(ValueError):
        sharding.group_range(4, 2, 2)


def _whole(w):
    import oracle
    ids = wl.make_ids(w)
    R = wl.make_rewards(w)
    z, dt = wl.logits_as_numpy(wl.make_logits_cpu(w))
    m, lens = oracle.mask(ids, w.P, w.C, w.eos_id)
    A = oracle.advantage(R, w.G)
    lp, lse = oracle.logp(z, dt, w.P, w.C, ids, lens)
    n_old, n_ref = wl.make_noise(w)
    old, ref = lp + n_old, lp + n_ref
    return ids, R, z, dt, old, ref


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        w = wl.variant(wl.TINY, B=4, G=4, old_sigma=0.1, ref_sigma=0.1, beta=0.04, seed=123)
        ids, R, z, dt, old, ref = _whole(w)
        sl = sharding.completion_slice(w.B, w.G, world, rank)
        norm = sharding.global_norm(w.B, w.G, w.C)
        _, lens = oracle.mask(ids[sl], w.P, w.C, w.eos_id)
        A = oracle.advantage(R[sl], w.G)
        lp, lse = oracle.logp(z[sl], dt, w.P, w.C, ids[sl], lens)
        loss, wt, _ = oracle.loss(lp, old[sl], ref[sl], A, lens, w.eps, w.beta, norm)
        d = oracle.dlogits(z[sl], dt, w.P, w.C, ids[sl], lens, lse, wt)
        t = torch.tensor([loss], dtype=torch.float64)
        dist.all_reduce(t)
        q.put((rank, float(t.item()), sl.start, sl.stop, d))
    finally:
        dist.destroy_process_group()


def test_two_rank_partials_add_up():
    import oracle
    w = wl.variant(wl.TINY, B=4, G=4, old_sigma=0.1, ref_sigma=0.1, beta=0.04, seed=123)
    ids, R, z, dt, old, ref = _whole(w)
    _, lens = oracle.mask(ids, w.P, w.C, w.eos_id)
    A = oracle.advantage(R, w.G)
    lp, lse = oracle.logp(z, dt, w.P, w.C, ids, lens)
    loss, wt, _ = oracle.loss(lp, old, ref, A, lens, w.eps, w.beta)
    d = oracle.dlogits(z, dt, w.P, w.C, ids, lens, lse, wt)

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, a, b, d_rank in got:
        assert abs(total - loss) <= 1e-12 * max(1.0, abs(loss)), (total, loss)
        assert np.array_equal(d_rank, d[a:b])


def _agg_rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        out = bench.rank_aggregate(dist, torch.device("cpu"), 0.5 + rank, 100 * (rank + 1),
                                   rank)
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_bench_rank_aggregate_two_ranks():
    """bench.py's whole-job figures over 2 gloo ranks: the slowest rank's time,
    the sum of scored tokens and of contrasted groups."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_agg_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r] == (1.5, 300, 1)


def _fits_rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["LOCAL_WORLD_SIZE"] = str(world)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import types

        import bench
        # rank 1's host reports too little memory for both ranks' pinned buffers
        bench.host_mem_available = lambda: (1 << 40) if rank == 0 else (1 << 10)
        b = types.SimpleNamespace(logits=torch.zeros((4, 1024), dtype=torch.bfloat16))
        q.put((rank, bench.e2e_fits(b, world, dist)))
    finally:
        dist.destroy_process_group()


def test_bench_e2e_skip_agrees_over_ranks():
    """The end-to-end leg has collectives inside, so when one rank's host
    cannot pin the buffers every rank skips it, with the reason."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + os.getpid() % 1000
    procs = [ctx.Process(target=_fits_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        ok, why = res[r]
        assert ok is False and "would pin" in why and "1.02e-06 GB available" in why
