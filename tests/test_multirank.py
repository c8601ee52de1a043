"""The multi-rank path on CPU: two gloo ranks (world_size 2).

The decode shards by request: rows and pages of different requests are
independent, so ranks need no exchange on the data path.  These tests run the
benchmark's rank plumbing (rendezvous, per-rank seeds, barrier, max over ranks)
under gloo, and check that evaluating disjoint request shards on two ranks and
gathering the results reproduces the single-process answer exactly.
"""
import os
import queue
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    # The CPU path under test: no GPU for the ranks even on a machine that has
    # one (two ranks on one GPU would also be refused by NCCL).
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    from mla_paged_kv_02_gb300 import synth

    try:
        w, r, _ = bench.dist_setup(None)
        assert (w, r) == (world, rank)
        assert dist.get_backend() == "gloo"
        # per-rank seeds differ (weak scaling: every rank has its own batch)
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(2, rank))
        assert len(set(seeds)) == world
        # max over ranks
        bench.barrier(world)
        assert bench.max_over_ranks(world, float(rank + 1)) == float(world)
        # request sharding: disjoint shards, gathered, equal the single-process result
        inp = synth.make_inputs("tiny", seed=3, kv_lens=[3, 70, 129, 200, 5], q_len=2, batch=5,
                                num_heads=4)
        mine = [b for b in range(inp.batch) if b % world == rank]
        out, lse = oracle.decode(synth.subset(inp, mine), threads=1)
        parts = [None] * world
        dist.all_gather_object(parts, (mine, out, lse))
        if rank == 0:
            full_o, full_l = oracle.decode(inp, threads=1)
            got_o = np.zeros_like(full_o)
            got_l = np.zeros_like(full_l)
            for reqs, o, l in parts:
                for k, b in enumerate(reqs):
                    got_o[b], got_l[b] = o[k], l[k]
            np.testing.assert_array_equal(got_o, full_o)
            np.testing.assert_array_equal(got_l, full_l)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e)))


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    try:
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=240)
        results = {}
        for _ in range(world):
            try:
                rank, msg = q.get(timeout=5)
            except queue.Empty:  # a rank that never reported is a failure below
                break
            results[rank] = msg
    finally:
        for p in procs:
            if p.is_alive():
                p.kill()
    assert results == {0: "ok", 1: "ok"}, results
