"""Decode context parallelism on CPU: the host-side sharding (which tokens a rank
holds, its local block table) and the exchange layout, with the oracle standing
in for each rank's shard computation.  Two gloo ranks (world_size 2) all-gather
their partials through the same function the GPU path uses, and the merged
result must equal the single-pass oracle.  No GPU is used.
"""
import os
import queue
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from mla_paged_kv_02_gb300 import dcp, synth


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_shard_bounds_tile_every_request_on_page_boundaries(world):
    lens = [1, 63, 64, 65, 200, 641, 4096, 3]
    per_rank = [dcp.shard_bounds(lens, world, r) for r in range(world)]
    for b, L in enumerate(lens):
        pos = 0
        for r in range(world):
            s, e = per_rank[r][b]
            assert s == pos and s <= e <= L
            assert s % 64 == 0 or s == L
            pos = e
        assert pos == L
        # page counts differ by at most one between ranks
        n = [-(-(per_rank[r][b][1] - per_rank[r][b][0]) // 64) for r in range(world)]
        assert max(n) - min(n) <= 1


def test_local_block_table_maps_local_tokens_to_their_global_pages():
    inp = synth.make_inputs("tiny", seed=31, kv_lens=[5, 130, 640, 1000], batch=4, num_heads=4)
    lens = [int(x) for x in inp.seq_lens]
    for world in (2, 3):
        for r in range(world):
            bounds = dcp.shard_bounds(lens, world, r)
            lbt = dcp.local_block_table(inp.block_table, bounds)
            for b, (s, e) in enumerate(bounds):
                for t in range(e - s):
                    g = s + t
                    assert int(lbt[b, t // 64]) == int(inp.block_table[b, g // 64])
                    assert g % 64 == t % 64
                n = -(-(e - s) // 64)
                assert bool((lbt[b, n:] == -1).all())


def test_single_rank_gather_is_the_partial_itself():
    p = torch.randn(2, 1, 3, 513)
    g = dcp.gather_partials(p)
    assert g.shape == (1, 2, 1, 3, 513) and torch.equal(g[0], p)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import oracle as orc
    from mla_paged_kv_02_gb300 import dcp as d
    from mla_paged_kv_02_gb300 import synth as sy

    try:
        dist.init_process_group("gloo")
        inp = sy.make_inputs("tiny", seed=32, kv_lens=[4, 70, 300, 129, 64], q_len=4, batch=5, num_heads=4,
                             sharp=3.0)
        lens = [int(x) for x in inp.seq_lens]
        bounds = d.shard_bounds(lens, world, rank)
        part = orc.decode_range(inp, [s for s, _ in bounds], [e for _, e in bounds], threads=1)
        gathered = d.gather_partials(torch.from_numpy(part))
        assert gathered.shape == (world,) + part.shape
        # shard-major: slot r holds rank r's partial
        assert torch.equal(gathered[rank], torch.from_numpy(part))
        if rank == 0:
            out, lse = orc.lse_merge(gathered.numpy())
            ref_o, ref_l = orc.decode(inp, threads=1)
            assert np.max(np.abs(out - ref_o)) <= 1e-12
            assert np.max(np.abs(lse - ref_l)) <= 1e-12
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e)))


def test_two_gloo_ranks_gather_and_merge_shard_partials():
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
            except queue.Empty:
                break
            results[rank] = msg
    finally:
        for p in procs:
            if p.is_alive():
                p.kill()
    assert results == {0: "ok", 1: "ok"}, results


def test_shard_partials_of_every_rank_merge_to_the_single_pass():
    # The same bookkeeping for three ranks evaluated in one process.
    inp = synth.make_inputs("tiny", seed=33, kv_lens=[8, 64, 65, 700], q_len=8, batch=4, num_heads=2)
    lens = [int(x) for x in inp.seq_lens]
    parts = []
    for r in range(3):
        bounds = dcp.shard_bounds(lens, 3, r)
        parts.append(oracle.decode_range(inp, [s for s, _ in bounds], [e for _, e in bounds]))
    out, lse = oracle.lse_merge(np.stack(parts))
    ref_o, ref_l = oracle.decode(inp)
    assert np.max(np.abs(out - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12
