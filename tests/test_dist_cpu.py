"""The benchmark's multi-rank logic on CPU (gloo, world size 2).

The forward step shards without exchange: each rank appends and runs its own
sessions.  These tests check that the session shards partition the sessions,
that windows built rank by rank equal the windows of a single process, and
that the timing reductions (barrier, max and sum over ranks) work.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import torch
    import torch.distributed as dist_mod

    import bench
    import engram_gram_conditional_gb300 as eg
    import synth

    d = bench.Dist()
    assert d.world == world and d.rank == rank and dist_mod.get_backend() == "gloo"
    w = synth.WORKLOADS["tiny"]
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    ctx = eg.engram_ctx_create(w.vocab, w.vc, tmap, w.hash_seeds, w.bucket_bases, heads=w.heads,
                               row_dim=w.row_dim, hc=w.hc, d=w.d)
    mine = bench.shard_sessions(7, rank, world)
    wins = {}
    for sid in mine:
        s = eg.engram_session_create(ctx)
        wins[sid] = eg.engram_session_append(s, synth.session_tokens(w, sid, 33))
        eg.engram_session_destroy(s)
    d.barrier()
    total = d.sum(float(len(mine)))
    slowest = d.max(float(rank + 1))
    gathered = [None] * world
    dist_mod.all_gather_object(gathered, {k: v.tolist() for k, v in wins.items()})
    queue.put((rank, mine, total, slowest, gathered))
    eg.engram_ctx_destroy(ctx)
    d.close()


def test_replica_sharding_and_timing_reductions():
    from engram_gram_conditional_gb300 import build

    build.build()
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    shards = [r[1] for r in results]
    assert sorted(sum(shards, [])) == list(range(7))          # a partition
    assert not set(shards[0]) & set(shards[1])
    for _, _, total, slowest, _ in results:
        assert total == 7.0 and slowest == 2.0
    # windows built rank by rank equal a single process's windows
    import engram_gram_conditional_gb300 as eg
    import synth

    w = synth.WORKLOADS["tiny"]
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    c = eg.engram_ctx_create(w.vocab, w.vc, tmap, w.hash_seeds, w.bucket_bases, heads=w.heads,
                             row_dim=w.row_dim, hc=w.hc, d=w.d)
    merged = {}
    for part in results[0][4]:
        merged.update({int(k): v for k, v in part.items()})
    for sid in range(7):
        s = eg.engram_session_create(c)
        ref = eg.engram_session_append(s, synth.session_tokens(w, sid, 33))
        assert np.array_equal(np.array(merged[sid], np.uint32), ref)
    eg.engram_ctx_destroy(c)


def test_shard_sessions_is_balanced():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    for n in (1, 7, 256, 1000):
        for world in (1, 2, 3, 8):
            parts = [bench.shard_sessions(n, r, world) for r in range(world)]
            assert sorted(sum(parts, [])) == list(range(n))
            sizes = [len(p) for p in parts]
            assert max(sizes) - min(sizes) <= 1
