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


# --------------------------------------------------------------------------
# A table sharded by bucket, rows exchanged by all-to-all (vLLM "Engram" wiki,
# section "데이터 병렬 토폴로지"): the routing on CPU ranks over gloo
# --------------------------------------------------------------------------
def _exchange_rank(rank, world, port, queue):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import torch
    import torch.distributed as dist

    import oracle as O
    import synth
    from engram_gram_conditional_gb300.sharded import RowExchange, bucket_range, row_range

    dist.init_process_group("gloo")
    w = synth.WORKLOADS["tiny"]
    g = O.Geom(vocab=w.vocab, vc=w.vc, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d)
    p = O.layer_params(g, w.hash_seeds, w.bucket_bases, 0)
    seed, rd, raw_bytes = w.table_seeds[0], w.row_dim, w.row_dim + 16
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    # this rank's own tokens: a ragged count, an image span (masked n-grams)
    T = 29 + 11 * rank
    toks = synth.session_tokens(w, rank, T)
    win = O.windows(g, tmap, toks, synth.image_flags(T, [(5, 2)]))
    ids_bm = np.ascontiguousarray(np.stack([O.hash_rows(g, p, x) for x in win]).T)  # [nb][T]
    # the rows this rank owns, and only those
    lo, hi = bucket_range(g.nb, world, rank)
    row_lo, row_hi = row_range(p.offset, p.prime, lo, hi)
    shard = [O.table_row(seed, r, rd) for r in range(row_lo, row_hi)]
    seen = []

    def gather(recv):
        ids = recv.numpy().view(np.uint32)
        out = np.zeros((len(ids), raw_bytes), np.uint8)
        for i, r in enumerate(ids):
            if r == O.MASKED:
                continue
            seen.append(int(r))
            codes, scales = shard[int(r) - row_lo]
            out[i, :rd] = codes
            out[i, rd:rd + rd // 32] = scales
        return torch.from_numpy(out)

    ex = RowExchange(g.nb, raw_bytes)
    raw = ex.exchange(torch.from_numpy(ids_bm.view(np.int32)), gather).numpy()
    # the single-rank lookup from the whole table
    want = np.zeros((g.nb, T, raw_bytes), np.uint8)
    for b in range(g.nb):
        for t in range(T):
            r = int(ids_bm[b, t])
            if r != O.MASKED:
                codes, scales = O.table_row(seed, r, rd)
                want[b, t, :rd] = codes
                want[b, t, rd:rd + rd // 32] = scales
    owned_only = all(row_lo <= r < row_hi for r in seen)
    queue.put((rank, bool(np.array_equal(raw, want)), owned_only, len(seen), (lo, hi)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 7])
def test_sharded_table_row_exchange_matches_one_rank(world):
    # 6 buckets over 2 ranks (3 each) or 7 ranks (one rank owns no bucket):
    # every rank's routed rows equal the whole table's rows bit for bit, and
    # an owner is only ever asked for rows of its own buckets
    import oracle as O

    O.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(ok for _, ok, _, _, _ in results)
    assert all(owned for _, _, owned, _, _ in results)
    ranges = [r[4] for r in results]
    assert ranges[0][0] == 0 and ranges[-1][1] == 6
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))  # contiguous, in rank order
    if world > 6:
        assert any(lo == hi for lo, hi in ranges) and sum(r[3] for r in results) > 0
