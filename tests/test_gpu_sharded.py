"""The kernels of a table sharded over ranks by bucket, on one GPU.

Nothing here runs more than one GPU: two contexts on the same device stand for
two ranks, each bound to the shard of its buckets (engram_layer_bind_shard).
The requester hashes bucket-major, each owner gathers the raw rows of its
buckets' ids from its shard, the blocks are concatenated in owner order (what
the all-to-all delivers; the routing itself is tested on gloo ranks in
test_dist_cpu.py), and the requester decodes them and runs the GEMM and the
gate.  The result must equal engram_forward_staged on the whole table bit for
bit: the same operand values reach the same kernels.
"""
import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from engram_gram_conditional_gb300.layer import EngramLayerSet
from engram_gram_conditional_gb300.sharded import bucket_range, row_range
from helpers import from_dev, prefill_windows, setup_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


class Owner:
    """A context bound to the shard of buckets [lo, hi) (the rows they span)."""

    def __init__(self, s, lo, hi, span):
        w = s.w
        self.m = EngramLayerSet.from_workload(w, s.tmap, device="cuda")
        _, prime, offset, _ = self.m.params[0]
        self.lo, self.hi = lo, hi
        self.row_lo, self.row_hi = row_range(offset, prime, lo, hi)
        n = self.row_hi - self.row_lo
        rd = w.row_dim
        self.table = torch.zeros(max(16, n * rd), dtype=torch.uint8, device="cuda")
        self.scales = torch.zeros(max(16, (n * rd // 32 + 15) // 16 * 16), dtype=torch.uint8,
                                  device="cuda")
        if n:
            eg.engram_table_fill(self.m.ctx, w.table_seeds[0],
                                 self.table.data_ptr() - self.row_lo * rd,
                                 self.scales.data_ptr() - self.row_lo * (rd // 32), self.row_lo,
                                 self.row_hi)
        self.span = eg.engram_scale_range(self.m.ctx, self.scales, n * (rd // 32))
        t = s.model.tensors[0]
        eg.engram_layer_bind_shard(self.m.ctx, 0, self.table if n else None,
                                   self.scales if n else None, n, t["wkv"], t["wq"], t["wk"],
                                   self.row_lo, *span)

    def close(self):
        self.m.close()


def sharded_forward(s, owners, win, hidden):
    """Hash (requester = owner 0's context), per-owner raw gathers, decode, GEMM + gate."""
    T = win.shape[0]
    ctx = owners[0].m.ctx
    rb = eg.engram_raw_row_bytes(ctx)
    d_win = to_dev(win)
    ids = torch.empty((s.w.nb, T), dtype=torch.int32, device="cuda")
    eg.engram_hash_by_bucket(ctx, 0, d_win, T, ids)
    blocks = []
    for o in owners:
        mine = ids[o.lo:o.hi].reshape(-1).contiguous()
        raw = torch.empty((mine.numel(), rb), dtype=torch.uint8, device="cuda")
        eg.engram_shard_gather_raw(o.m.ctx, 0, mine, mine.numel(), raw)
        blocks.append(raw)
    raw_bm = torch.cat(blocks).view(s.w.nb, T, rb)
    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                     device="cuda")
    d_h = to_dev(hidden)
    d_g = torch.full((T, s.w.hc), float("nan"), device="cuda")
    eg.engram_stage_raw_rows(ctx, 0, ids, raw_bm, T, ws)
    eg.engram_forward_staged_rows(ctx, 0, d_win, T, d_h, ws, d_g)
    for o in owners:
        eg.engram_sync(o.m.ctx)
    return ids, raw_bm, from_dev(d_h, np.uint16), d_g.cpu().numpy()


def whole_table_forward(s, win, hidden):
    T = win.shape[0]
    ctx = s.model.ctx
    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                     device="cuda")
    d_h = to_dev(hidden)
    d_g = torch.full((T, s.w.hc), float("nan"), device="cuda")
    eg.engram_forward_staged(ctx, 0, to_dev(win), T, d_h, ws, d_g)
    eg.engram_sync(ctx)
    return from_dev(d_h, np.uint16), d_g.cpu().numpy()


@pytest.mark.parametrize("name,ranks,sizes", [("tiny", 2, [(1, 64), (3, 43)]),
                                              ("tiny", 4, [(2, 70)]),
                                              ("prefill_2048", 2, [(1, 256), (1, 2048)])])
def test_sharded_rows_give_the_staged_forward(name, ranks, sizes):
    s = setup_workload(name)
    owners = []
    try:
        _, prime, offset, _ = s.model.params[0]
        parts = [bucket_range(s.w.nb, ranks, r) for r in range(ranks)]
        # each rank's span of its shard, combined (what the ranks' all-reduce does)
        rd = s.w.row_dim
        spans = []
        for lo, hi in parts:
            row_lo, row_hi = row_range(offset, prime, lo, hi)
            sc = s.model.tensors[0]["scales"][row_lo * (rd // 32):row_hi * (rd // 32)]
            spans.append(eg.engram_scale_range(s.model.ctx, sc, sc.numel()))
        span = (min(a for a, _ in spans), max(b for _, b in spans))
        assert span == (119, 127)
        owners = [Owner(s, lo, hi, span) for lo, hi in parts]
        info_full = eg.engram_layer_info(s.model.ctx, 0)
        info_shard = eg.engram_layer_info(owners[0].m.ctx, 0)
        for k in ("fp16_operands", "a_exp_shift", "wkv_exp", "scale_min", "scale_max"):
            assert info_full[k] == info_shard[k], k
        for sessions, per in sizes:
            win, _, _ = prefill_windows(s, sessions, per, spans=[(per // 3, 4)])
            T = win.shape[0]
            hidden = synth.hidden_bf16(s.w, T)
            ids, raw_bm, h, gates = sharded_forward(s, owners, win, hidden)
            # bucket-major ids are the transposed row indices
            d_rows = torch.empty((T, s.w.nb), dtype=torch.int32, device="cuda")
            eg.engram_hash(s.model.ctx, 0, to_dev(win), T, d_rows)
            assert np.array_equal(from_dev(ids, np.uint32), from_dev(d_rows, np.uint32).T)
            # raw rows: the table's bytes (codes, scales, zero padding); masked rows zero
            raw = raw_bm.cpu().numpy()
            idn = from_dev(ids, np.uint32)
            for b, t in [(0, 0), (s.w.nb - 1, T - 1), (s.w.nb // 2, T // 2)]:
                r = int(idn[b, t])
                if r == eg.MASKED:
                    assert (raw[b, t] == 0).all()
                    continue
                codes, scl = O.table_row(s.w.table_seeds[0], r, rd)
                assert np.array_equal(raw[b, t, :rd], codes)
                assert np.array_equal(raw[b, t, rd:rd + rd // 32], scl)
                assert (raw[b, t, rd + rd // 32:] == 0).all()
            h_ref, g_ref = whole_table_forward(s, win, hidden)
            assert np.array_equal(h, h_ref), (name, ranks, T)
            assert np.array_equal(gates, g_ref), (name, ranks, T)
    finally:
        for o in owners:
            o.close()
        s.close()


def test_shard_gather_outside_the_shard_and_global_calls():
    s = setup_workload("tiny")
    owner = None
    try:
        owner = Owner(s, 0, 3, (119, 127))
        ctx = owner.m.ctx
        rb = eg.engram_raw_row_bytes(ctx)
        # an id outside the shard: a zero row and ENGRAM_EBOUNDS once; the
        # largest id inside it: its row
        ids = torch.tensor([owner.row_hi, eg.MASKED, owner.row_hi - 1],
                           dtype=torch.int64).to(torch.int32).cuda()
        raw = torch.full((3, rb), 7, dtype=torch.uint8, device="cuda")
        eg.engram_shard_gather_raw(ctx, 0, ids, 3, raw)
        with pytest.raises(eg.EngramError) as e:
            eg.engram_sync(ctx)
        assert e.value.status == eg.EBOUNDS
        r = raw.cpu().numpy()
        assert (r[0] == 0).all() and (r[1] == 0).all()
        codes, scl = O.table_row(s.w.table_seeds[0], owner.row_hi - 1, s.w.row_dim)
        assert np.array_equal(r[2, :s.w.row_dim], codes)
        eg.engram_sync(ctx)  # cleared
        # calls that index the table with global rows refuse a shard
        win, _, _ = prefill_windows(s, 1, 16)
        d_win = to_dev(win)
        d_h = to_dev(synth.hidden_bf16(s.w, 16))
        ws = torch.empty(max(eg.engram_workspace_bytes(ctx, 16),
                             eg.engram_forward_staged_workspace_bytes(ctx, 16)),
                         dtype=torch.uint8, device="cuda")
        for call in (lambda: eg.engram_forward(ctx, 0, d_win, 16, d_h, ws),
                     lambda: eg.engram_forward_staged(ctx, 0, d_win, 16, d_h, ws),
                     lambda: eg.engram_forward_noalloc(ctx, 0, d_win, 16, d_h)):
            with pytest.raises(eg.EngramError) as e:
                call()
            assert e.value.status == eg.ESTATE
    finally:
        if owner:
            owner.close()
        s.close()
