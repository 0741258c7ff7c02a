"""An Engram table sharded over data-parallel ranks by bucket, exchanged by all-to-all.

Source: the vLLM "Engram" feature wiki, section "데이터 병렬 토폴로지"
(embedding_across_dp): the hash heads are spread over the co-located
replicas; each step a replica receives the row ids of every replica's tokens
for its own heads, looks them up and sends the rows back.  The FlagScale
plugin article describes the same exchange, an all-to-all where a replicated
table would need an all-reduce.

Rank r owns the contiguous bucket range ``bucket_range(nb, world, r)``, hence
the contiguous row range ``[offset[b_lo], offset[b_hi])`` of the layer's
table (the buckets' prime ranges are laid out in bucket order), and holds only
those rows.  One step, on each rank's own T tokens:

1. the rank hashes its windows bucket-major, ids [nb][T]
   (``engram_hash_by_bucket``);
2. all-to-all: the owner of buckets [lo, hi) receives ids[lo:hi] of every rank;
3. the owner gathers the raw MXFP8 rows of those ids from its shard
   (``engram_shard_gather_raw``: row_dim codes and row_dim / 32 scale bytes,
   row_dim + 16 bytes a row, half the bytes of the dequantised BF16 row);
4. all-to-all back: every rank receives raw rows [nb][T][raw] in bucket order;
5. the rank decodes them into its staged operand (``engram_stage_raw_rows``)
   and runs the GEMM and the gate on its own tokens
   (``engram_forward_staged_rows``).

This module holds the exchange's bookkeeping and its collectives only; the
hashing, the gather and the decode run in the library's kernels, and the
exchange (``RowExchange``) takes the owner's gather as a callable, so the same
routing runs on GPU tensors over NCCL and on CPU tensors over gloo.
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist

from . import (engram_forward_staged_rows, engram_hash_by_bucket, engram_layer_bind_shard,
               engram_raw_row_bytes, engram_scale_range, engram_shard_gather_raw,
               engram_stage_raw_rows, engram_table_fill)


def bucket_range(nb: int, world: int, rank: int):
    """Buckets [lo, hi) owned by a rank: contiguous, as even as possible."""
    return nb * rank // world, nb * (rank + 1) // world


def row_range(offset, prime, lo: int, hi: int):
    """Rows [row_lo, row_hi) of the layer's table that buckets [lo, hi) span."""
    offset = [int(x) for x in offset]
    prime = [int(x) for x in prime]
    if lo >= hi:
        base = offset[lo] if lo < len(offset) else offset[-1] + prime[-1]
        return base, base
    return offset[lo], offset[hi - 1] + prime[hi - 1]


class RowExchange:
    """The two all-to-alls of one step: row ids out to their owners, raw rows back."""

    def __init__(self, nb: int, raw_bytes: int, group=None):
        self.nb = nb
        self.raw_bytes = raw_bytes
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.ranges = [bucket_range(nb, self.world, r) for r in range(self.world)]

    def token_counts(self, T: int, device) -> list:
        t = torch.tensor([T], dtype=torch.int64, device=device)
        out = [torch.zeros_like(t) for _ in range(self.world)]
        dist.all_gather(out, t, group=self.group)
        return [int(x.item()) for x in out]

    def exchange(self, ids_bm: torch.Tensor, gather_raw: Callable[[torch.Tensor], torch.Tensor],
                 counts=None) -> torch.Tensor:
        """ids_bm: this rank's row ids, int32 [nb][T] (bucket-major, contiguous).
        gather_raw(ids) -> uint8 [len(ids)][raw_bytes]: the owner's lookup of the
        ids it received (every rank's ids of its buckets, rank by rank).
        Returns this rank's raw rows, uint8 [nb][T][raw_bytes], in bucket order."""
        nb, T = ids_bm.shape
        assert nb == self.nb and ids_bm.is_contiguous()
        counts = self.token_counts(T, ids_bm.device) if counts is None else counts
        lo, hi = self.ranges[self.rank]
        mine = hi - lo
        # 1: ids out, owner o gets rows [lo_o, hi_o) of ids_bm (contiguous)
        send_splits = [(h - l) * T for l, h in self.ranges]
        recv_splits = [mine * t for t in counts]
        recv_ids = torch.empty(sum(recv_splits), dtype=ids_bm.dtype, device=ids_bm.device)
        dist.all_to_all_single(recv_ids, ids_bm.reshape(-1), recv_splits, send_splits,
                               group=self.group)
        # 2: the owner's lookup, in the order received
        raw = gather_raw(recv_ids)
        assert raw.dtype == torch.uint8 and raw.numel() == recv_ids.numel() * self.raw_bytes
        # 3: raw rows back; owner o's block is buckets [lo_o, hi_o) x T, so the
        # blocks of owners 0, 1, ... concatenate to [nb][T][raw] in bucket order
        back = torch.empty(nb * T * self.raw_bytes, dtype=torch.uint8, device=ids_bm.device)
        dist.all_to_all_single(back, raw.reshape(-1), [s * self.raw_bytes for s in send_splits],
                               [s * self.raw_bytes for s in recv_splits], group=self.group)
        return back.view(nb, T, self.raw_bytes)


def _round16(n: int) -> int:
    return (n + 15) // 16 * 16


class ShardedLayer:
    """One Engram layer of an ``EngramLayerSet`` whose table is sharded over the
    ranks of ``group`` (one rank per GPU): this rank holds the rows of its
    buckets, filled on the device, and whole wkv / w_q / w_k."""

    def __init__(self, model, layer: int, table_seed: int, wkv, wq, wk, group=None):
        from .layer import _as_device

        self.model, self.layer = model, layer
        ctx = model.ctx
        mult, prime, offset, rows = model.params[layer]
        self.nb = model.nb
        self.exchange_ = RowExchange(self.nb, engram_raw_row_bytes(ctx), group)
        lo, hi = self.exchange_.ranges[self.exchange_.rank]
        self.row_lo, self.row_hi = row_range(offset, prime, lo, hi)
        n = self.row_hi - self.row_lo
        rd = model.geom["row_dim"]
        dev = model.device
        self.table = torch.zeros(_round16(max(n, 1) * rd), dtype=torch.uint8, device=dev)
        self.scales = torch.zeros(_round16(max(n, 1) * rd // 32), dtype=torch.uint8, device=dev)
        if n:
            # the fill writes row r at data + r row_dim: offset the base so that
            # rows [row_lo, row_hi) land at the start of the shard
            engram_table_fill(ctx, table_seed, self.table.data_ptr() - self.row_lo * rd,
                              self.scales.data_ptr() - self.row_lo * (rd // 32), self.row_lo,
                              self.row_hi)
        # the whole table's exponent span: every rank's shard span, combined
        smin, smax = engram_scale_range(ctx, self.scales, n * (rd // 32))
        span = torch.tensor([smin, -smax], dtype=torch.int64, device=dev)
        dist.all_reduce(span, op=dist.ReduceOp.MIN, group=group)
        self.scale_min, self.scale_max = int(span[0]), int(-span[1])
        self.wkv = _as_device(wkv, torch.int16, dev).view(model.N, model.K)
        self.wq = _as_device(wq, torch.float32, dev).view(-1)
        self.wk = _as_device(wk, torch.float32, dev).view(-1)
        engram_layer_bind_shard(ctx, layer, self.table if n else None,
                                self.scales if n else None, n, self.wkv, self.wq, self.wk,
                                self.row_lo, self.scale_min, self.scale_max)

    def forward(self, d_windows: torch.Tensor, T: int, d_hidden: torch.Tensor,
                d_workspace: torch.Tensor, d_gates=None):
        """The layer's step on this rank's T tokens (windows [T][4], hidden
        [T][hc][d] updated in place, workspace of
        engram_forward_staged_workspace_bytes(ctx, T) bytes), on torch's
        current stream; the all-to-alls run between the hash and the decode."""
        ctx, layer = self.model.ctx, self.layer
        stream = torch.cuda.current_stream()
        ids = torch.empty((self.nb, T), dtype=torch.int32, device=d_windows.device)
        engram_hash_by_bucket(ctx, layer, d_windows, T, ids, stream)
        rb = self.exchange_.raw_bytes

        def gather(recv_ids):
            raw = torch.empty((recv_ids.numel(), rb), dtype=torch.uint8, device=recv_ids.device)
            engram_shard_gather_raw(ctx, layer, recv_ids, recv_ids.numel(), raw, stream)
            return raw

        raw_bm = self.exchange_.exchange(ids, gather)
        engram_stage_raw_rows(ctx, layer, ids, raw_bm, T, d_workspace, stream)
        engram_forward_staged_rows(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates,
                                   stream)
