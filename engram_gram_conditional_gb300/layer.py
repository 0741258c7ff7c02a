"""Device memory plumbing for a set of Engram layers.

PyTorch allocates the device buffers (HBM); a table read through UVA lives in
the library's registered, huge-page-advised host memory
(engram_host_table_alloc).  The library fills the tables on the device and
binds the weights.  No forward arithmetic happens here.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import (BIND_TABLE_BF16, engram_ctx_create, engram_ctx_destroy, engram_host_table_alloc,
               engram_host_table_free, engram_layer_bind, engram_layer_params, engram_table_fill,
               engram_table_fill_bf16)


def _round16(n: int) -> int:
    return (n + 15) // 16 * 16


def _as_device(x, dtype, device):
    if isinstance(x, torch.Tensor):
        return x.to(device=device, dtype=dtype).contiguous()
    return torch.from_numpy(np.ascontiguousarray(x)).view(dtype).to(device)


class EngramLayerSet:
    """One context (geometry, token map, hash parameters) and its layers' weights."""

    def __init__(self, vocab, vc, token_map, layer_seeds, bucket_bases, *, min_n=2, max_n=4,
                 heads=8, row_dim=256, hc=4, d=5120, pad_cid=0, eps=1e-6, device="cuda"):
        self.device = torch.device(device)
        self.geom = dict(vocab=vocab, vc=vc, min_n=min_n, max_n=max_n, heads=heads,
                         row_dim=row_dim, hc=hc, d=d, pad_cid=pad_cid, eps=eps)
        self.nb = (max_n - min_n + 1) * heads
        self.K = self.nb * row_dim
        self.N = (hc + 1) * d
        self.ctx = engram_ctx_create(vocab, vc, token_map, layer_seeds, bucket_bases, min_n=min_n,
                                     max_n=max_n, heads=heads, row_dim=row_dim, hc=hc, d=d,
                                     pad_cid=pad_cid, eps=eps)
        self.n_layers = len(layer_seeds)
        self.params = [engram_layer_params(self.ctx, l, self.nb) for l in range(self.n_layers)]
        self.tensors = [dict() for _ in range(self.n_layers)]
        self._host = []  # (address, bytes) of host tables from engram_host_table_alloc

    @classmethod
    def from_workload(cls, w, token_map, device="cuda"):
        return cls(w.vocab, w.vc, token_map, w.hash_seeds, w.bucket_bases, min_n=w.min_n,
                   max_n=w.max_n, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d,
                   pad_cid=w.pad_cid, eps=w.eps, device=device)

    def rows(self, layer: int) -> int:
        return self.params[layer][3]

    def bind(self, layer: int, table_seed: int, wkv, wq, wk, host_table: bool = False,
             stream=None, flags: int = 0, table=None):
        """Allocate and fill the layer's table, upload wkv / w_q / w_k, bind.

        The table is MXFP8 (codes and E8M0 scales), or with flags containing
        BIND_TABLE_BF16 the same rows stored as BF16 values without scales.
        ``table``: instead of the generated contents, a host MXFP8 table
        (codes uint8 [R][row_dim], scales uint8 [R][row_dim / 32]) with R at
        least the layer's row count, copied as it is (rows past the layer's
        count stay allocated but outside the bound table)."""
        rows = self.rows(layer)
        rd = self.geom["row_dim"]

        def buf(nbytes):
            # host tables: the library's registered, huge-page-advised host
            # memory (zeroed); device tables: HBM from torch
            if not host_table:
                return torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
            ptr = engram_host_table_alloc(nbytes)
            self._host.append((ptr, nbytes))
            arr = np.ctypeslib.as_array((ctypes.c_uint8 * nbytes).from_address(ptr))
            return torch.from_numpy(arr)

        if table is not None:
            codes = np.ascontiguousarray(table[0], np.uint8).reshape(-1)
            scl = np.ascontiguousarray(table[1], np.uint8).reshape(-1)
            assert codes.size >= rows * rd and scl.size * 32 == codes.size and not flags & BIND_TABLE_BF16
            table_t = buf(_round16(codes.size))
            scales = buf(_round16(scl.size))
            table_t[:codes.size].copy_(torch.from_numpy(codes))
            scales[:scl.size].copy_(torch.from_numpy(scl))
            table = table_t
        elif flags & BIND_TABLE_BF16:
            table = buf(_round16(rows * rd * 2))
            scales = None
            engram_table_fill_bf16(self.ctx, table_seed, table, 0, rows, stream)
        else:
            table = buf(_round16(rows * rd))
            scales = buf(_round16(rows * rd // 32))
            engram_table_fill(self.ctx, table_seed, table, scales, 0, rows, stream)
        d_wkv = _as_device(wkv, torch.int16, self.device).view(self.N, self.K)
        d_wq = _as_device(wq, torch.float32, self.device).view(-1)
        d_wk = _as_device(wk, torch.float32, self.device).view(-1)
        engram_layer_bind(self.ctx, layer, table, scales, rows, d_wkv, d_wq, d_wk, flags)
        self.tensors[layer] = dict(table=table, scales=scales, wkv=d_wkv, wq=d_wq, wk=d_wk,
                                   table_seed=table_seed)
        return self.tensors[layer]

    def close(self):
        if self.ctx is not None:
            if self._host:
                torch.cuda.synchronize(self.device)  # no kernel reads a table freed below
            engram_ctx_destroy(self.ctx)
            self.ctx = None
        self.tensors = []
        for ptr, nbytes in self._host:
            engram_host_table_free(ptr, nbytes)
        self._host = []
