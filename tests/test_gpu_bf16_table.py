"""The BF16-table storage variant (ENGRAM_BIND_TABLE_BF16), through the C ABI.

The table holds each row's dequantised values as BF16 (2 x row_dim bytes, no
scales), the second storage format on the pages ([zhuai], the w8a8
repository's BF16 table).  Filled from the same seed, its values are the
MXFP8 table's E4M3(code) x 2^(scale - 127), which BF16 holds exactly, so the
gather must match the oracle's bit for bit and the forward must match both the
oracle and an MXFP8 layer on the same BF16 operand path.
"""
import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from helpers import (check_hidden, from_dev, geom, prefill_windows, setup_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def tiny_bf16_table():
    s = setup_workload("tiny", flags=eg.BIND_TABLE_BF16)
    yield s
    s.close()


@pytest.fixture(scope="module")
def tiny_mxfp8_bf16_ops():
    s = setup_workload("tiny", flags=eg.BIND_BF16_OPERANDS)
    yield s
    s.close()


def staged(s, win, hidden):
    T = win.shape[0]
    ctx = s.model.ctx
    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                     device="cuda")
    d_h = to_dev(hidden)
    d_g = torch.full((T, s.w.hc), float("nan"), device="cuda")
    eg.engram_forward_staged(ctx, 0, to_dev(win), T, d_h, ws, d_g)
    eg.engram_sync(ctx)
    return from_dev(d_h, np.uint16), d_g.cpu().numpy()


def test_layer_info_reports_the_bf16_table(tiny_bf16_table):
    info = eg.engram_layer_info(tiny_bf16_table.model.ctx, 0)
    assert info["bound"] == 1 and info["table_bf16"] == 1
    assert info["fp16_operands"] == 0 and info["bucket_gather"] == 0


def test_table_fill_equals_the_dequantised_mxfp8_rows(tiny_bf16_table):
    s = tiny_bf16_table
    t = s.model.tensors[0]["table"].cpu().numpy().view(np.uint16)
    rd = s.w.row_dim
    rows = s.model.rows(0)
    for r in list(range(0, rows, 97)) + [rows - 1]:
        codes, scales = O.table_row(s.w.table_seeds[0], r, rd)
        want = np.array([O.bf16_from_double(O.e4m3_value(int(codes[c])) *
                                            O.e8m0_value(int(scales[c // 32])))
                         for c in range(rd)], np.uint16)
        assert np.array_equal(t[r * rd:(r + 1) * rd], want), r


@pytest.mark.parametrize("sessions,per", [(1, 64), (3, 70)])
def test_gather_bit_exact(tiny_bf16_table, sessions, per):
    s = tiny_bf16_table
    win, _, _ = prefill_windows(s, sessions, per)
    T = win.shape[0]
    d_rows = torch.empty((T, s.w.nb), dtype=torch.int32, device="cuda")
    d_emb = torch.empty((T, s.w.K), dtype=torch.int16, device="cuda")
    eg.engram_hash(s.model.ctx, 0, to_dev(win), T, d_rows)
    eg.engram_gather_dequant(s.model.ctx, 0, d_rows, T, d_emb)
    eg.engram_sync(s.model.ctx)
    rows, emb = from_dev(d_rows, np.uint32), from_dev(d_emb, np.uint16)
    g = geom(s.w)
    for t in range(T):
        assert np.array_equal(emb[t], O.gather(g, s.w.table_seeds[0], rows[t])), t


@pytest.mark.parametrize("sessions,per,spans", [(1, 64, [(20, 4)]), (2, 129, [(128, 1)])])
def test_staged_forward_matches_oracle_and_mxfp8(tiny_bf16_table, tiny_mxfp8_bf16_ops, sessions,
                                                 per, spans):
    s = tiny_bf16_table
    win, _, _ = prefill_windows(s, sessions, per, spans)
    T = win.shape[0]
    hidden = synth.hidden_bf16(s.w, T)
    h, gates = staged(s, win, hidden)
    ref = O.forward(geom(s.w), s.w.table_seeds[0], s.oparams[0], s.W[0], s.wq[0], s.wk[0], win,
                    hidden, np.arange(T), nthreads=4)
    check_hidden(h, ref["h_bf16"], "bf16 table staged")
    assert np.abs(gates - ref["gates"]).max() <= 1e-3
    # the MXFP8 layer on the BF16 operand path stages the same operand rows
    h2, g2 = staged(tiny_mxfp8_bf16_ops, win, hidden)
    assert np.array_equal(h, h2) and np.array_equal(gates, g2)


def test_fused_entries_refuse_a_bf16_table(tiny_bf16_table):
    s = tiny_bf16_table
    ctx = s.model.ctx
    win, _, _ = prefill_windows(s, 1, 16)
    T = win.shape[0]
    d_w = to_dev(win)
    d_h = to_dev(synth.hidden_bf16(s.w, T))
    ws = torch.empty(max(16, eg.engram_workspace_bytes(ctx, T)), dtype=torch.uint8, device="cuda")
    d_kv = torch.empty((T, s.w.N), dtype=torch.float32, device="cuda")
    for call in (lambda: eg.engram_forward(ctx, 0, d_w, T, d_h, ws),
                 lambda: eg.engram_project_windows(ctx, 0, d_w, T, d_kv)):
        with pytest.raises(eg.EngramError) as e:
            call()
        assert e.value.status == eg.EUNSUPPORTED


def test_full_geometry_prefill_sampled():
    s = setup_workload("prefill_2048", flags=eg.BIND_TABLE_BF16)
    try:
        win, _, _ = prefill_windows(s, 1, 2048, spans=[(1000, 8)])
        hidden = synth.hidden_bf16(s.w, 2048)
        h, gates = staged(s, win, hidden)
        sample = np.array([0, 1, 127, 128, 999, 1000, 1008, 1009, 2047])
        ref = O.forward(geom(s.w), s.w.table_seeds[0], s.oparams[0], s.W[0], s.wq[0], s.wk[0],
                        win, hidden, sample, nthreads=8)
        check_hidden(h[sample], ref["h_bf16"], "bf16 table prefill")
        assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3
    finally:
        s.close()


def test_bf16_table_in_pinned_host_memory_two_step():
    # a BF16 table read through UVA, staged and run with the two-step API
    s = setup_workload("tiny", host_table=True, flags=eg.BIND_TABLE_BF16)
    try:
        t = s.model.tensors[0]["table"]
        assert not t.is_cuda and t.is_pinned()
        win, _, _ = prefill_windows(s, 2, 90, spans=[(40, 3)])
        T = win.shape[0]
        hidden = synth.hidden_bf16(s.w, T)
        ctx = s.model.ctx
        ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                         device="cuda")
        d_w, d_h = to_dev(win), to_dev(hidden)
        eg.engram_stage_rows(ctx, 0, d_w, T, ws)
        eg.engram_forward_staged_rows(ctx, 0, d_w, T, d_h, ws)
        eg.engram_sync(ctx)
        ref = O.forward(geom(s.w), s.w.table_seeds[0], s.oparams[0], s.W[0], s.wq[0], s.wk[0], win,
                        hidden, np.arange(T), nthreads=4)
        check_hidden(from_dev(d_h, np.uint16), ref["h_bf16"], "bf16 host table")
    finally:
        s.close()
