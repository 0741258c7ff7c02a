"""The pre-pass through the staged path (engram_prepass) and the gate on a
BF16 kv (engram_gate_bf16kv), through the C ABI.

The pre-pass computes kv = e wkv^T from the windows alone ("DeepSeek V4.1
Flash 的 Engram", section "提前投影": hashing, gather and projection need only
the tokens).  As fp32 it must meet the projection's fp32 accumulation bound
against the oracle.  As BF16 it must be, bit for bit, the fp32 pre-pass output
rounded once to nearest even: both come from the same GEMM in the same
accumulation order.  The BF16-kv gate must match the oracle's gate evaluated
on the very BF16 kv the GPU read.
"""
import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from helpers import (bf16_f64, check_hidden, check_kv, from_dev, geom, prefill_windows,
                     setup_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def tiny():
    s = setup_workload("tiny")
    yield s
    s.close()


@pytest.fixture(scope="module")
def prefill():
    s = setup_workload("prefill_2048")
    yield s
    s.close()


def rne_bf16(f32: np.ndarray) -> np.ndarray:
    """fp32 -> BF16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def prepass(s, win, kv_format):
    T = win.shape[0]
    ctx = s.model.ctx
    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                     device="cuda")
    dtype = torch.float32 if kv_format == eg.KV_F32 else torch.int16
    d_kv = torch.full((T, s.w.N), -1, dtype=dtype, device="cuda")
    eg.engram_prepass(ctx, 0, to_dev(win), T, d_kv, kv_format, ws)
    eg.engram_sync(ctx)
    return d_kv.cpu().numpy() if kv_format == eg.KV_F32 else from_dev(d_kv, np.uint16)


@pytest.mark.parametrize("sessions,per", [(1, 64), (3, 43), (1, 1), (2, 100)])
def test_prepass_f32_meets_the_fp32_bound_tiny(tiny, sessions, per):
    win, _, _ = prefill_windows(tiny, sessions, per)
    kv = prepass(tiny, win, eg.KV_F32)
    g = geom(tiny.w)
    for t in range(win.shape[0]):
        e = O.gather(g, tiny.w.table_seeds[0], O.hash_rows(g, tiny.oparams[0], win[t]))
        check_kv(kv[t], O.project(g, tiny.W[0], e), tiny.W[0], e, tiny.w.K, f"token {t}")


@pytest.mark.parametrize("T", [1, 77, 256, 300, 2048])
def test_prepass_full_geometry(prefill, T):
    # 1, 77: one 128-token block (single CTAs, stream K); 256, 300: CTA pairs with
    # stream K (300: an odd block count); 2,048: pairs, whole tiles
    win, _, _ = prefill_windows(prefill, 1, T)
    kv32 = prepass(prefill, win, eg.KV_F32)
    kv16 = prepass(prefill, win, eg.KV_BF16)
    assert np.array_equal(kv16, rne_bf16(kv32)), "BF16 kv is not the fp32 kv rounded once"
    sample = sorted({0, T // 2, T - 1})
    ref = O.forward(geom(prefill.w), prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0],
                    prefill.wq[0], prefill.wk[0], win, synth.hidden_bf16(prefill.w, T),
                    np.array(sample), nthreads=8, want_e=True, want_kv=True, want_h64=False)
    for i, t in enumerate(sample):
        check_kv(kv32[t], ref["kv"][i], prefill.W[0], ref["e"][i], prefill.w.K, f"token {t}")


def test_gate_bf16kv_matches_the_oracle_gate_on_the_same_kv(tiny):
    win, _, _ = prefill_windows(tiny, 2, 70, spans=[(30, 4)])
    T = win.shape[0]
    kv16 = prepass(tiny, win, eg.KV_BF16)
    hidden = synth.hidden_bf16(tiny.w, T)
    ctx = tiny.model.ctx
    d_h = to_dev(hidden)
    d_g = torch.full((T, tiny.w.hc), float("nan"), device="cuda")
    eg.engram_gate_bf16kv(ctx, 0, to_dev(kv16), to_dev(win), T, d_h, d_g)
    eg.engram_sync(ctx)
    g = geom(tiny.w)
    exp_h = np.zeros_like(hidden)
    exp_g = np.zeros((T, tiny.w.hc))
    kv64 = bf16_f64(kv16)
    for t in range(T):
        _, exp_h[t], exp_g[t] = O.gate(g, kv64[t], int(win[t][0]), hidden[t], tiny.wq[0],
                                       tiny.wk[0])
    got = from_dev(d_h, np.uint16)
    check_hidden(got, exp_h, "bf16-kv gate")
    assert np.abs(d_g.cpu().numpy() - exp_g).max() <= 1e-3
    img = win[:, 0] == 0xFFFFFFFF
    assert img.any() and np.array_equal(got[img], hidden[img])  # image rows untouched


@pytest.mark.parametrize("T", [256, 2048])
def test_prepass_then_gate_equals_the_forward(prefill, T):
    # fp32 kv: the two calls give the forward's result (within the tolerance)
    win, _, _ = prefill_windows(prefill, 1, T, spans=[(100, 8)])
    hidden = synth.hidden_bf16(prefill.w, T)
    kv32 = prepass(prefill, win, eg.KV_F32)
    ctx = prefill.model.ctx
    d_h = to_dev(hidden)
    d_g = torch.empty((T, prefill.w.hc), device="cuda")
    eg.engram_gate(ctx, 0, torch.from_numpy(kv32).cuda(), to_dev(win), T, d_h, d_g)
    eg.engram_sync(ctx)
    sample = np.array([0, 99, 100, 107, 108, T - 1])
    ref = O.forward(geom(prefill.w), prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0],
                    prefill.wq[0], prefill.wk[0], win, hidden, sample, nthreads=8)
    check_hidden(from_dev(d_h, np.uint16)[sample], ref["h_bf16"], "pre-pass + gate")
    assert np.abs(d_g.cpu().numpy()[sample] - ref["gates"]).max() <= 1e-3


def test_prepass_on_a_bf16_table():
    s = setup_workload("tiny", flags=eg.BIND_TABLE_BF16)
    try:
        win, _, _ = prefill_windows(s, 1, 64)
        kv = prepass(s, win, eg.KV_F32)
        g = geom(s.w)
        for t in range(64):
            e = O.gather(g, s.w.table_seeds[0], O.hash_rows(g, s.oparams[0], win[t]))
            check_kv(kv[t], O.project(g, s.W[0], e), s.W[0], e, s.w.K, f"token {t}")
    finally:
        s.close()


def test_prepass_rejects_an_unknown_kv_format(tiny):
    win, _, _ = prefill_windows(tiny, 1, 8)
    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(tiny.model.ctx, 8),
                     dtype=torch.uint8, device="cuda")
    d_kv = torch.empty((8, tiny.w.N), device="cuda")
    with pytest.raises(eg.EngramError) as e:
        eg.engram_prepass(tiny.model.ctx, 0, to_dev(win), 8, d_kv, 7, ws)
    assert e.value.status == eg.EINVAL


def test_back_to_back_calls_on_one_stream_share_a_workspace(prefill):
    # Kernels of consecutive calls overlap (programmatic dependent launch);
    # chained on one stream with one workspace and no synchronisation between
    # them, every call must still give the result it gives alone.
    ctx = prefill.model.ctx
    w = prefill.w
    T1, T2, T3 = 256, 2048, 77
    win1, _, _ = prefill_windows(prefill, 1, T1, spans=[(10, 3)])
    win2, _, _ = prefill_windows(prefill, 2, T2 // 2)
    win3, _, _ = prefill_windows(prefill, 1, T3)
    h1, h2, h3 = (synth.hidden_bf16(w, T) for T in (T1, T2, T3))
    ws = torch.empty(max(eg.engram_forward_staged_workspace_bytes(ctx, T) for T in (T1, T2, T3)) +
                     eg.engram_workspace_bytes(ctx, T2), dtype=torch.uint8, device="cuda")

    def alone(fn):
        out = fn()
        eg.engram_sync(ctx)
        return [x.cpu().numpy() for x in out]

    def staged(win, h):
        d_h = to_dev(h)
        eg.engram_forward_staged(ctx, 0, to_dev(win), win.shape[0], d_h, ws, None)
        return [d_h]

    def prepass_gate(win, h, fmt):
        T = win.shape[0]
        d_kv = torch.empty((T, w.N), dtype=torch.float32 if fmt == eg.KV_F32 else torch.int16,
                           device="cuda")
        d_w, d_h = to_dev(win), to_dev(h)
        eg.engram_prepass(ctx, 0, d_w, T, d_kv, fmt, ws)
        (eg.engram_gate if fmt == eg.KV_F32 else eg.engram_gate_bf16kv)(ctx, 0, d_kv, d_w, T, d_h)
        return [d_h, d_kv]

    def fused(win, h):
        d_h = to_dev(h)
        eg.engram_forward(ctx, 0, to_dev(win), win.shape[0], d_h, ws, None)
        return [d_h]

    calls = [lambda: prepass_gate(win1, h1, eg.KV_F32), lambda: staged(win2, h2),
             lambda: prepass_gate(win3, h3, eg.KV_BF16), lambda: staged(win1, h1),
             lambda: fused(win2, h2), lambda: staged(win3, h3)]
    ref = [alone(c) for c in calls]
    outs = [c() for c in calls]  # back to back
    eg.engram_sync(ctx)
    for i, (o, r) in enumerate(zip(outs, ref)):
        for a, b in zip(o, r):
            assert np.array_equal(a.cpu().numpy(), b), f"call {i}"
    # the staged forward of a small batch (the gate as the stream-K GEMM's
    # epilogue) and the stream-K pre-pass plus the gate kernel compute the same
    # step; the gate's sums are added in another order, so compare within the
    # tolerance of the oracle check
    check_hidden(ref[3][0].view(np.uint16), ref[0][0].view(np.uint16), "staged vs pre-pass + gate")


@pytest.mark.parametrize("T", [256, 2048])
def test_gate_bf16kv_full_geometry_sampled(prefill, T):
    # the BF16-kv gate at full geometry (decode-sized and prefill-sized batches),
    # against the oracle's gate on the same BF16 kv, with an image span
    win, _, _ = prefill_windows(prefill, 1, T, spans=[(40, 5)])
    kv16 = prepass(prefill, win, eg.KV_BF16)
    hidden = synth.hidden_bf16(prefill.w, T)
    ctx = prefill.model.ctx
    d_h = to_dev(hidden)
    d_g = torch.full((T, prefill.w.hc), float("nan"), device="cuda")
    eg.engram_gate_bf16kv(ctx, 0, to_dev(kv16), to_dev(win), T, d_h, d_g)
    eg.engram_sync(ctx)
    got = from_dev(d_h, np.uint16)
    gates = d_g.cpu().numpy()
    g = geom(prefill.w)
    sample = [0, 39, 40, 44, 45, T // 2, T - 1]
    kv64 = bf16_f64(kv16[sample])
    for i, t in enumerate(sample):
        _, exp_h, exp_g = O.gate(g, kv64[i], int(win[t][0]), hidden[t], prefill.wq[0],
                                 prefill.wk[0])
        check_hidden(got[t], exp_h, f"token {t}")
        assert np.abs(gates[t] - exp_g).max() <= 1e-3
    assert np.array_equal(got[40:45], hidden[40:45])  # image rows untouched
