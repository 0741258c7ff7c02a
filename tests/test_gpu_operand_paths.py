"""GPU parity of the operand encodings a bind chooses, and of the gather's bounds check.

A bound layer feeds the tensor cores FP16 operands that hold the BF16 values
exactly when its table's E8M0 exponents span at most 23 values: each decoded
value is code x 2^(e - 127 + shift) with shift = 122 - smin for a span of at
most 12 and 112 - smin for a span of 13 to 22.  A wider span falls back to
BF16 operands by itself.  wkv is held as an FP16 copy scaled by 2^wkv_exp,
exact for every weight above 2^-28 of the largest; smaller weights round.
Generated tables span 119..127 and take only the first shift, so these tests
bind host-generated tables (synth.mxfp8_table) whose exponents span more, and
a wkv holding weights far below its largest.  The oracle reads the same host
tables and the exact BF16 weights.
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

TINY_ROWS = 6126        # primes 1009..1033
SMALL_BASE = 20_000     # full geometry over a small table: 24 primes above 20,000


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


def run_forward(s, win, hidden, staged):
    T = win.shape[0]
    ctx = s.model.ctx
    wsb = (eg.engram_forward_staged_workspace_bytes if staged else eg.engram_workspace_bytes)
    ws = torch.empty(max(16, wsb(ctx, T)), dtype=torch.uint8, device="cuda")
    d_h = to_dev(hidden)
    d_g = torch.full((T, s.w.hc), float("nan"), device="cuda")
    (eg.engram_forward_staged if staged else eg.engram_forward)(ctx, 0, to_dev(win), T, d_h,
                                                               ws, d_g)
    eg.engram_sync(ctx)
    return from_dev(d_h, np.uint16), d_g.cpu().numpy()


def gather_rows(s, win):
    T = win.shape[0]
    d_rows = torch.empty((T, s.w.nb), dtype=torch.int32, device="cuda")
    eg.engram_hash(s.model.ctx, 0, to_dev(win), T, d_rows)
    d_emb = torch.empty((T, s.w.K), dtype=torch.int16, device="cuda")
    eg.engram_gather_dequant(s.model.ctx, 0, d_rows, T, d_emb)
    eg.engram_sync(s.model.ctx)
    return from_dev(d_rows, np.uint32), from_dev(d_emb, np.uint16)


def check_layer_against_oracle(s, win, hidden, sample, what):
    rows, emb = gather_rows(s, win)
    ref = s.oracle_forward(0, win, hidden, sample, nthreads=16, want_e=True, want_h64=False)
    assert np.array_equal(rows[sample], ref["rows"]), what
    assert np.array_equal(emb[sample], ref["e"]), what  # dequantised rows, bit-exact
    for staged in (False, True):
        h, gates = run_forward(s, win, hidden, staged)
        check_hidden(h[sample], ref["h_bf16"], f"{what} staged={staged}")
        assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3, f"{what} staged={staged}"
        image = win[:, 0] == eg.DEAD
        assert np.array_equal(h[image], hidden[image]) and (gates[image] == 0).all()


# (scale_lo, scale_hi) -> operand path the bind must choose
SPANS = [
    ((115, 127), "fp16", 122 - 115),   # span 12: the first shift
    ((114, 127), "fp16", 112 - 114),   # span 13: the second shift
    ((105, 127), "fp16", 112 - 105),   # span 22: the widest FP16 span
    ((104, 127), "bf16", None),        # span 23: BF16 operands, chosen by the bind
]


@pytest.mark.parametrize("span,path,shift", SPANS, ids=lambda v: str(v))
def test_scale_span_selects_the_operand_path_tiny(span, path, shift):
    table = synth.mxfp8_table(TINY_ROWS, 32, 7, *span)
    s = setup_workload("tiny", tables={0: table})
    try:
        info = eg.engram_layer_info(s.model.ctx, 0)
        assert (info["scale_min"], info["scale_max"]) == span
        assert info["fp16_operands"] == (path == "fp16")
        if shift is not None:
            assert info["a_exp_shift"] == shift
        win, _, _ = prefill_windows(s, 3, 70, spans=[(0, 2), (50, 9)])
        hidden = synth.hidden_bf16(s.w, win.shape[0])
        check_layer_against_oracle(s, win, hidden, np.arange(win.shape[0]), f"tiny {span}")
    finally:
        s.close()


@pytest.mark.parametrize("span,path,shift", SPANS[1:], ids=lambda v: str(v))
def test_scale_span_selects_the_operand_path_full_geometry(span, path, shift):
    # 256-wide rows: the single fused kernel gathers whole rows (bucket gather)
    w = synth.WORKLOADS["prefill_2048"]
    rows = O.layer_params(geom(w), w.hash_seeds, [SMALL_BASE], 0).rows
    table = synth.mxfp8_table(rows, 256, 8, *span)
    s = setup_workload("prefill_2048", tables={0: table}, bucket_bases=[SMALL_BASE])
    try:
        info = eg.engram_layer_info(s.model.ctx, 0)
        assert (info["scale_min"], info["scale_max"]) == span
        assert info["fp16_operands"] == (path == "fp16")
        assert info["bucket_gather"] == (path == "fp16")
        if shift is not None:
            assert info["a_exp_shift"] == shift
        rng = np.random.default_rng(11)
        # 1,024 tokens fill the GPU (CTA pairs, no split); 300 run split K / stream K
        for T in (1024, 300):
            win, _, _ = prefill_windows(s, 2, T // 2, spans=[(100, 5)])
            hidden = synth.hidden_bf16(s.w, T)
            sample = np.unique(np.concatenate([[0, 1, 127, 128, 104, 105, T - 1],
                                               rng.integers(0, T, 25)]))
            check_layer_against_oracle(s, win, hidden, sample, f"full {span} T={T}")
    finally:
        s.close()


def test_wkv_weights_far_below_the_largest():
    # Some weights far below the largest: whole value rows and every 11th key
    # weight at 2^-44 .. 2^-34 (the FP16 copy, scaled by 2^wkv_exp, holds them
    # as subnormals that round or flush to zero).  kv stays within the fp32
    # bound plus the FP16 rounding of those weights; hidden and gates within the
    # usual tolerance of the oracle on the exact BF16 weights.
    w = synth.WORKLOADS["tiny"]
    W = synth.wkv_bf16(w).copy()
    Wf = bf16_f64(W)
    rng = np.random.default_rng(5)
    tiny_rows = np.arange(700, 712)          # value rows (the value is rows 512..767)
    mask = np.zeros(W.shape, bool)
    mask[tiny_rows] = True
    mask[:512, ::11] = True
    mag = np.ldexp(1.0 + rng.integers(0, 128, W.shape) / 128.0, rng.integers(-44, -34, W.shape))
    sign = rng.choice([-1.0, 1.0], W.shape)
    Wf = np.where(mask, sign * mag, Wf)
    W = synth.to_bf16_bits(Wf.astype(np.float32))
    assert np.array_equal(bf16_f64(W)[mask], Wf[mask])  # the tiny weights are exact in BF16
    s = setup_workload("tiny", wkv={0: W})
    try:
        info = eg.engram_layer_info(s.model.ctx, 0)
        assert info["fp16_operands"] == 1
        scale = 2.0 ** info["wkv_exp"]
        Wd = bf16_f64(W)
        W16 = (Wd * scale).astype(np.float16).astype(np.float64) / scale
        assert (W16[mask] != Wd[mask]).mean() > 0.5      # most tiny weights do round
        assert (W16[mask] == 0).any()
        big = np.abs(Wd) >= np.abs(Wd).max() * 2.0**-28   # exact above 2^-28 of the largest
        assert (W16[big] == Wd[big]).all()
        win, _, _ = prefill_windows(s, 2, 64, spans=[(10, 3)])
        T = win.shape[0]
        hidden = synth.hidden_bf16(s.w, T)
        d_kv = torch.full((T, s.w.N), float("nan"), device="cuda")
        eg.engram_project_windows(s.model.ctx, 0, to_dev(win), T, d_kv)
        eg.engram_sync(s.model.ctx)
        kv = d_kv.cpu().numpy()
        ref = s.oracle_forward(0, win, hidden, np.arange(T), nthreads=8, want_e=True,
                               want_kv=True)
        for t in range(T):
            e = bf16_f64(ref["e"][t])
            fp16_err = np.abs(e) @ np.abs(Wd - W16).T
            err = np.abs(kv[t].astype(np.float64) - ref["kv"][t])
            fp32 = s.w.K * 2.0**-24 * (np.abs(e) @ np.abs(Wd).T) + 1e-30
            assert (err <= fp32 + fp16_err).all(), t
            # rows without tiny weights: the plain fp32 bound
            clean = ~mask.any(axis=1)
            check_kv(kv[t][clean], ref["kv"][t][clean], W[clean], ref["e"][t], s.w.K, f"t {t}")
        for staged in (False, True):
            h, gates = run_forward(s, win, hidden, staged)
            check_hidden(h, ref["h_bf16"], f"tiny weights staged={staged}")
            assert np.abs(gates - ref["gates"]).max() <= 1e-3
    finally:
        s.close()


def test_gather_index_outside_the_table_sets_ebounds():
    # A row index equal to the row count lands on a spare row that the table
    # allocation holds past the bound rows, so even a broken guard would read
    # owned memory.  The gather must zero that slice, leave every other slice
    # as the oracle decodes it, and report ENGRAM_EBOUNDS once through
    # engram_sync, which clears the error word.
    table = synth.mxfp8_table(TINY_ROWS + 1, 32, 9, 119, 127)
    table[0][TINY_ROWS] = 0x38                   # the spare row: all 1.0
    s = setup_workload("tiny", tables={0: table})
    try:
        win, _, _ = prefill_windows(s, 1, 8)
        rows, _ = gather_rows(s, win)
        bad = rows.copy()
        bad[3, 2] = TINY_ROWS
        bad[5, 4] = eg.MASKED
        d_rows = to_dev(bad)
        d_emb = torch.full((8, s.w.K), -1, dtype=torch.int16, device="cuda")
        eg.engram_gather_dequant(s.model.ctx, 0, d_rows, 8, d_emb)
        with pytest.raises(eg.EngramError) as e:
            eg.engram_sync(s.model.ctx)
        assert e.value.status == eg.EBOUNDS
        emb = from_dev(d_emb, np.uint16).reshape(8, s.w.nb, 32)
        assert (emb[3, 2] == 0).all() and (emb[5, 4] == 0).all()
        g = geom(s.w)
        for t in range(8):
            ok = bad[t].copy()
            if t == 3:
                ok[2] = eg.MASKED                    # zeros, as a masked row
            assert np.array_equal(emb[t].reshape(-1), O.gather_table(g, *table, ok)), t
        # the error word was cleared: a valid call afterwards syncs cleanly
        eg.engram_gather_dequant(s.model.ctx, 0, to_dev(rows), 8, d_emb)
        eg.engram_sync(s.model.ctx)
    finally:
        s.close()
