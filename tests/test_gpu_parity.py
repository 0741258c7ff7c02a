"""GPU parity of every step against the CPU oracle, through the C ABI.

Integer and byte results (table contents, row indices, dequantised rows) must
be bit-exact; floating-point results follow the tolerances in helpers.py.
Sizes: the tiny workload in full (several tiles in N, ragged token counts in
M), and the 2,048-token prefill at full geometry (all indices, sampled rows
of the oracle's fp64 result).
"""
import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from golden_io import load_hash_worked
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


@pytest.fixture(scope="module")
def tiny_bf16():
    s = setup_workload("tiny", flags=eg.BIND_BF16_OPERANDS)
    yield s
    s.close()


def test_layer_info_selects_the_operand_path(tiny, tiny_bf16, prefill):
    for s in (tiny, prefill):
        info = eg.engram_layer_info(s.model.ctx, 0)
        assert info["bound"] == 1 and info["rows"] == s.model.rows(0)
        assert (info["scale_min"], info["scale_max"]) == (119, 127)  # table exponents
        assert info["fp16_operands"] == 1 and info["a_exp_shift"] == 3
        wmax = np.abs(bf16_f64(s.W[0])).max()
        assert 2.0**14 <= wmax * 2.0 ** info["wkv_exp"] <= 2.0**15
    assert eg.engram_layer_info(tiny_bf16.model.ctx, 0)["fp16_operands"] == 0


def gpu_rows(s, win, layer=0):
    T = win.shape[0]
    d_win = to_dev(win)
    d_rows = torch.empty((T, s.w.nb), dtype=torch.int32, device="cuda")
    eg.engram_hash(s.model.ctx, layer, d_win, T, d_rows)
    eg.engram_sync(s.model.ctx)
    return from_dev(d_rows, np.uint32), d_rows


def gpu_emb(s, d_rows, T, layer=0):
    d_emb = torch.empty((T, s.w.K), dtype=torch.int16, device="cuda")
    eg.engram_gather_dequant(s.model.ctx, layer, d_rows, T, d_emb)
    eg.engram_sync(s.model.ctx)
    return d_emb


# ---- a0: table contents --------------------------------------------------------------

def test_table_fill_tiny_whole_table(tiny):
    t = tiny.model.tensors[0]
    rows = tiny.model.rows(0)
    data = t["table"].cpu().numpy()[: rows * 32].reshape(rows, 32)
    scl = t["scales"].cpu().numpy()[:rows]
    for r in range(rows):
        c, s = O.table_row(t["table_seed"], r, 32)
        assert np.array_equal(data[r], c) and scl[r] == s[0], r


def test_table_fill_full_geometry_sampled(prefill):
    t = prefill.model.tensors[0]
    rows = prefill.model.rows(0)
    rng = np.random.default_rng(0)
    sample = np.concatenate([[0, 1, rows - 2, rows - 1], rng.integers(0, rows, 400)])
    data = t["table"].view(-1)
    scl = t["scales"].view(-1)
    for r in sample.tolist():
        c, s = O.table_row(t["table_seed"], r, 256)
        assert np.array_equal(data[r * 256:(r + 1) * 256].cpu().numpy(), c), r
        assert np.array_equal(scl[r * 8:(r + 1) * 8].cpu().numpy(), s), r


# ---- a2 / a3: hash and gather, bit-exact ------------------------------------------------

@pytest.mark.parametrize("sessions,per", [(1, 64), (3, 43), (1, 1)])
def test_hash_and_gather_tiny_bit_exact(tiny, sessions, per):
    win, _, _ = prefill_windows(tiny, sessions, per, spans=[(5, 3)] if per > 10 else [])
    T = win.shape[0]
    rows, d_rows = gpu_rows(tiny, win)
    g = geom(tiny.w)
    for t in range(T):
        ref = O.hash_rows(g, tiny.oparams[0], win[t])
        assert np.array_equal(rows[t], ref), t
    emb = from_dev(gpu_emb(tiny, d_rows, T), np.uint16)
    for t in range(T):
        assert np.array_equal(emb[t], O.gather(g, tiny.w.table_seeds[0], rows[t])), t


def test_hash_full_geometry_bit_exact(prefill):
    win, _, _ = prefill_windows(prefill, 1, 2048)
    rows, d_rows = gpu_rows(prefill, win)
    g = geom(prefill.w)
    for t in range(2048):
        assert np.array_equal(rows[t], O.hash_rows(g, prefill.oparams[0], win[t])), t
    # every index inside its bucket
    p = prefill.oparams[0]
    for b in range(24):
        assert (rows[:, b] >= p.offset[b]).all() and (rows[:, b] < p.offset[b] + p.prime[b]).all()
    emb = from_dev(gpu_emb(prefill, d_rows, 2048), np.uint16)
    rng = np.random.default_rng(1)
    for t in [0, 1, 2, 3, 2047] + rng.integers(0, 2048, 59).tolist():
        assert np.array_equal(emb[t], O.gather(g, prefill.w.table_seeds[0], rows[t])), t


def test_hash_hand_worked_values_on_gpu():
    # the hand-worked fixture (two general multiplier tables over primes
    # 1009..1033) through engram_hash: products above 2^32, products that wrap
    # 2^64 and a DEAD slot, against values worked out by hand
    primes, offsets, tables, cases = load_hash_worked()
    tmap = np.arange(4096, dtype=np.uint32) % 1000
    ctx = eg.engram_ctx_create(4096, 1000, tmap, [1], [1000], heads=2, row_dim=32, hc=1, d=256)
    try:
        _, prime, offset, _ = eg.engram_layer_params(ctx, 0, 6)
        assert np.array_equal(prime, primes) and np.array_equal(offset, offsets)
        for name in sorted(tables):
            eg.engram_layer_set_multipliers(ctx, 0, tables[name])
            mine = [(w, r) for t, w, r in cases if t == name]
            # a ragged batch: the worked windows repeated 37 times
            win = np.array([w for w, _ in mine] * 37, np.uint32)
            want = np.array([r for _, r in mine] * 37, np.uint32)
            d_rows = torch.empty((len(win), 6), dtype=torch.int32, device="cuda")
            eg.engram_hash(ctx, 0, to_dev(win), len(win), d_rows)
            torch.cuda.synchronize()
            assert np.array_equal(from_dev(d_rows, np.uint32), want), name
    finally:
        eg.engram_ctx_destroy(ctx)


# ---- a4: projection ---------------------------------------------------------------------

@pytest.mark.parametrize("sessions,per", [(1, 64), (3, 43), (1, 1), (2, 100)])
def test_project_tiny(tiny, sessions, per):
    win, _, _ = prefill_windows(tiny, sessions, per)
    T = win.shape[0]
    rows, d_rows = gpu_rows(tiny, win)
    d_emb = gpu_emb(tiny, d_rows, T)
    d_kv = torch.empty((T, tiny.w.N), dtype=torch.float32, device="cuda")
    eg.engram_project(tiny.model.ctx, 0, d_emb, T, d_kv)
    eg.engram_sync(tiny.model.ctx)
    kv = d_kv.cpu().numpy()
    g = geom(tiny.w)
    for t in range(T):
        e = O.gather(g, tiny.w.table_seeds[0], O.hash_rows(g, tiny.oparams[0], win[t]))
        ref = O.project(g, tiny.W[0], e)
        check_kv(kv[t], ref, tiny.W[0], e, tiny.w.K, f"token {t}")
    # the fused hash+gather+projection: FP16 operands hold the same values and
    # the scalings are powers of two, so kv matches the unfused BF16 GEMM
    d_kv2 = torch.full_like(d_kv, float("nan"))
    eg.engram_project_windows(tiny.model.ctx, 0, to_dev(win), T, d_kv2)
    eg.engram_sync(tiny.model.ctx)
    kv2 = d_kv2.cpu().numpy()
    for t in range(T):
        e = O.gather(g, tiny.w.table_seeds[0], O.hash_rows(g, tiny.oparams[0], win[t]))
        check_kv(kv2[t], O.project(g, tiny.W[0], e), tiny.W[0], e, tiny.w.K, f"fused token {t}")


def test_project_full_geometry_sampled(prefill):
    win, _, _ = prefill_windows(prefill, 1, 2048)
    T = 2048
    d_kv = torch.empty((T, prefill.w.N), dtype=torch.float32, device="cuda")
    eg.engram_project_windows(prefill.model.ctx, 0, to_dev(win), T, d_kv)
    eg.engram_sync(prefill.model.ctx)
    g = geom(prefill.w)
    sample = [0, 127, 128, 2047, 1000, 1500]
    ref = O.forward(g, prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0], prefill.wq[0],
                    prefill.wk[0], win, synth.hidden_bf16(prefill.w, T), np.array(sample),
                    nthreads=8, want_e=True, want_kv=True, want_h64=False)
    for i, t in enumerate(sample):
        check_kv(d_kv[t].cpu().numpy(), ref["kv"][i], prefill.W[0], ref["e"][i], prefill.w.K,
                 f"token {t}")


# ---- a5: the gate alone, on the oracle's kv -------------------------------------------

def test_gate_alone_on_oracle_kv(tiny):
    win, _, _ = prefill_windows(tiny, 1, 64, spans=[(30, 4)])
    T = 64
    hidden = synth.hidden_bf16(tiny.w, T)
    g = geom(tiny.w)
    ref = O.forward(g, tiny.w.table_seeds[0], tiny.oparams[0], tiny.W[0], tiny.wq[0], tiny.wk[0],
                    win, hidden, np.arange(T), want_kv=True, want_h64=False)
    kv32 = ref["kv"].astype(np.float32)
    exp_h = np.zeros_like(ref["h_bf16"])
    exp_g = np.zeros_like(ref["gates"])
    for t in range(T):
        _, exp_h[t], exp_g[t] = O.gate(g, kv32[t].astype(np.float64), int(win[t][0]), hidden[t],
                                       tiny.wq[0], tiny.wk[0])
    d_h = to_dev(hidden)
    d_g = torch.empty((T, tiny.w.hc), dtype=torch.float32, device="cuda")
    eg.engram_gate(tiny.model.ctx, 0, torch.from_numpy(kv32).cuda(), to_dev(win), T, d_h, d_g)
    eg.engram_sync(tiny.model.ctx)
    check_hidden(from_dev(d_h, np.uint16), exp_h, "gate")
    assert np.abs(d_g.cpu().numpy() - exp_g).max() <= 1e-3
    assert np.array_equal(from_dev(d_h, np.uint16)[30:34], hidden[30:34])  # image rows


# ---- a7: the fused forward --------------------------------------------------------------

def run_forward(s, win, hidden, layer=0, staged=False):
    T = win.shape[0]
    d_h = to_dev(hidden)
    ws = (eg.engram_forward_staged_workspace_bytes if staged else eg.engram_workspace_bytes)
    d_ws = torch.empty(max(16, ws(s.model.ctx, T)), dtype=torch.uint8, device="cuda")
    d_g = torch.full((T, s.w.hc), float("nan"), dtype=torch.float32, device="cuda")
    fwd = eg.engram_forward_staged if staged else eg.engram_forward
    fwd(s.model.ctx, layer, to_dev(win), T, d_h, d_ws, d_g)
    eg.engram_sync(s.model.ctx)
    return from_dev(d_h, np.uint16), d_g.cpu().numpy()


@pytest.mark.parametrize("entry", ["fused", "staged"])
@pytest.mark.parametrize("path", ["fp16", "bf16"])
@pytest.mark.parametrize("sessions,per,spans", [(1, 64, [(20, 4)]), (3, 70, [(0, 2), (50, 9)]),
                                                (1, 1, []), (2, 129, [(128, 1)])])
def test_forward_tiny_all_tokens(tiny, tiny_bf16, path, entry, sessions, per, spans):
    tiny = tiny if path == "fp16" else tiny_bf16
    win, _, _ = prefill_windows(tiny, sessions, per, spans)
    T = win.shape[0]
    hidden = synth.hidden_bf16(tiny.w, T)
    h, gates = run_forward(tiny, win, hidden, staged=entry == "staged")
    ref = O.forward(geom(tiny.w), tiny.w.table_seeds[0], tiny.oparams[0], tiny.W[0], tiny.wq[0],
                    tiny.wk[0], win, hidden, np.arange(T), nthreads=4)
    check_hidden(h, ref["h_bf16"], "forward")
    assert np.abs(gates - ref["gates"]).max() <= 1e-3
    image = win[:, 0] == eg.DEAD
    assert np.array_equal(h[image], hidden[image])
    assert (gates[image] == 0).all()
    # rows whose every n-gram is masked keep their hidden bit for bit
    allmasked = (win[:, 1] == eg.DEAD) & ~image
    assert np.array_equal(h[allmasked], hidden[allmasked])


@pytest.fixture(scope="module")
def prefill_ref(prefill):
    """The oracle's step on every token of the 2,048-token prefill (16 threads)."""
    win, _, _ = prefill_windows(prefill, 1, 2048)
    hidden = synth.hidden_bf16(prefill.w, 2048)
    ref = O.forward(geom(prefill.w), prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0],
                    prefill.wq[0], prefill.wk[0], win, hidden, np.arange(2048), nthreads=16,
                    want_e=True, want_h64=False)
    return win, hidden, ref


def test_gather_full_geometry_every_row(prefill, prefill_ref):
    # every dequantised row of the 2,048 tokens (24 x 256 values each), bit-exact
    win, _, ref = prefill_ref
    rows, d_rows = gpu_rows(prefill, win)
    assert np.array_equal(rows, ref["rows"])
    emb = from_dev(gpu_emb(prefill, d_rows, 2048), np.uint16)
    assert np.array_equal(emb, ref["e"])


@pytest.mark.parametrize("entry", ["fused", "staged"])
def test_forward_full_geometry_every_token(prefill, prefill_ref, entry):
    # hidden and gates of all 2,048 tokens against the oracle
    win, hidden, ref = prefill_ref
    T = 2048
    h, gates = run_forward(prefill, win, hidden, staged=entry == "staged")
    check_hidden(h, ref["h_bf16"], f"forward 2048 {entry}")
    assert np.abs(gates - ref["gates"]).max() <= 1e-3


def test_prepass_and_gate_full_geometry_every_token(prefill, prefill_ref):
    # the hidden-independent projection (a2-a4 fused) then the gate kernel
    win, hidden, ref = prefill_ref
    T = 2048
    d_kv = torch.empty((T, prefill.w.N), dtype=torch.float32, device="cuda")
    eg.engram_project_windows(prefill.model.ctx, 0, to_dev(win), T, d_kv)
    d_h = to_dev(hidden)
    d_g = torch.empty((T, prefill.w.hc), dtype=torch.float32, device="cuda")
    eg.engram_gate(prefill.model.ctx, 0, d_kv, to_dev(win), T, d_h, d_g)
    eg.engram_sync(prefill.model.ctx)
    check_hidden(from_dev(d_h, np.uint16), ref["h_bf16"], "project_windows + gate")
    assert np.abs(d_g.cpu().numpy() - ref["gates"]).max() <= 1e-3


@pytest.mark.parametrize("entry", ["fused", "staged"])
@pytest.mark.parametrize("T", [1, 77, 256, 300, 600])
def test_small_batches_split_k(prefill, entry, T):
    # batches whose output tiles do not fill the GPU twice split K over
    # several CTAs; the last split of each tile quadrant sums the parked
    # partials and runs the gate epilogue
    win, _, _ = prefill_windows(prefill, 1, T, spans=[(T // 2, 3)] if T > 8 else [])
    hidden = synth.hidden_bf16(prefill.w, T)
    h, gates = run_forward(prefill, win, hidden, staged=entry == "staged")
    sample = np.unique(np.array([0, T // 2 - 1, T // 2, T // 2 + 3, 127, 128, T - 2, T - 1])
                       .clip(0, T - 1))
    ref = O.forward(geom(prefill.w), prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0],
                    prefill.wq[0], prefill.wk[0], win, hidden, sample, nthreads=8)
    check_hidden(h[sample], ref["h_bf16"], f"{entry} split-K T={T}")
    assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3
    image = win[:, 0] == eg.DEAD
    assert np.array_equal(h[image], hidden[image]) and (gates[image] == 0).all()
    # every token against the unsplit projection and the gate kernel
    d_kv = torch.empty((T, prefill.w.N), dtype=torch.float32, device="cuda")
    eg.engram_project_windows(prefill.model.ctx, 0, to_dev(win), T, d_kv)
    d_h = to_dev(hidden)
    d_g = torch.empty((T, prefill.w.hc), dtype=torch.float32, device="cuda")
    eg.engram_gate(prefill.model.ctx, 0, d_kv, to_dev(win), T, d_h, d_g)
    eg.engram_sync(prefill.model.ctx)
    check_hidden(h, from_dev(d_h, np.uint16), f"{entry} split-K vs unsplit chain")
    assert np.abs(gates - d_g.cpu().numpy()).max() <= 1e-3
    # the same inputs give the same bits on a second call (the reduction order
    # does not depend on which split arrives last)
    h2, g2 = run_forward(prefill, win, hidden, staged=entry == "staged")
    assert np.array_equal(h, h2) and np.array_equal(gates, g2)


@pytest.mark.parametrize("T", [77, 256, 2048])
def test_staged_in_two_calls_matches_one_call(prefill, T):
    # engram_stage_rows + engram_forward_staged_rows is engram_forward_staged
    # split in two: the same kernels on the same inputs, bit for bit; the two
    # steps of two batches are interleaved on two streams and two workspaces
    win, _, _ = prefill_windows(prefill, 1, T, spans=[(T // 3, 5)])
    win2, _, _ = prefill_windows(prefill, 2, T // 2 + 1)
    win2 = win2[:T]
    hidden = synth.hidden_bf16(prefill.w, T)
    ctx = prefill.model.ctx
    ref1, g1 = run_forward(prefill, win, hidden, staged=True)
    ref2, g2 = run_forward(prefill, win2, hidden, staged=True)
    wsb = eg.engram_forward_staged_workspace_bytes(ctx, T)
    ws = [torch.empty(wsb, dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_w = [to_dev(win), to_dev(win2)]
    d_h = [to_dev(hidden), to_dev(hidden)]
    d_g = [torch.full((T, prefill.w.hc), float("nan"), device="cuda") for _ in range(2)]
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    staged = [torch.cuda.Event() for _ in range(2)]
    side.wait_stream(main)
    for i in range(2):
        eg.engram_stage_rows(ctx, 0, d_w[i], T, ws[i], side.cuda_stream)
        staged[i].record(side)
    for i in range(2):
        main.wait_event(staged[i])
        eg.engram_forward_staged_rows(ctx, 0, d_w[i], T, d_h[i], ws[i], d_g[i], main.cuda_stream)
    eg.engram_sync(ctx)
    assert np.array_equal(from_dev(d_h[0], np.uint16), ref1)
    assert np.array_equal(from_dev(d_h[1], np.uint16), ref2)
    assert np.array_equal(d_g[0].cpu().numpy(), g1) and np.array_equal(d_g[1].cpu().numpy(), g2)


@pytest.mark.parametrize("flags", [0, eg.BIND_BF16_OPERANDS])
def test_staged_pairs_with_an_odd_block_count(flags):
    # 2,176 tokens = 17 blocks of 128: the last CTA pair has no second block,
    # its odd CTA reads zero-filled operand rows and writes nothing
    s = setup_workload("prefill_2048", flags=flags)
    try:
        T = 2176
        win, _, _ = prefill_windows(s, 2, T // 2, spans=[(500, 6)])
        hidden = synth.hidden_bf16(s.w, T)
        h, gates = run_forward(s, win, hidden, staged=True)
        sample = np.array([0, 255, 256, 2047, 2048, 2049, 2100, 2175, 500, 506, 1588])
        ref = O.forward(geom(s.w), s.w.table_seeds[0], s.oparams[0], s.W[0], s.wq[0], s.wk[0],
                        win, hidden, sample, nthreads=8)
        check_hidden(h[sample], ref["h_bf16"], f"2176 tokens flags={flags}")
        assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3
        image = win[:, 0] == eg.DEAD
        assert image.sum() == 12 and np.array_equal(h[image], hidden[image])
    finally:
        s.close()


@pytest.mark.parametrize("T,span", [(2048, (256, 768)), (2048, (0, 2048)), (5400, (512, 3072)),
                                    (5400, (300, 4700)), (5400, (0, 5400)), (5000, (4800, 100))])
def test_staged_with_long_image_spans(prefill, T, span):
    # A batch longer than one chunk (about 4,864 tokens here) runs chunk by
    # chunk, and each chunk's GEMM runs only its 256-token units that hold a
    # text row (those of image rows only get no items and their gates are
    # written as 0); a single chunk runs every unit, and a short last chunk
    # (136 tokens at 5,000) runs the small-batch path with stream K.  Either
    # way every row matches the oracle: image rows bit for bit with gates 0,
    # text rows (the first after a span too) within tolerance.
    win, _, _ = prefill_windows(prefill, 1, T, spans=[span])
    hidden = synth.hidden_bf16(prefill.w, T)
    h, gates = run_forward(prefill, win, hidden, staged=True)
    image = win[:, 0] == eg.DEAD
    assert image.sum() == min(span[1], T - span[0])
    assert np.array_equal(h[image], hidden[image]) and (gates[image] == 0).all()
    assert not np.isnan(gates).any()
    lo, n = span
    sample = np.unique(np.clip(np.array([0, lo - 1, lo, lo + 255, lo + n - 1, lo + n, lo + n + 1,
                                         lo + n + 2, T - 1, 1500, 100, 4863, 4864, 5000]), 0, T - 1))
    ref = O.forward(geom(prefill.w), prefill.w.table_seeds[0], prefill.oparams[0], prefill.W[0],
                    prefill.wq[0], prefill.wk[0], win, hidden, sample, nthreads=16)
    check_hidden(h[sample], ref["h_bf16"], f"image span {span}")
    assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3


def test_forward_edge_cases(tiny):
    ctx = tiny.model.ctx
    eg.engram_forward(ctx, 0, None, 0, None, None)  # T = 0
    win, _, _ = prefill_windows(tiny, 1, 40, spans=[(0, 40)])  # all image rows
    hidden = synth.hidden_bf16(tiny.w, 40)
    h, gates = run_forward(tiny, win, hidden)
    assert np.array_equal(h, hidden) and (gates == 0).all()


def test_forward_full_geometry_bf16_operands_sampled():
    s = setup_workload("prefill_2048", flags=eg.BIND_BF16_OPERANDS)
    try:
        assert eg.engram_layer_info(s.model.ctx, 0)["fp16_operands"] == 0
        win, _, _ = prefill_windows(s, 1, 2048, spans=[(1000, 100)])
        hidden = synth.hidden_bf16(s.w, 2048)
        h, gates = run_forward(s, win, hidden)
        sample = np.array([0, 127, 128, 999, 1000, 1100, 1101, 1102, 2047])
        ref = O.forward(geom(s.w), s.w.table_seeds[0], s.oparams[0], s.W[0], s.wq[0], s.wk[0],
                        win, hidden, sample, nthreads=8)
        check_hidden(h[sample], ref["h_bf16"], "forward 2048 bf16 operands")
        assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3
    finally:
        s.close()


def test_bounded_wait_times_out_and_the_context_stays_usable(tiny):
    # the GEMM's operand loads are withheld, so the tensor-core issuer's wait
    # for them runs out after the wait limit; the call reports ETIMEOUT
    ctx = tiny.model.ctx
    win, _, _ = prefill_windows(tiny, 1, 64)
    hidden = synth.hidden_bf16(tiny.w, 64)
    eg.engram_ctx_set_wait_limit(ctx, 50_000_000)  # 50 ms
    eg.engram_debug_starve_operand(ctx, True)
    d_h = to_dev(hidden)
    ws = torch.empty(max(16, eg.engram_workspace_bytes(ctx, 64)), dtype=torch.uint8, device="cuda")
    import time

    t0 = time.time()
    eg.engram_forward(ctx, 0, to_dev(win), 64, d_h, ws)
    with pytest.raises(eg.EngramError) as e:
        eg.engram_sync(ctx)
    assert e.value.status == eg.ETIMEOUT
    assert time.time() - t0 < 5.0
    eg.engram_debug_starve_operand(ctx, False)
    eg.engram_ctx_set_wait_limit(ctx, 4_000_000_000)
    h, gates = run_forward(tiny, win, hidden)
    ref = O.forward(geom(tiny.w), tiny.w.table_seeds[0], tiny.oparams[0], tiny.W[0], tiny.wq[0],
                    tiny.wk[0], win, hidden, np.arange(64))
    check_hidden(h, ref["h_bf16"], "after a time-out")
