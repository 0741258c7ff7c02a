"""Parity at the full sizes of the decode, long-prefill and host-table workloads.

Indices and table rows are checked bit-exact on every position the oracle
can afford; hidden states and gates on sampled positions.  The same windows
feed every layer of the two-layer workload: tokens enter the history once.
"""
import dataclasses

import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from helpers import (check_hidden, from_dev, geom, setup_workload, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


def forward(s, win, hidden, layer, staged):
    T = win.shape[0]
    ctx = s.model.ctx
    ws_bytes = (eg.engram_forward_staged_workspace_bytes if staged else eg.engram_workspace_bytes)
    ws = torch.empty(max(16, ws_bytes(ctx, T)), dtype=torch.uint8, device="cuda")
    d_h = to_dev(hidden)
    d_g = torch.full((T, s.w.hc), float("nan"), device="cuda")
    (eg.engram_forward_staged if staged else eg.engram_forward)(ctx, layer, to_dev(win), T, d_h,
                                                               ws, d_g)
    eg.engram_sync(ctx)
    return from_dev(d_h, np.uint16), d_g.cpu().numpy()


def check_sample(s, layer, win, hidden, h, gates, sample, what):
    ref = O.forward(geom(s.w), s.w.table_seeds[layer], s.oparams[layer], s.W[layer], s.wq[layer],
                    s.wk[layer], win, hidden, np.asarray(sample), nthreads=16)
    check_hidden(h[sample], ref["h_bf16"], what)
    assert np.abs(gates[sample] - ref["gates"]).max() <= 1e-3, what
    return ref


def test_decode_256_sessions_on_the_384m_row_table():
    s = setup_workload("decode_256")
    try:
        w = s.w
        assert s.model.rows(0) == 384_006_168
        S = w.sessions
        streams = np.stack([synth.session_tokens(w, i, w.history + 3) for i in range(S)])
        sess = [eg.engram_session_create(s.model.ctx) for _ in range(S)]
        for i, ss in enumerate(sess):
            eg.engram_session_append(ss, streams[i, :w.history])
        hidden = synth.hidden_bf16(w, S)
        g = geom(w)
        for step in range(3):
            win = eg.engram_batch_append(sess, streams[:, w.history + step])
            # every session's window equals the oracle's window of its whole stream
            for i in range(0, S, 17):
                ref_w = O.windows(g, s.tmap, streams[i, :w.history + step + 1])[-1]
                assert np.array_equal(win[i], ref_w)
            # every row index of the step, bit-exact
            d_rows = torch.empty((S, w.nb), dtype=torch.int32, device="cuda")
            eg.engram_hash(s.model.ctx, 0, to_dev(win), S, d_rows)
            rows = from_dev(d_rows, np.uint32)
            for i in range(S):
                assert np.array_equal(rows[i], O.hash_rows(g, s.oparams[0], win[i])), (step, i)
            for staged in (False, True):
                h, gates = forward(s, win, hidden, 0, staged)
                check_sample(s, 0, win, hidden, h, gates, [0, 1, 100, 255, 128 + step],
                             f"decode step {step} staged={staged}")
            hidden = h
        for ss in sess:
            eg.engram_session_destroy(ss)
    finally:
        s.close()


def test_long_prefill_two_layers_one_history():
    s = setup_workload("prefill_50k_2layer")
    try:
        w = s.w
        T = w.tokens_per_session
        toks = synth.session_tokens(w, 0, T)
        im = synth.image_flags(T, w.image_spans)
        sess = eg.engram_session_create(s.model.ctx)
        win = eg.engram_session_append(sess, toks, im)  # appended once, used by both layers
        eg.engram_session_destroy(sess)
        g = geom(w)
        assert np.array_equal(win, O.windows(g, s.tmap, toks, im))
        hidden = synth.hidden_bf16(w, T)
        spans = [st for st, _ in w.image_spans]
        sample = sorted({0, 1, 2, 3, T - 1} | {p + d for p in spans for d in (-1, 0, 1023, 1024, 1025, 1026)}
                        | set(np.random.default_rng(3).integers(0, T, 6).tolist()))
        for layer in range(2):
            p = s.oparams[layer]
            # both layers hash the same windows with their own parameters
            d_rows = torch.empty((T, w.nb), dtype=torch.int32, device="cuda")
            eg.engram_hash(s.model.ctx, layer, to_dev(win), T, d_rows)
            eg.engram_sync(s.model.ctx)
            rows = from_dev(d_rows, np.uint32)
            for t in sample:
                assert np.array_equal(rows[t], O.hash_rows(g, p, win[t])), (layer, t)
            for staged in (True, False):
                h, gates = forward(s, win, hidden, layer, staged)
                ref = check_sample(s, layer, win, hidden, h, gates, sample,
                                   f"layer {layer} staged={staged}")
                image = win[:, 0] == eg.DEAD
                assert image.sum() == 3 * 1024
                assert np.array_equal(h[image], hidden[image])
        assert not np.array_equal(s.oparams[0].prime, s.oparams[1].prime)
    finally:
        s.close()


def test_host_table_read_through_uva():
    # the 384M-row table would pin 101 GB of host memory; pinned memory cannot
    # be paged out, so the test keeps well inside the host's RAM: 64M rows
    with open("/proc/meminfo") as f:
        info = {ln.split(":")[0]: int(ln.split()[1]) * 1024 for ln in f if ":" in ln}
    avail = info.get("MemAvailable", 0)
    if avail < 48 * 2**30:
        pytest.skip(f"only {avail / 2**30:.0f} GB of host memory available")
    s = setup_workload("host_table_8x1024", host_table=True, bucket_bases=[2_666_666])
    try:
        w = s.w
        t = s.model.tensors[0]
        assert not t["table"].is_cuda and t["table"].is_pinned()
        T = w.sessions * w.tokens_per_session
        wins = []
        for i in range(w.sessions):
            ss = eg.engram_session_create(s.model.ctx)
            wins.append(eg.engram_session_append(ss, synth.session_tokens(w, i, w.tokens_per_session)))
            eg.engram_session_destroy(ss)
        win = np.concatenate(wins)
        hidden = synth.hidden_bf16(w, T)
        # table contents written through UVA by the fill kernel
        for r in [0, 1, s.model.rows(0) - 1, 31_415_926]:
            c, sc = O.table_row(w.table_seeds[0], r, 256)
            assert np.array_equal(t["table"][r * 256:(r + 1) * 256].numpy(), c)
            assert np.array_equal(t["scales"][r * 8:(r + 1) * 8].numpy(), sc)
        # the unfused gather through UVA, bit-exact
        g = geom(w)
        d_rows = torch.empty((T, w.nb), dtype=torch.int32, device="cuda")
        eg.engram_hash(s.model.ctx, 0, to_dev(win), T, d_rows)
        d_emb = torch.empty((T, w.K), dtype=torch.int16, device="cuda")
        eg.engram_gather_dequant(s.model.ctx, 0, d_rows, T, d_emb)
        eg.engram_sync(s.model.ctx)
        rows, emb = from_dev(d_rows, np.uint32), from_dev(d_emb, np.uint16)
        for tt in [0, 1023, 1024, 8191, 4000]:
            assert np.array_equal(emb[tt], O.gather(g, w.table_seeds[0], rows[tt]))
        for staged in (True, False):
            h, gates = forward(s, win, hidden, 0, staged)
            check_sample(s, 0, win, hidden, h, gates, [0, 1023, 1024, 5000, 8191],
                         f"host table staged={staged}")
    finally:
        s.close()
