"""engram_forward_noalloc against engram_forward, through the C ABI.

engram_forward_noalloc serves callers that cannot allocate device memory: a
serving engine that reserves the GPU's memory for its own pools, or a plugin
host that forbids its plugins to allocate.  It runs the same fused forward but
keeps its scratch in the library's built-in device buffer instead of a
caller-provided workspace.  Its results must match engram_forward's on the
same inputs, call after call (the buffer keeps the previous call's contents,
and nothing it leaves behind may leak into the next result).

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import re

import numpy as np
import pytest
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from helpers import check_hidden, from_dev, prefill_windows, setup_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()
    assert torch.cuda.is_available()


def forward_both(s, win, hidden):
    """(hidden, gates) of engram_forward with its own workspace, and of the no-alloc call."""
    T = win.shape[0]
    ctx = s.model.ctx
    d_win = to_dev(win)
    h_ref, h_new = to_dev(hidden), to_dev(hidden)
    g_ref = torch.full((T, s.w.hc), float("nan"), device="cuda")
    g_new = torch.full((T, s.w.hc), float("nan"), device="cuda")
    ws = torch.empty(max(16, eg.engram_workspace_bytes(ctx, T)), dtype=torch.uint8, device="cuda")
    eg.engram_forward(ctx, 0, d_win, T, h_ref, ws, g_ref)
    eg.engram_forward_noalloc(ctx, 0, d_win, T, h_new, g_new)
    eg.engram_sync(ctx)
    return (from_dev(h_ref, np.uint16), g_ref.cpu().numpy(), from_dev(h_new, np.uint16),
            g_new.cpu().numpy())


@pytest.mark.parametrize("name,sessions,per,spans", [
    ("tiny", 2, 97, [(10, 6)]),
    ("prefill_2048", 1, 2048, [(300, 64)]),
])
def test_noalloc_matches_forward_on_two_calls_in_a_row(name, sessions, per, spans):
    s = setup_workload(name)
    try:
        for call in range(2):
            # a different batch per call: the second call runs over the first's scratch
            win, _, _ = prefill_windows(s, sessions, per if call == 0 else per - 37, spans)
            hidden = synth.normal_bf16((win.shape[0], s.w.hc, s.w.d), 1.0, 5, 900 + call)
            h_ref, g_ref, h_new, g_new = forward_both(s, win, hidden)
            check_hidden(h_new, h_ref, f"{name} call {call}")
            assert np.abs(g_new - g_ref).max() <= 1e-3
            image = win[:, 0] == eg.DEAD
            assert np.array_equal(h_new[image], hidden[image])
    finally:
        s.close()


def stated_limit(ctx):
    """The largest batch the call accepts, as its own rejection message states it."""
    with pytest.raises(eg.EngramError) as e:
        eg.engram_forward_noalloc(ctx, 0, 16, 1 << 24, 16)  # rejected before any launch
    assert e.value.status == eg.EINVAL and "8 MiB" in e.value.message
    return int(re.search(r"at most (\d+) tokens", e.value.message).group(1))


def test_noalloc_rejects_batches_above_its_buffer():
    s = setup_workload("tiny")
    try:
        ctx = s.model.ctx
        limit = stated_limit(ctx)
        # rejected before any pointer is touched or any kernel launched
        with pytest.raises(eg.EngramError) as e:
            eg.engram_forward_noalloc(ctx, 0, 16, limit + 1, 16)
        assert e.value.status == eg.EINVAL
        # a bad layer is reported as such, whatever the batch size
        with pytest.raises(eg.EngramError) as e:
            eg.engram_forward_noalloc(ctx, 7, 16, 1 << 24, 16)
        assert e.value.status == eg.EINVAL and "layer" in e.value.message
        eg.engram_forward_noalloc(ctx, 0, None, 0, None)  # T = 0: nothing to do
    finally:
        s.close()


def test_noalloc_at_its_size_limit_full_geometry():
    # the largest accepted batch (the buffer nearly full, the tile counters at
    # its end) against engram_forward; one token more is rejected
    s = setup_workload("prefill_2048")
    try:
        ctx = s.model.ctx
        T = stated_limit(ctx)
        assert T == 8592  # hc 4, d 5,120
        per = (T + 3) // 4
        win, _, _ = prefill_windows(s, 4, per, [(500, 7)])
        win = win[:T]
        for call in range(2):
            hidden = synth.normal_bf16((T, s.w.hc, s.w.d), 1.0, 6, 910 + call)
            h_ref, g_ref, h_new, g_new = forward_both(s, win, hidden)
            check_hidden(h_new, h_ref, f"{T} tokens, call {call}")
            assert np.abs(g_new - g_ref).max() <= 1e-3
        with pytest.raises(eg.EngramError) as e:
            eg.engram_forward_noalloc(ctx, 0, to_dev(win[:1]), T + 1, 16)
        assert e.value.status == eg.EINVAL
    finally:
        s.close()
