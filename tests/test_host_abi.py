"""Host-side tests of the C ABI (no GPU): exports, validation, parameters, sessions.

The library's hash parameters come from its own code (Miller-Rabin primes and a
host Philox); the oracle's from trial division and its own Philox.  Both follow
the same reading of the pages and must agree exactly.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from engram_gram_conditional_gb300 import build

    build.build()
    O.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "engram.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(engram_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 20
    L = eg.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(eg.EXPORTS) == names


def tiny_ctx(**kw):
    w = synth.WORKLOADS["tiny"]
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    args = dict(min_n=2, max_n=4, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d)
    args.update(kw)
    return eg.engram_ctx_create(w.vocab, w.vc, tmap, w.hash_seeds, w.bucket_bases, **args), tmap


@pytest.mark.parametrize("bad", [
    dict(row_dim=48), dict(heads=0), dict(heads=9), dict(max_n=5), dict(min_n=3, max_n=2),
    dict(hc=0), dict(d=200), dict(pad_cid=1000), dict(min_n=2, max_n=2, heads=1, row_dim=32),
])
def test_ctx_create_rejects_bad_geometry(bad):
    with pytest.raises(eg.EngramError) as e:
        tiny_ctx(**bad)
    assert e.value.status == eg.EINVAL


def test_ctx_create_rejects_map_outside_vc():
    tmap = np.zeros(16, np.uint32)
    tmap[3] = 8
    with pytest.raises(eg.EngramError) as e:
        eg.engram_ctx_create(16, 8, tmap, [1], [100], heads=1, row_dim=64, hc=1, d=256)
    assert e.value.status == eg.EINVAL


@pytest.mark.parametrize("name", ["tiny", "prefill_2048", "prefill_50k_2layer", "decode_256"])
def test_layer_params_match_the_oracle(name):
    w = synth.WORKLOADS[name]
    tmap = np.zeros(w.vocab, np.uint32)
    ctx = eg.engram_ctx_create(w.vocab, w.vc, tmap, w.hash_seeds, w.bucket_bases, heads=w.heads,
                               row_dim=w.row_dim, hc=w.hc, d=w.d)
    g = O.Geom(vocab=w.vocab, vc=w.vc, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d)
    for layer in range(len(w.hash_seeds)):
        mult, prime, offset, rows = eg.engram_layer_params(ctx, layer, w.nb)
        ref = O.layer_params(g, w.hash_seeds, w.bucket_bases, layer)
        assert np.array_equal(mult, ref.mult)
        assert np.array_equal(prime, ref.prime)
        assert np.array_equal(offset, ref.offset)
        assert rows == ref.rows
    eg.engram_ctx_destroy(ctx)


def test_layer_params_reproduce_the_printed_row_counts():
    tmap = np.zeros(129_280, np.uint32)
    ctx = eg.engram_ctx_create(129_280, 100_000, tmap, [1, 14], [16_000_000, 16_000_000])
    assert eg.engram_layer_params(ctx, 0, 24)[3] == 384_006_168
    assert eg.engram_layer_params(ctx, 1, 24)[3] == 384_016_682
    eg.engram_ctx_destroy(ctx)


def test_set_multipliers_and_layer_range():
    ctx, _ = tiny_ctx()
    m = (np.arange(24, dtype=np.uint64).reshape(6, 4) * 2 + 1)
    eg.engram_layer_set_multipliers(ctx, 0, m)
    assert np.array_equal(eg.engram_layer_params(ctx, 0, 6)[0], m)
    with pytest.raises(eg.EngramError) as e:
        eg.engram_layer_params(ctx, 1, 6)
    assert e.value.status == eg.EINVAL
    eg.engram_ctx_destroy(ctx)


# ---- sessions -----------------------------------------------------------------------

def oracle_windows(tmap, tokens, image=None):
    w = synth.WORKLOADS["tiny"]
    g = O.Geom(vocab=w.vocab, vc=w.vc, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d)
    return O.windows(g, tmap, tokens, image)


def test_append_matches_oracle_windows_with_images():
    ctx, tmap = tiny_ctx()
    s = eg.engram_session_create(ctx)
    toks = synth.zipf_tokens(300, 4096, seed=3)
    im = synth.image_flags(300, [(10, 5), (100, 40), (299, 1)])
    win = eg.engram_session_append(s, toks, im)
    assert np.array_equal(win, oracle_windows(tmap, toks, im))
    assert (win[10:15, 0] == eg.DEAD).all()
    eg.engram_session_destroy(s)
    eg.engram_ctx_destroy(ctx)


def test_span_append_equals_token_by_token():
    ctx, tmap = tiny_ctx()
    toks = synth.zipf_tokens(50, 4096, seed=4)
    a = eg.engram_session_create(ctx)
    b = eg.engram_session_create(ctx)
    wa = eg.engram_session_append(a, toks)
    wb = np.concatenate([eg.engram_session_append(b, toks[i:i + 1]) for i in range(50)])
    wc = eg.engram_session_append(eg.engram_session_create(ctx), toks[:17])
    assert np.array_equal(wa, wb)
    assert np.array_equal(wa[:17], wc)
    eg.engram_ctx_destroy(ctx)


def test_fork_isolates_history_and_reset_empties_it():
    ctx, tmap = tiny_ctx()
    p = eg.engram_session_create(ctx)
    eg.engram_session_append(p, [1, 2, 3])
    f = eg.engram_session_fork(p)
    wf = eg.engram_session_append(f, [7, 8])
    wp = eg.engram_session_append(p, [9])
    assert np.array_equal(wf, oracle_windows(tmap, [1, 2, 3, 7, 8])[3:])
    assert np.array_equal(wp, oracle_windows(tmap, [1, 2, 3, 9])[3:])
    eg.engram_session_reset(f)
    fresh = eg.engram_session_create(ctx)
    assert np.array_equal(eg.engram_session_append(f, [5, 6]),
                          eg.engram_session_append(fresh, [5, 6]))
    for s in (p, f, fresh):
        eg.engram_session_destroy(s)
    eg.engram_ctx_destroy(ctx)


def test_append_twice_shifts_the_windows():
    # a token appended twice (e.g. once per Engram layer) shifts later n-grams
    ctx, tmap = tiny_ctx()
    a, b = eg.engram_session_create(ctx), eg.engram_session_create(ctx)
    eg.engram_session_append(a, [11, 12])
    eg.engram_session_append(b, [11, 12])
    eg.engram_session_append(b, [12])
    assert not np.array_equal(eg.engram_session_append(a, [13]), eg.engram_session_append(b, [13]))
    eg.engram_ctx_destroy(ctx)


def test_bad_token_appends_nothing():
    ctx, tmap = tiny_ctx()
    s = eg.engram_session_create(ctx)
    eg.engram_session_append(s, [1, 2])
    for bad in ([3, 4096], [-1], [5, 6, 99999]):
        with pytest.raises(eg.EngramError) as e:
            eg.engram_session_append(s, bad)
        assert e.value.status == eg.EINVAL
    # an image position ignores its token value
    w = eg.engram_session_append(s, [123456], [1])
    assert w[0, 0] == eg.DEAD
    assert np.array_equal(eg.engram_session_append(s, [3]),
                          oracle_windows(tmap, [1, 2, 0, 3], [0, 0, 1, 0])[3:])
    eg.engram_ctx_destroy(ctx)


def test_batch_append_is_one_token_per_session():
    ctx, tmap = tiny_ctx()
    rng = np.random.default_rng(0)
    hist = [synth.zipf_tokens(3, 4096, seed=10 + i) for i in range(8)]
    ss = [eg.engram_session_create(ctx) for _ in range(8)]
    for s, h in zip(ss, hist):
        eg.engram_session_append(s, h)
    seqs = [list(h) for h in hist]
    imgs = [[0] * len(h) for h in hist]
    for step in range(5):
        tok = rng.integers(0, 4096, 8).astype(np.int32)
        img = (rng.random(8) < 0.2).astype(np.uint8)
        win = eg.engram_batch_append(ss, tok, img)
        for i in range(8):
            seqs[i].append(int(tok[i]))
            imgs[i].append(int(img[i]))
            ref = oracle_windows(tmap, seqs[i], np.array(imgs[i], np.uint8))[-1]
            assert np.array_equal(win[i], ref)
    for s in ss:
        eg.engram_session_destroy(s)
    eg.engram_ctx_destroy(ctx)


def test_device_calls_validate_before_launch():
    ctx, _ = tiny_ctx()
    for fn, args in [
        (eg.engram_gather_dequant, (0, 16, 4, 16)),
        (eg.engram_project, (0, 16, 4, 16)),
        (eg.engram_gate, (0, 16, 16, 4, 16)),
        (eg.engram_forward, (0, 16, 4, 16, 16)),
        (eg.engram_project_windows, (0, 16, 4, 16)),
        (eg.engram_forward_staged, (0, 16, 4, 16, 16)),
        (eg.engram_stage_rows, (0, 16, 4, 16)),
        (eg.engram_forward_staged_rows, (0, 16, 4, 16, 16)),
        (eg.engram_prepass, (0, 16, 4, 16, eg.KV_BF16, 16)),
        (eg.engram_gate_bf16kv, (0, 16, 16, 4, 16)),
    ]:
        with pytest.raises(eg.EngramError) as e:
            fn(ctx, *args)
        assert e.value.status == eg.ESTATE  # layer not bound
    with pytest.raises(eg.EngramError) as e:
        eg.engram_hash(ctx, 0, 16, -1, 16)
    assert e.value.status == eg.EINVAL
    with pytest.raises(eg.EngramError) as e:
        eg.engram_hash(ctx, 3, 16, 1, 16)
    assert e.value.status == eg.EINVAL
    with pytest.raises(eg.EngramError) as e:
        eg.engram_hash(ctx, 0, 8, 1, 16)  # misaligned windows
    assert e.value.status == eg.EINVAL
    eg.engram_hash(ctx, 0, None, 0, None)  # T = 0 is a no-op
    # gate sums [T][hc][d/256][3] fp32, gates [T][hc] and the counters (two per
    # 128-token block and TMEM quadrant), each 256-byte aligned
    assert eg.engram_workspace_bytes(ctx, 64) == 64 * 2 * 1 * 3 * 4 + 64 * 2 * 4 + 256
    assert eg.engram_workspace_bytes(ctx, 0) == 0
    eg.engram_ctx_destroy(ctx)


def test_last_error_is_set_and_cleared():
    ctx, _ = tiny_ctx()
    with pytest.raises(eg.EngramError):
        eg.engram_layer_params(ctx, 9, 6)
    assert "layer" in eg.engram_last_error()
    eg.engram_layer_params(ctx, 0, 6)
    assert eg.engram_last_error() == ""
    eg.engram_ctx_destroy(ctx)
