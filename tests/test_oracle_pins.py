"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a value printed
on the pages (row counts), a published known-answer vector (Philox), a library
routine implementing a standard (torch's OCP FP8 / BF16 conversions, numpy's
fp64 matmul, sympy's primality test), a closed form of the gate, or an
invariant that a dropped term, a wrong sign or a wrong index would break.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from golden_io import load_hash_worked

TINY = O.Geom(vocab=4096, vc=1000, heads=2, row_dim=32, hc=2, d=256)
FULL = O.Geom(vocab=129_280, vc=100_000)


def sigmoid(x):
    return 1.0 / (1.0 + math.exp(-x))


# --------------------------------------------------------------------------
# Philox4x32-10 against the published known-answer vectors
# --------------------------------------------------------------------------
def test_philox_known_answers(golden):
    rows = golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = O.philox4x32_10(v[0:4], v[4:6])
        assert [int(x) for x in out] == v[6:10]


# --------------------------------------------------------------------------
# Prime buckets: the printed per-layer row counts
# --------------------------------------------------------------------------
def test_row_counts_printed_on_the_pages(golden):
    kv = {r[0]: int(r[1]) for r in golden("engram_row_counts.txt")}
    g = O.Geom(vocab=129_280, vc=100_000, heads=kv["buckets_per_layer"] // 3)
    bases = [kv["bucket_base"]] * 2
    l1 = O.layer_params(g, [1, 14], bases, 0)
    l14 = O.layer_params(g, [1, 14], bases, 1)
    assert l1.rows == kv["rows_layer_1"]
    assert l14.rows == kv["rows_layer_14"]
    gib = (l1.rows + l14.rows) * 256 / 2**30
    assert round(gib) == kv["code_gib_two_layers_rounded"]
    # layer 14 continues after layer 1: no prime is shared
    assert set(l1.prime.tolist()).isdisjoint(l14.prime.tolist())
    assert int(l14.prime.min()) > int(l1.prime.max())


def test_primality_against_sympy():
    sympy = pytest.importorskip("sympy")
    for n in list(range(0, 3000)) + list(range(16_000_000, 16_001_000)):
        assert O.is_prime(n) == sympy.isprime(n), n
    ps = O.primes_above(1000, 6)
    assert ps.tolist() == [sympy.nextprime(1000, i) for i in range(1, 7)]


def test_tiny_layer_params_structure():
    p = O.layer_params(TINY, [1], [1000], 0)
    assert p.prime.tolist() == [1009, 1013, 1019, 1021, 1031, 1033]
    assert p.rows == 6126
    assert p.offset.tolist() == [0] + np.cumsum(p.prime[:-1]).tolist()


@pytest.mark.parametrize("g,base", [(FULL, 666_666), (TINY, 1000)])
def test_layer_params_invariants(g, base):
    seeds, bases = [3, 4], [base, base]
    for layer in range(2):
        p = O.layer_params(g, seeds, bases, layer)
        primes = [int(x) for x in p.prime]
        assert all(a < b for a, b in zip(primes, primes[1:]))
        assert primes[0] > base and all(O.is_prime(x) for x in primes)
        # offsets are prefix sums: bucket ranges are disjoint and cover [0, rows)
        assert int(p.offset[0]) == 0
        for b in range(1, g.nb):
            assert int(p.offset[b]) == int(p.offset[b - 1]) + primes[b - 1]
        assert int(p.offset[-1]) + primes[-1] == p.rows
        # multipliers: odd, no product with a compressed id can wrap 64 bits,
        # shared by every bucket of the layer
        bound = (2**64 - 1) // g.vc
        for j in range(g.max_n):
            m = int(p.mult[0, j])
            assert m % 2 == 1 and m < bound
            assert (g.vc - 1) * m < 2**64
            assert all(int(p.mult[b, j]) == m for b in range(g.nb))
    # different seeds give different multipliers
    a = O.layer_params(g, [3, 4], bases, 0).mult
    b = O.layer_params(g, [3, 4], bases, 1).mult
    assert not np.array_equal(a, b)


# --------------------------------------------------------------------------
# OCP MX element decodes against torch's FP8 dtypes; BF16 RNE against torch
# --------------------------------------------------------------------------
def test_e4m3_all_codes_against_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = O.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert O.e4m3_value(0x7E) == 448.0
    assert O.e4m3_value(0x01) == 2.0**-9
    assert math.isnan(O.e4m3_value(0x7F)) and math.isnan(O.e4m3_value(0xFF))


def test_e8m0_all_codes_against_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for e in range(256):
        v = O.e8m0_value(e)
        if math.isnan(ref[e]):
            assert math.isnan(v), e
        else:
            assert v == ref[e] == 2.0 ** (e - 127), e


def test_bf16_rne_against_torch():
    rng = np.random.default_rng(5)
    # float32 inputs: torch's fp32 -> bf16 conversion is a single RNE step
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),           # subnormals
        np.array([3.3895314e38, 3.39e38, 1e-45, -0.0, 0.0, np.inf, -np.inf], np.float32),
    ])
    # exact ties: bf16 value + half an ulp (low 16 bits = 0x8000), odd and even
    ties = (rng.integers(0x3F80, 0x4700, 4000, dtype=np.uint32) << 16) | 0x8000
    vals = np.concatenate([vals, ties.view(np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, r in zip(vals.tolist(), ref.tolist()):
        assert O.bf16_from_double(x) == r, (x, hex(r))
    # round trip of every finite bf16 pattern of one binade and the special ones
    for bits in list(range(0x3F80, 0x4000)) + [0x0001, 0x807F, 0x7F7F, 0xFF7F]:
        assert O.bf16_from_double(O.bf16_value(bits)) == bits


def test_dequant_exact_in_bf16_for_table_scales():
    # every finite E4M3 code times every scale the tables use is exact in BF16
    for c in range(256):
        x = O.e4m3_value(c)
        if math.isnan(x):
            continue
        for s in range(119, 128):
            v = x * O.e8m0_value(s)
            assert O.bf16_value(O.bf16_from_double(v)) == v


# --------------------------------------------------------------------------
# Table contents: finite codes, uniform code and scale distributions
# --------------------------------------------------------------------------
def test_table_contents_distribution():
    counts = np.zeros(256, np.int64)
    scounts = np.zeros(256, np.int64)
    for row in range(0, 40_000_000_000, 40_000_000_000 // 400):
        codes, scales = O.table_row(7, row, 256)
        np.add.at(counts, codes, 1)
        np.add.at(scounts, scales, 1)
    assert counts[0x7F] == 0 and counts[0xFF] == 0
    finite = np.delete(counts, [0x7F, 0xFF])
    exp = counts.sum() / 254
    assert finite.min() > 0.75 * exp and finite.max() < 1.25 * exp
    assert scounts[:119].sum() == 0 and scounts[128:].sum() == 0
    s = scounts[119:128]
    assert s.min() > 0.75 * s.mean() and s.max() < 1.25 * s.mean()
    # rows and seeds differ
    assert not np.array_equal(O.table_row(7, 5, 256)[0], O.table_row(7, 6, 256)[0])
    assert not np.array_equal(O.table_row(7, 5, 256)[0], O.table_row(8, 5, 256)[0])
    # 64-bit row numbers reach the counter's high word
    assert not np.array_equal(O.table_row(7, 5, 256)[0], O.table_row(7, 5 + 2**32, 256)[0])


# --------------------------------------------------------------------------
# Windows: history, pad before the start, DEAD for image positions
# --------------------------------------------------------------------------
def test_windows_hand_built():
    g = O.Geom(vocab=16, vc=8, pad_cid=0, heads=1, row_dim=32, hc=1, d=32)
    tmap = np.array([0, 1, 2, 3, 4, 5, 6, 7, 3, 3, 1, 1, 7, 6, 5, 4], np.uint32)
    w = O.windows(g, tmap, [5, 9, 5, 2, 12])
    assert w.tolist() == [[5, 0, 0, 0], [3, 5, 0, 0], [5, 3, 5, 0], [2, 5, 3, 5], [7, 2, 5, 3]]
    im = np.array([0, 1, 1, 0, 0, 0], np.uint8)
    w = O.windows(g, tmap, [1, 0, 0, 2, 3, 4], im)
    D = O.DEAD
    assert w.tolist() == [[1, 0, 0, 0], [D, 1, 0, 0], [D, D, 1, 0], [2, D, D, 1], [3, 2, D, D],
                          [4, 3, 2, D]]
    g2 = O.Geom(vocab=16, vc=8, pad_cid=6, heads=1, row_dim=32, hc=1, d=32)
    assert O.windows(g2, tmap, [1]).tolist() == [[1, 6, 6, 6]]
    with pytest.raises(ValueError):
        O.windows(g, tmap, [16])
    with pytest.raises(ValueError):
        O.windows(g, tmap, [-1])


# --------------------------------------------------------------------------
# Hash: brute force over a tiny compressed vocabulary
# --------------------------------------------------------------------------
G7 = O.Geom(vocab=7, vc=7, heads=8, row_dim=32, hc=1, d=32)


def _all_windows(vc):
    c = np.arange(vc, dtype=np.uint32)
    return np.stack(np.meshgrid(c, c, c, c, indexing="ij"), -1).reshape(-1, 4)


@pytest.fixture(scope="module")
def brute7():
    p = O.layer_params(G7, [9], [50], 0)
    wins = _all_windows(7)
    rows = np.stack([O.hash_rows(G7, p, w) for w in wins])
    return p, wins, rows


def test_hash_rows_inside_own_bucket(brute7):
    p, wins, rows = brute7
    for b in range(G7.nb):
        lo, hi = int(p.offset[b]), int(p.offset[b]) + int(p.prime[b])
        assert rows[:, b].min() >= lo and rows[:, b].max() < hi


def test_hash_order_n_reads_only_the_suffix_n_gram(brute7):
    p, wins, rows = brute7
    for n in range(2, 5):
        bs = slice((n - 2) * 8, (n - 1) * 8)
        key = [tuple(w[:n]) for w in wins]
        seen = {}
        for k, r in zip(key, rows[:, bs]):
            if k in seen:
                assert np.array_equal(seen[k], r)
            seen[k] = r
        # and does depend on every one of its n positions
        for j in range(n):
            w2 = wins.copy()
            w2[:, j] = (w2[:, j] + 1) % 7
            r2 = np.stack([O.hash_rows(G7, p, w) for w in w2[:200]])
            assert (r2[:, bs] != rows[:200, bs]).any(axis=1).mean() > 0.9


def test_hash_heads_never_all_collide(brute7):
    # bucket sizes are distinct primes: two different n-grams can share a row
    # in one head, but not in all eight heads of their order
    p, wins, rows = brute7
    for n in range(2, 5):
        bs = slice((n - 2) * 8, (n - 1) * 8)
        grams = {}
        for w, r in zip(wins, rows[:, bs]):
            grams.setdefault(tuple(w[:n]), tuple(r))
        assert len(set(grams.values())) == len(grams) == 7**n
        # single-head collisions do occur (the buckets are small): the heads differ
        per_head = [len({v[k] for v in grams.values()}) for k in range(8)]
        assert min(per_head) < len(grams) or n == 2


def test_hash_dead_masks_exactly_the_orders_that_touch_it():
    p = O.layer_params(FULL, [1], [666_666], 0)
    base = np.array([11, 22, 33, 44], np.uint32)
    full = O.hash_rows(FULL, p, base)
    assert (full != O.MASKED).all()
    for j in range(4):
        w = base.copy()
        w[j] = O.DEAD
        r = O.hash_rows(FULL, p, w)
        for n in range(2, 5):
            bs = slice((n - 2) * 8, (n - 1) * 8)
            if n > j:
                assert (r[bs] == O.MASKED).all()
            else:
                assert np.array_equal(r[bs], full[bs])


def test_merged_tokens_hash_alike():
    g = O.Geom(vocab=4096, vc=1000)
    tmap = np.arange(4096, dtype=np.uint32) % 1000
    p = O.layer_params(g, [1], [666_666], 0)
    a = O.windows(g, tmap, [5, 1005, 2005, 42])
    b = O.windows(g, tmap, [3005, 5, 1005, 42 + 1000])
    assert np.array_equal(a, b)
    assert np.array_equal(O.hash_rows(g, p, a[-1]), O.hash_rows(g, p, b[-1]))


def test_hash_general_multiplier_table():
    # distinct multipliers per (bucket, position): the kernels consume the same table
    p = O.layer_params(G7, [9], [50], 0)
    rng = np.random.default_rng(0)
    m2 = (rng.integers(0, 2**40, (G7.nb, 4), dtype=np.uint64) * 2 + 1).astype(np.uint64)
    q = O.LayerParams(m2, p.prime, p.offset, p.rows)
    w = np.array([1, 2, 3, 4], np.uint32)
    r1, r2 = O.hash_rows(G7, p, w), O.hash_rows(G7, q, w)
    assert not np.array_equal(r1, r2)
    for b in range(G7.nb):
        assert int(p.offset[b]) <= r2[b] < int(p.offset[b] + p.prime[b])


G_WORKED = O.Geom(vocab=4096, vc=1000, heads=2, row_dim=32, hc=1, d=32)


def test_hash_hand_worked_values():
    # x = XOR of the products c_{t-j} m[b][j] (wrapping 64-bit), row = offset +
    # x mod prime: every value worked by hand in the fixture, including products
    # above 2^32, products that wrap 2^64 and an n-gram holding DEAD
    primes, offsets, tables, cases = load_hash_worked()
    assert len(cases) == 5 and G_WORKED.nb == len(primes)
    for name, win, want in cases:
        p = O.LayerParams(tables[name], primes, offsets, int(offsets[-1] + primes[-1]))
        got = O.hash_rows(G_WORKED, p, np.array(win, np.uint32))
        assert got.tolist() == want, (name, win)


# --------------------------------------------------------------------------
# Gather: decoded rows, masked rows are zero, bucket-major concatenation
# --------------------------------------------------------------------------
def test_gather_layout_and_masking():
    g = TINY
    rows = np.array([5, O.MASKED, 6000, 17, 1009, 3], np.uint32)
    e = O.gather(g, 101, rows)
    torch_vals = torch.from_numpy(e.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, r in enumerate(rows):
        seg = torch_vals[b * 32:(b + 1) * 32]
        if r == O.MASKED:
            assert (e[b * 32:(b + 1) * 32] == 0).all()
            continue
        codes, scales = O.table_row(101, int(r), 32)
        fp8 = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
        ref = fp8 * 2.0 ** (scales[0].astype(np.int64) - 127)
        assert np.array_equal(seg, ref)


def test_gather_full_rows_use_one_scale_per_32_values():
    g = FULL
    rng = np.random.default_rng(8)
    rows = rng.integers(0, 384_006_168, g.nb).astype(np.uint32)
    rows[[3, 17]] = O.MASKED
    e = O.gather(g, 77, rows)
    vals = torch.from_numpy(e.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, r in enumerate(rows):
        seg = vals[b * 256:(b + 1) * 256]
        if r == O.MASKED:
            assert (e[b * 256:(b + 1) * 256] == 0).all()
            continue
        codes, scales = O.table_row(77, int(r), 256)
        fp8 = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
        sc = torch.from_numpy(scales).view(torch.float8_e8m0fnu).double().numpy()
        assert np.array_equal(seg, fp8 * np.repeat(sc, 32))


@pytest.mark.parametrize("lo,hi", [(119, 127), (105, 127), (104, 127), (1, 254)])
def test_gather_from_a_table_in_memory_against_torch(lo, hi):
    # an explicit table with any E8M0 span: each value is torch's OCP E4M3
    # decode times 2^(e - 127) rounded once to BF16 (exact for spans inside
    # 2^-27..2^0; the widest span also overflows to inf and rounds subnormals)
    g = FULL
    codes, scales = synth.mxfp8_table(50, 256, 3, lo, hi)
    rows = np.array([(7 * b) % 50 for b in range(g.nb)], np.uint32)
    rows[[2, 11]] = O.MASKED
    e = O.gather_table(g, codes, scales, rows)
    vals = torch.from_numpy(e.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, r in enumerate(rows):
        seg = vals[b * 256:(b + 1) * 256]
        if r == O.MASKED:
            assert (e[b * 256:(b + 1) * 256] == 0).all()
            continue
        fp8 = torch.from_numpy(codes[r]).view(torch.float8_e4m3fn).double().numpy()
        ref = fp8 * np.ldexp(1.0, np.repeat(scales[r].astype(np.int64) - 127, 32))
        # one round-to-nearest-even to BF16 (the fp32 step is exact for these
        # 4-bit significands); the identity wherever the product fits BF16
        ref16 = torch.from_numpy(ref).float().to(torch.bfloat16).double().numpy()
        if hi <= 127:
            assert np.array_equal(ref16, ref)
        assert np.array_equal(seg, ref16), (lo, hi, b)
    with pytest.raises(ValueError):
        O.gather_table(g, codes, scales, np.full(g.nb, 50, np.uint32))


def test_gather_from_memory_matches_the_generated_contents():
    g = TINY
    rows = np.array([5, O.MASKED, 6000, 17, 1009, 3], np.uint32)
    table = [O.table_row(101, r, 32) for r in range(6126)]
    codes = np.stack([c for c, _ in table])
    scales = np.stack([s for _, s in table])
    assert np.array_equal(O.gather_table(g, codes, scales, rows), O.gather(g, 101, rows))


# --------------------------------------------------------------------------
# Projection against numpy's fp64 matmul
# --------------------------------------------------------------------------
def test_project_against_numpy():
    g = TINY
    rng = np.random.default_rng(1)
    from synth import to_bf16_bits
    w = to_bf16_bits(rng.standard_normal((g.N, g.K)).astype(np.float32))
    e = to_bf16_bits(rng.standard_normal(g.K).astype(np.float32) * 30)
    as64 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    ref = as64(w) @ as64(e)
    kv = O.project(g, w, e)
    assert np.allclose(kv, ref, rtol=1e-12, atol=1e-9)


# --------------------------------------------------------------------------
# Gate: closed forms and invariants
# --------------------------------------------------------------------------
GG = O.Geom(vocab=8, vc=8, heads=1, row_dim=32, hc=2, d=256)


def _bf(x):
    from synth import to_bf16_bits
    return to_bf16_bits(np.asarray(x, np.float32))


def _as64(bits):
    return torch.from_numpy(np.asarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_gate_zero_key_gives_sigmoid_of_floor():
    rng = np.random.default_rng(2)
    h = _bf(rng.standard_normal((2, 256)))
    kv = np.zeros(3 * 256)
    kv[512:] = rng.standard_normal(256)
    ones = np.ones((2, 256), np.float32)
    ho, h16, gates = O.gate(GG, kv, 1, h, ones, ones)
    assert gates == pytest.approx([sigmoid(1e-3)] * 2, abs=1e-15)
    assert gates[0] == pytest.approx(0.5002499999791666, abs=1e-15)
    np.testing.assert_allclose(ho, _as64(h) + sigmoid(1e-3) * kv[512:], rtol=0, atol=1e-14)


def test_gate_zero_hidden_gives_sigmoid_of_floor():
    rng = np.random.default_rng(3)
    kv = rng.standard_normal(3 * 256)
    h = np.zeros((2, 256), np.uint16)
    ones = np.ones((2, 256), np.float32)
    _, _, gates = O.gate(GG, kv, 1, h, ones, ones)
    assert gates == pytest.approx([sigmoid(1e-3)] * 2, abs=1e-15)


def test_gate_aligned_key_closed_form():
    # h = k and unit weights: dot = sqrt(d) m/(m+eps) with m = mean(h^2),
    # so gate = sigmoid(d^(1/4) sqrt(m/(m+eps)))
    rng = np.random.default_rng(4)
    h = _bf(rng.standard_normal((2, 256)))
    kv = np.zeros(3 * 256)
    kv[:512] = _as64(h).reshape(-1)
    ones = np.ones((2, 256), np.float32)
    _, _, gates = O.gate(GG, kv, 1, h, ones, ones)
    for b in range(2):
        m = float(np.mean(_as64(h[b]) ** 2))
        dot = math.sqrt(256) * m / (m + 1e-6)
        assert gates[b] == pytest.approx(sigmoid(math.sqrt(dot)), rel=1e-12)
    assert gates[0] == pytest.approx(sigmoid(4.0), rel=1e-5)  # d^(1/4) = 4


def test_gate_sign_scale_and_weight_invariants():
    rng = np.random.default_rng(6)
    h = _bf(rng.standard_normal((2, 256)))
    kv = rng.standard_normal(3 * 256)
    wq = (1 + 0.1 * rng.standard_normal((2, 256))).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal((2, 256))).astype(np.float32)
    _, _, g0 = O.gate(GG, kv, 1, h, wq, wk)
    # flipping the key's sign flips the dot: gate -> 1 - gate
    kvn = kv.copy()
    kvn[:512] *= -1
    _, _, g1 = O.gate(GG, kvn, 1, h, wq, wk)
    np.testing.assert_allclose(g1, 1 - g0, atol=1e-14)
    # scaling the key does not change the gate (RMS normalisation), up to eps
    kv2 = kv.copy()
    kv2[:512] *= 8
    _, _, g2 = O.gate(GG, kv2, 1, h, wq, wk)
    np.testing.assert_allclose(g2, g0, atol=1e-6)
    # doubling both weights multiplies the dot by 4: logit doubles
    _, _, g3 = O.gate(GG, kv, 1, h, 2 * wq, 2 * wk)
    logit = lambda g: math.log(g / (1 - g))
    for b in range(2):
        assert logit(g3[b]) == pytest.approx(2 * logit(g0[b]), rel=1e-9)
    # each branch uses its own key and weights: swapping branches swaps gates
    kvs = kv.copy()
    kvs[:256], kvs[256:512] = kv[256:512], kv[:256]
    _, _, g4 = O.gate(GG, kvs, 1, h[::-1].copy(), wq[::-1].copy(), wk[::-1].copy())
    np.testing.assert_allclose(g4, g0[::-1], atol=1e-14)
    # large dot saturates
    kv5 = kv.copy()
    kv5[:512] = _as64(h).reshape(-1)
    wq5 = np.full((2, 256), 40.0, np.float32)
    _, _, g5 = O.gate(GG, kv5, 1, h, wq5, wq5)
    assert (g5 > 1 - 1e-12).all()
    _, _, g6 = O.gate(GG, -kv5, 1, h, wq5, wq5)
    assert (g6 < 1e-12).all()


def test_gate_value_is_last_d_rows_and_image_rows_pass_through():
    rng = np.random.default_rng(7)
    h = _bf(rng.standard_normal((2, 256)))
    kv = rng.standard_normal(3 * 256)
    ones = np.ones((2, 256), np.float32)
    ho, h16, g = O.gate(GG, kv, 1, h, ones, ones)
    for b in range(2):
        np.testing.assert_allclose(ho[b] - _as64(h[b]), g[b] * kv[512:], atol=1e-12)
        assert np.array_equal(h16[b], _bf(ho[b]))
    ho, h16, g = O.gate(GG, kv, O.DEAD, h, ones, ones)
    assert np.array_equal(h16, h) and (g == 0).all()


# --------------------------------------------------------------------------
# The step composed, on the tiny workload
# --------------------------------------------------------------------------
def test_forward_composes_the_steps():
    import synth
    w = synth.WORKLOADS["tiny"]
    g = O.Geom(vocab=w.vocab, vc=w.vc, heads=w.heads, row_dim=w.row_dim, hc=w.hc, d=w.d)
    p = O.layer_params(g, w.hash_seeds, w.bucket_bases, 0)
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    toks = synth.session_tokens(w, 0, 16)
    im = synth.image_flags(16, [(6, 2)])
    wins = O.windows(g, tmap, toks, im)
    hid = synth.hidden_bf16(w, 16)
    W = synth.wkv_bf16(w)
    wq, wk = synth.wq_wk(w)
    out = O.forward(g, w.table_seeds[0], p, W, wq, wk, wins, hid, np.arange(16), nthreads=3,
                    want_e=True, want_kv=True)
    for t in range(16):
        rows = O.hash_rows(g, p, wins[t])
        assert np.array_equal(out["rows"][t], rows)
        e = O.gather(g, w.table_seeds[0], rows)
        assert np.array_equal(out["e"][t], e)
        kv = O.project(g, W, e)
        assert np.array_equal(out["kv"][t], kv)
        ho, h16, gates = O.gate(g, kv, int(wins[t][0]), hid[t], wq, wk)
        assert np.array_equal(out["h_bf16"][t], h16)
        assert np.array_equal(out["gates"][t], gates)
    # image rows unchanged; the text row right after an image span is all-masked
    assert np.array_equal(out["h_bf16"][6], hid[6]) and np.array_equal(out["h_bf16"][7], hid[7])
    assert (out["rows"][8] == O.MASKED).all()
    assert np.array_equal(out["h_bf16"][8], hid[8])
    # DEAD at t-2 masks only the 3- and 4-grams
    assert (out["rows"][9][:2] != O.MASKED).all() and (out["rows"][9][2:] == O.MASKED).all()
