"""Seeded synthetic inputs for the Engram forward step.

This module only draws inputs: token streams, the compression map, image
spans, hidden states, wkv and the norm weights.  It holds none of the method's
arithmetic (no hashing, decoding, projection or gating), so both the CUDA path
and the CPU oracle may take their inputs from it.

The pages' real workloads (DeepSeek tokenizer, safetensors weights, prompts)
are not available; these stand-ins keep their shapes, sizes and structure:
Zipf(1.1) token ranks over the 129,280-entry vocabulary, a surjective
many-to-one compression map, image spans of DEAD positions, BF16 hidden
states and wkv, and norm weights near 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# Standard deviation of a dequantised table value for tables whose codes are
# uniform over the 254 finite E4M3 codes (RMS 100.06) and whose scales are
# uniform over 2^-8..2^0 (RMS 0.385): 100.06 * 0.385 = 38.5.
TABLE_VALUE_RMS = 38.5


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=np.array([seed, stream], np.uint64)))


def zipf_tokens(n: int, vocab: int, seed: int, s: float = 1.1, stream: int = 10) -> np.ndarray:
    """n token ids with rank ~ Zipf(s) over [1, vocab] (inverse CDF); token = rank - 1."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** -s)
    cdf /= cdf[-1]
    u = _rng(seed, stream).random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def token_map(vocab: int, vc: int, seed: int, stream: int = 11) -> np.ndarray:
    """Surjective many-to-one map: identity below vc, uniform in [0, vc) above."""
    m = np.arange(vocab, dtype=np.uint32)
    if vocab > vc:
        m[vc:] = _rng(seed, stream).integers(0, vc, vocab - vc, dtype=np.uint32)
    return m


def image_flags(n: int, spans) -> np.ndarray:
    """u8 flags, 1 inside each [start, start + length) span."""
    f = np.zeros(n, np.uint8)
    for start, length in spans:
        f[start:start + length] = 1
    return f


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, sigma: float, seed: int, stream: int, chunk: int = 1 << 24) -> np.ndarray:
    """BF16 bit patterns of N(0, sigma^2) draws (drawn in float32, then rounded)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    g = _rng(seed, stream)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = to_bf16_bits(g.standard_normal(m, dtype=np.float32) * np.float32(sigma))
    return out.reshape(shape)


def norm_weights(hc: int, d: int, seed: int, stream: int) -> np.ndarray:
    """Pre-multiplied norm weights 1 + 0.1 N(0, 1), fp32 [hc][d]."""
    g = _rng(seed, stream)
    return (1.0 + 0.1 * g.standard_normal((hc, d))).astype(np.float32)


def mxfp8_table(rows: int, row_dim: int, seed: int, scale_lo: int, scale_hi: int,
                stream: int = 50):
    """A host MXFP8 table: codes uint8 [rows][row_dim] uniform over the 254
    finite E4M3 codes (0x7F and 0xFF excluded) and E8M0 exponents uint8
    [rows][row_dim / 32] uniform over [scale_lo, scale_hi]."""
    g = _rng(seed, stream)
    idx = g.integers(0, 254, (rows, row_dim), dtype=np.uint16)
    codes = (idx + (idx >= 127)).astype(np.uint8)
    scales = g.integers(scale_lo, scale_hi + 1, (rows, row_dim // 32), dtype=np.uint16)
    return codes, scales.astype(np.uint8)


@dataclass
class Workload:
    """One benchmark / parity configuration (sizes as the pages' workloads)."""

    name: str
    vocab: int
    vc: int
    heads: int
    row_dim: int
    hc: int
    d: int
    bucket_bases: list            # per layer, in layer order
    hash_seeds: list              # per layer
    table_seeds: list             # per layer
    wkv_sigma: float
    sessions: int = 1             # independent histories
    tokens_per_session: int = 64  # tokens appended per session (prefill)
    history: int = 0              # tokens appended before the measured step (decode)
    steps: int = 1                # decode steps (one token per session per step)
    image_spans: list = field(default_factory=list)  # (start, length) per session
    host_table: bool = False
    seed: int = 0
    min_n: int = 2
    max_n: int = 4
    pad_cid: int = 0
    eps: float = 1e-6

    @property
    def nb(self) -> int:
        return (self.max_n - self.min_n + 1) * self.heads

    @property
    def K(self) -> int:
        return self.nb * self.row_dim

    @property
    def N(self) -> int:
        return (self.hc + 1) * self.d


def _full(**kw) -> dict:
    base = dict(vocab=129_280, vc=100_000, heads=8, row_dim=256, hc=4, d=5120,
                wkv_sigma=1.0 / (np.sqrt(6144.0) * TABLE_VALUE_RMS))
    base.update(kw)
    return base


WORKLOADS = {
    # 64 tokens, V 4096 -> 1000 ids, 3 orders x 2 heads of 32-wide rows, hc 2 x 256.
    "tiny": Workload(name="tiny", vocab=4096, vc=1000, heads=2, row_dim=32, hc=2, d=256,
                     bucket_bases=[1000], hash_seeds=[1], table_seeds=[101],
                     wkv_sigma=1.0 / np.sqrt(192.0), tokens_per_session=64),
    # One 2,048-token prefill, full geometry, 16.0M-row table.
    "prefill_2048": Workload(name="prefill_2048", **_full(
        bucket_bases=[666_666], hash_seeds=[1], table_seeds=[101], tokens_per_session=2048)),
    # 256 sessions x (3-token history, then 1 token per step for 100 steps); 384M rows.
    "decode_256": Workload(name="decode_256", **_full(
        bucket_bases=[16_000_000], hash_seeds=[1], table_seeds=[101], sessions=256,
        tokens_per_session=1, history=3, steps=100)),
    # 50,032 tokens, 3 image spans of 1,024, two layers with 64M-row tables each.
    "prefill_50k_2layer": Workload(name="prefill_50k_2layer", **_full(
        bucket_bases=[2_666_666, 2_666_666], hash_seeds=[1, 14], table_seeds=[101, 114],
        tokens_per_session=50_032, image_spans=[(8000, 1024), (24000, 1024), (40000, 1024)])),
    # 8 sessions x 1,024 tokens, 384M-row table in pinned host memory.
    "host_table_8x1024": Workload(name="host_table_8x1024", **_full(
        bucket_bases=[16_000_000], hash_seeds=[1], table_seeds=[101], sessions=8,
        tokens_per_session=1024, host_table=True)),
}


def session_tokens(w: Workload, session: int, count: int, offset: int = 0) -> np.ndarray:
    """Token ids [offset, offset + count) of one session's stream (deterministic)."""
    toks = zipf_tokens(offset + count, w.vocab, seed=w.seed * 1_000_003 + session)
    return toks[offset:offset + count]


def hidden_bf16(w: Workload, T: int, stream: int = 20) -> np.ndarray:
    return normal_bf16((T, w.hc, w.d), 1.0, w.seed, stream)


def wkv_bf16(w: Workload, layer: int = 0) -> np.ndarray:
    return normal_bf16((w.N, w.K), w.wkv_sigma, w.seed, 30 + layer)


def wq_wk(w: Workload, layer: int = 0):
    return norm_weights(w.hc, w.d, w.seed, 40 + 2 * layer), norm_weights(w.hc, w.d, w.seed,
                                                                         41 + 2 * layer)
