"""Shared helpers of the GPU parity tests: setup of a workload on the device and
the comparison rules.

Tolerances (floating point; integer and byte results are compared exactly):
  hidden  GPU BF16 vs the oracle's fp64 result rounded once to BF16:
          max |diff| <= max(2e-2, 1 BF16 ulp of the reference), mean <= 2e-3
          (one ulp covers a rounding flip where the fp32 and fp64 sums sit on
          either side of a BF16 rounding boundary)
  gates   |diff| <= 1e-3
  kv      |diff| <= K 2^-24 sum_i |W_oi e_i| + 1e-30 (fp32 accumulation bound)
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import engram_gram_conditional_gb300 as eg
import oracle as O
import synth
from engram_gram_conditional_gb300.layer import EngramLayerSet


def bf16_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, np.uint16))
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.frexp(np.where(ax > 0, ax, 1.0))[1]
    return np.where(ax > 0, np.ldexp(1.0, e - 8), 2.0**-133)


def check_hidden(got_bits, ref_bits, what=""):
    g, r = bf16_f64(got_bits), bf16_f64(ref_bits)
    err = np.abs(g - r)
    tol = np.maximum(2e-2, bf16_ulp(r))
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} values beyond tolerance, max err "
                           f"{err.max():.4g} at {np.unravel_index(np.argmax(err), err.shape)}")
    assert err.mean() <= 2e-3, f"{what}: mean err {err.mean():.4g}"
    return float(err.max()), float(err.mean())


def check_kv(got, ref64, W_bits, e_bits, K, what=""):
    Wf = bf16_f64(W_bits)
    ef = bf16_f64(e_bits)
    bound = K * 2.0**-24 * (np.abs(ef) @ np.abs(Wf).T) + 1e-30
    err = np.abs(got.astype(np.float64) - ref64)
    assert (err <= bound).all(), f"{what}: kv beyond the fp32 bound, worst {(err / bound).max():.3g}x"


def geom(w) -> O.Geom:
    return O.Geom(vocab=w.vocab, vc=w.vc, min_n=w.min_n, max_n=w.max_n, heads=w.heads,
                  row_dim=w.row_dim, hc=w.hc, d=w.d, pad_cid=w.pad_cid, eps=w.eps)


@dataclass
class Setup:
    w: object
    tmap: np.ndarray
    model: EngramLayerSet
    W: list
    wq: list
    wk: list
    oparams: list
    tables: list = None  # per layer: None (generated contents) or host (codes, scales)

    def table(self, layer=0):
        return None if self.tables is None else self.tables[layer]

    def oracle_forward(self, layer, win, hidden, idx, **kw):
        """The oracle's step on positions idx, over this layer's table."""
        return O.forward(geom(self.w), self.w.table_seeds[layer], self.oparams[layer],
                         self.W[layer], self.wq[layer], self.wk[layer], win, hidden,
                         np.asarray(idx), table=self.table(layer), **kw)

    def close(self):
        self.model.close()
        torch.cuda.empty_cache()


def setup_workload(name: str, layers=None, host_table=False, flags=0, tables=None, wkv=None,
                   **overrides) -> Setup:
    """Bind the workload's layers.  tables / wkv: optional {layer: host MXFP8
    table (codes, scales)} / {layer: BF16 wkv bits} in place of the generated
    table contents / the synthetic wkv."""
    import dataclasses

    w = dataclasses.replace(synth.WORKLOADS[name], **overrides) if overrides else \
        synth.WORKLOADS[name]
    tables = tables or {}
    wkv = wkv or {}
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    model = EngramLayerSet.from_workload(w, tmap, device="cuda")
    layers = range(len(w.hash_seeds)) if layers is None else layers
    W, WQ, WK = [], [], []
    for l in range(len(w.hash_seeds)):
        if l in layers:
            Wl = wkv[l] if l in wkv else synth.wkv_bf16(w, l)
            q, k = synth.wq_wk(w, l)
            model.bind(l, w.table_seeds[l], Wl, q, k, host_table=host_table, flags=flags,
                       table=tables.get(l))
        else:
            Wl = q = k = None
        W.append(Wl)
        WQ.append(q)
        WK.append(k)
    g = geom(w)
    op = [O.layer_params(g, w.hash_seeds, w.bucket_bases, l) for l in range(len(w.hash_seeds))]
    torch.cuda.synchronize()
    tl = [tables.get(l) for l in range(len(w.hash_seeds))] if tables else None
    return Setup(w, tmap, model, W, WQ, WK, op, tl)


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32,
            np.dtype(np.uint8): np.uint8}.get(a.dtype, a.dtype)
    return torch.from_numpy(a.view(view)).cuda()


def from_dev(t: torch.Tensor, dtype) -> np.ndarray:
    return t.cpu().numpy().view(dtype)


def prefill_windows(s: Setup, sessions: int, per_session: int, spans=()):
    """Windows of `sessions` independent prefills, concatenated (via the library's append)."""
    out, toks, ims = [], [], []
    for i in range(sessions):
        t = synth.session_tokens(s.w, i, per_session)
        im = synth.image_flags(per_session, spans)
        sess = eg.engram_session_create(s.model.ctx)
        out.append(eg.engram_session_append(sess, t, im))
        eg.engram_session_destroy(sess)
        toks.append(t)
        ims.append(im)
    return np.concatenate(out), toks, ims
