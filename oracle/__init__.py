"""CPU oracle of the Engram per-layer forward step (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  The product
package never imports this module and this module never imports the product.

Every function cites the passage of the pages it follows in ``oracle.c``; the
readings taken where the pages are silent are listed in ``oracle.h``.  Parity
unpinned against the real model: the hash multipliers and the table contents
(both build conventions, since the pages print no value of either).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

DEAD = 0xFFFFFFFF
MASKED = 0xFFFFFFFF


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, no GPU)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", _SRC, "-o", tmp,
             "-lpthread", "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Geom(C.Structure):
    _fields_ = [
        ("vocab", C.c_uint32), ("vc", C.c_uint32), ("min_n", C.c_uint32),
        ("max_n", C.c_uint32), ("heads", C.c_uint32), ("row_dim", C.c_uint32),
        ("hc", C.c_uint32), ("d", C.c_uint32), ("pad_cid", C.c_uint32),
        ("reserved", C.c_uint32), ("eps", C.c_double),
    ]


@dataclass(frozen=True)
class Geom:
    """Geometry of one Engram layer (field meanings as in oracle.h)."""

    vocab: int
    vc: int
    min_n: int = 2
    max_n: int = 4
    heads: int = 8
    row_dim: int = 256
    hc: int = 4
    d: int = 5120
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

    def c(self) -> _Geom:
        return _Geom(self.vocab, self.vc, self.min_n, self.max_n, self.heads, self.row_dim,
                     self.hc, self.d, self.pad_cid, 0, self.eps)


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        P = C.POINTER
        u8p, u16p, u32p, u64p = (P(C.c_uint8), P(C.c_uint16), P(C.c_uint32), P(C.c_uint64))
        i32p, i64p, f32p, f64p = P(C.c_int32), P(C.c_int64), P(C.c_float), P(C.c_double)
        gp = P(_Geom)
        sig = {
            "orc_philox4x32_10": (None, [u32p, u32p, u32p]),
            "orc_table_code": (C.c_uint8, [C.c_uint64, C.c_uint64, C.c_uint32]),
            "orc_table_scale": (C.c_uint8, [C.c_uint64, C.c_uint64, C.c_uint32]),
            "orc_table_row": (None, [C.c_uint64, C.c_uint64, C.c_uint32, u8p, u8p]),
            "orc_e4m3_value": (C.c_double, [C.c_uint8]),
            "orc_e8m0_value": (C.c_double, [C.c_uint8]),
            "orc_bf16_from_double": (C.c_uint16, [C.c_double]),
            "orc_bf16_value": (C.c_double, [C.c_uint16]),
            "orc_is_prime": (C.c_int, [C.c_uint64]),
            "orc_primes_above": (None, [C.c_uint64, C.c_int, u64p]),
            "orc_layer_params": (C.c_int, [gp, C.c_int, u64p, u64p, C.c_int, u64p, u64p, u64p,
                                           u64p]),
            "orc_windows": (C.c_int, [gp, u32p, i32p, u8p, C.c_int64, u32p]),
            "orc_hash": (None, [gp, u64p, u64p, u64p, u32p, u32p]),
            "orc_gather": (None, [gp, C.c_uint64, u32p, u16p]),
            "orc_gather_table": (C.c_int, [gp, u8p, u8p, C.c_uint64, u32p, u16p]),
            "orc_project": (None, [gp, u16p, u16p, f64p]),
            "orc_gate": (None, [gp, f64p, C.c_uint32, u16p, f32p, f32p, f64p, u16p, f64p]),
            "orc_forward": (C.c_int, [gp, C.c_uint64, u64p, u64p, u64p, u16p, f32p, f32p, u32p,
                                      u16p, i64p, C.c_int64, C.c_int, u32p, u16p, f64p, f64p,
                                      f64p, u16p]),
            "orc_forward_table": (C.c_int, [gp, u8p, u8p, C.c_uint64, u64p, u64p, u64p, u16p,
                                            f32p, f32p, u32p, u16p, i64p, C.c_int64, C.c_int,
                                            u32p, u16p, f64p, f64p, f64p, u16p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _p(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.POINTER(ctype))


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


# -- element functions --------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c, C.c_uint32), _p(k, C.c_uint32), _p(out, C.c_uint32))
    return out


def table_code(seed: int, row: int, col: int) -> int:
    return int(lib().orc_table_code(seed, row, col))


def table_scale(seed: int, row: int, group: int) -> int:
    return int(lib().orc_table_scale(seed, row, group))


def table_row(seed: int, row: int, row_dim: int):
    codes = np.zeros(row_dim, np.uint8)
    scales = np.zeros(max(1, row_dim // 32), np.uint8)
    lib().orc_table_row(seed, row, row_dim, _p(codes, C.c_uint8), _p(scales, C.c_uint8))
    return codes, scales[: row_dim // 32]


def e4m3_value(code: int) -> float:
    return float(lib().orc_e4m3_value(code))


def e8m0_value(e: int) -> float:
    return float(lib().orc_e8m0_value(e))


def bf16_from_double(x: float) -> int:
    return int(lib().orc_bf16_from_double(float(x)))


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16_value(bits))


def is_prime(n: int) -> bool:
    return bool(lib().orc_is_prime(n))


def primes_above(base: int, count: int) -> np.ndarray:
    out = np.zeros(count, np.uint64)
    lib().orc_primes_above(base, count, _p(out, C.c_uint64))
    return out


# -- the method's steps -------------------------------------------------------

@dataclass
class LayerParams:
    mult: np.ndarray    # uint64 [nb][4]
    prime: np.ndarray   # uint64 [nb]
    offset: np.ndarray  # uint64 [nb]
    rows: int


def layer_params(g: Geom, seeds, bucket_bases, layer: int) -> LayerParams:
    s = _c(seeds, np.uint64)
    bb = _c(bucket_bases, np.uint64)
    mult = np.zeros((g.nb, 4), np.uint64)
    prime = np.zeros(g.nb, np.uint64)
    offset = np.zeros(g.nb, np.uint64)
    rows = np.zeros(1, np.uint64)
    gc = g.c()
    rc = lib().orc_layer_params(C.byref(gc), len(s), _p(s, C.c_uint64), _p(bb, C.c_uint64), layer,
                                _p(mult, C.c_uint64), _p(prime, C.c_uint64),
                                _p(offset, C.c_uint64), _p(rows, C.c_uint64))
    if rc != 0:
        raise ValueError(f"orc_layer_params failed ({rc})")
    return LayerParams(mult, prime, offset, int(rows[0]))


def windows(g: Geom, token_map, tokens, is_image=None) -> np.ndarray:
    tm = _c(token_map, np.uint32)
    tk = _c(tokens, np.int32)
    im = _c(np.zeros(len(tk), np.uint8) if is_image is None else is_image, np.uint8)
    out = np.zeros((len(tk), 4), np.uint32)
    gc = g.c()
    rc = lib().orc_windows(C.byref(gc), _p(tm, C.c_uint32), _p(tk, C.c_int32), _p(im, C.c_uint8),
                           len(tk), _p(out, C.c_uint32))
    if rc != 0:
        raise ValueError("token outside the vocabulary")
    return out


def hash_rows(g: Geom, p: LayerParams, window) -> np.ndarray:
    w = _c(window, np.uint32)
    rows = np.zeros(g.nb, np.uint32)
    gc = g.c()
    lib().orc_hash(C.byref(gc), _p(p.mult, C.c_uint64), _p(p.prime, C.c_uint64),
                   _p(p.offset, C.c_uint64), _p(w, C.c_uint32), _p(rows, C.c_uint32))
    return rows


def gather(g: Geom, seed: int, rows) -> np.ndarray:
    r = _c(rows, np.uint32)
    e = np.zeros(g.K, np.uint16)
    gc = g.c()
    lib().orc_gather(C.byref(gc), seed, _p(r, C.c_uint32), _p(e, C.c_uint16))
    return e


def gather_table(g: Geom, codes, scales, rows) -> np.ndarray:
    """Dequantised vector of one token's rows read from a table held in memory:
    codes uint8 [R][row_dim], scales uint8 [R][row_dim / 32]."""
    c = _c(codes, np.uint8)
    sc = _c(scales, np.uint8)
    nrows = c.size // g.row_dim
    assert c.size == nrows * g.row_dim and sc.size >= nrows * (g.row_dim // 32)
    r = _c(rows, np.uint32)
    e = np.zeros(g.K, np.uint16)
    gc = g.c()
    if lib().orc_gather_table(C.byref(gc), _p(c, C.c_uint8), _p(sc, C.c_uint8), nrows,
                              _p(r, C.c_uint32), _p(e, C.c_uint16)) != 0:
        raise ValueError("row index outside the table")
    return e


def project(g: Geom, w_bf16: np.ndarray, e_bf16) -> np.ndarray:
    w = _c(w_bf16, np.uint16)
    e = _c(e_bf16, np.uint16)
    assert w.size == g.N * g.K and e.size == g.K
    kv = np.zeros(g.N, np.float64)
    gc = g.c()
    lib().orc_project(C.byref(gc), _p(w, C.c_uint16), _p(e, C.c_uint16), _p(kv, C.c_double))
    return kv


def gate(g: Geom, kv, c_t: int, h_bf16, wq, wk):
    kv = _c(kv, np.float64)
    h = _c(h_bf16, np.uint16)
    q = _c(wq, np.float32)
    k = _c(wk, np.float32)
    h_out = np.zeros(g.hc * g.d, np.float64)
    h_out16 = np.zeros(g.hc * g.d, np.uint16)
    gates = np.zeros(g.hc, np.float64)
    gc = g.c()
    lib().orc_gate(C.byref(gc), _p(kv, C.c_double), c_t, _p(h, C.c_uint16), _p(q, C.c_float),
                   _p(k, C.c_float), _p(h_out, C.c_double), _p(h_out16, C.c_uint16),
                   _p(gates, C.c_double))
    return h_out.reshape(g.hc, g.d), h_out16.reshape(g.hc, g.d), gates


def forward(g: Geom, seed: int, p: LayerParams, w_bf16, wq, wk, windows_, hidden_bf16, idx,
            nthreads: int = 1, want_e: bool = False, want_kv: bool = False,
            want_h64: bool = True, table=None) -> dict:
    """The whole step on the positions ``idx`` (threads over positions).

    ``table``: None (rows from the generated contents of ``seed``) or a pair
    (codes uint8 [R][row_dim], scales uint8 [R][row_dim / 32]) held in memory."""
    w = _c(w_bf16, np.uint16)
    q = _c(wq, np.float32)
    k = _c(wk, np.float32)
    win = _c(windows_, np.uint32)
    hid = _c(hidden_bf16, np.uint16)
    ix = _c(idx, np.int64)
    n = len(ix)
    T = win.shape[0]
    assert win.shape == (T, 4) and hid.size == T * g.hc * g.d
    assert w.size == g.N * g.K and q.size == g.hc * g.d and k.size == g.hc * g.d
    assert n == 0 or (ix.min() >= 0 and ix.max() < T)
    out = {
        "rows": np.zeros((n, g.nb), np.uint32),
        "e": np.zeros((n, g.K), np.uint16) if want_e else None,
        "kv": np.zeros((n, g.N), np.float64) if want_kv else None,
        "gates": np.zeros((n, g.hc), np.float64),
        "h": np.zeros((n, g.hc, g.d), np.float64) if want_h64 else None,
        "h_bf16": np.zeros((n, g.hc, g.d), np.uint16),
    }
    gc = g.c()
    tail = (_p(p.mult, C.c_uint64), _p(p.prime, C.c_uint64), _p(p.offset, C.c_uint64),
            _p(w, C.c_uint16), _p(q, C.c_float), _p(k, C.c_float), _p(win, C.c_uint32),
            _p(hid, C.c_uint16), _p(ix, C.c_int64), n, nthreads, _p(out["rows"], C.c_uint32),
            _p(out["e"], C.c_uint16), _p(out["kv"], C.c_double), _p(out["gates"], C.c_double),
            _p(out["h"], C.c_double), _p(out["h_bf16"], C.c_uint16))
    if table is None:
        rc = lib().orc_forward(C.byref(gc), seed, *tail)
    else:
        codes, scales = _c(table[0], np.uint8), _c(table[1], np.uint8)
        nrows = codes.size // g.row_dim
        assert scales.size >= nrows * (g.row_dim // 32)
        rc = lib().orc_forward_table(C.byref(gc), _p(codes, C.c_uint8), _p(scales, C.c_uint8),
                                     nrows, *tail)
    if rc != 0:
        raise RuntimeError("orc_forward failed")
    return out
