"""Python binding of libengram.so, the Engram per-layer forward step on one GB300.

Argument marshalling only: every function below forwards to the C function of
the same name declared in ``include/engram.h``; every step of the forward path
runs in the library's CUDA kernels.  Pointers may be given as ints, torch
tensors (``data_ptr()``) or numpy arrays (host memory); streams as ints,
``torch.cuda.Stream`` objects or None (legacy default stream).  A non-zero
status raises ``EngramError`` with the library's message.  If the library has
not been built the first call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libengram.so")

DEAD = 0xFFFFFFFF
MASKED = 0xFFFFFFFF

STATUS = {0: "OK", 1: "EINVAL", 2: "ENOMEM", 3: "ECUDA", 4: "ESTATE", 5: "ETIMEOUT",
          6: "EUNSUPPORTED", 7: "EBOUNDS"}
OK, EINVAL, ENOMEM, ECUDA, ESTATE, ETIMEOUT, EUNSUPPORTED, EBOUNDS = range(8)

# Names exported by the library (the declarations of include/engram.h).
EXPORTS = (
    "engram_ctx_create", "engram_ctx_destroy", "engram_layer_params",
    "engram_layer_set_multipliers", "engram_layer_bind", "engram_layer_info",
    "engram_table_fill", "engram_table_fill_bf16",
    "engram_session_create", "engram_session_fork", "engram_session_reset",
    "engram_session_destroy", "engram_session_append", "engram_batch_append",
    "engram_workspace_bytes", "engram_hash", "engram_gather_dequant", "engram_project",
    "engram_gate", "engram_forward", "engram_forward_noalloc", "engram_forward_staged",
    "engram_forward_staged_workspace_bytes", "engram_stage_rows", "engram_forward_staged_rows",
    "engram_project_windows", "engram_prepass", "engram_gate_bf16kv",
    "engram_layer_bind_shard", "engram_scale_range", "engram_hash_by_bucket",
    "engram_raw_row_bytes", "engram_host_table_alloc", "engram_host_table_free",
    "engram_shard_gather_raw", "engram_stage_raw_rows",
    "engram_sync", "engram_ctx_set_wait_limit", "engram_debug_starve_operand",
    "engram_last_error",
)


class EngramError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class CtxDesc(C.Structure):
    _fields_ = [
        ("vocab", C.c_uint32), ("vc", C.c_uint32), ("min_n", C.c_uint32), ("max_n", C.c_uint32),
        ("heads", C.c_uint32), ("row_dim", C.c_uint32), ("hc", C.c_uint32), ("d", C.c_uint32),
        ("pad_cid", C.c_uint32), ("n_layers", C.c_uint32), ("eps", C.c_double),
        ("layer_seeds", C.POINTER(C.c_uint64)), ("bucket_bases", C.POINTER(C.c_uint64)),
    ]


BIND_BF16_OPERANDS = 1
BIND_TABLE_BF16 = 2
KV_F32, KV_BF16 = 0, 1  # engram_prepass: kv as fp32, or rounded once to BF16


class LayerWeights(C.Structure):
    _fields_ = [
        ("table", C.c_void_p), ("scales", C.c_void_p), ("rows", C.c_uint64),
        ("wkv", C.c_void_p), ("wq", C.c_void_p), ("wk", C.c_void_p), ("flags", C.c_uint32),
    ]


class LayerInfo(C.Structure):
    _fields_ = [
        ("rows", C.c_uint64), ("bound", C.c_int32), ("fp16_operands", C.c_int32),
        ("scale_min", C.c_uint32), ("scale_max", C.c_uint32), ("wkv_exp", C.c_int32),
        ("a_exp_shift", C.c_int32), ("bucket_gather", C.c_int32), ("table_bf16", C.c_int32),
    ]


_lib = None


def lib() -> C.CDLL:
    """Load libengram.so (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(engram_gram_conditional_gb300.build.build())")
        L = C.CDLL(LIB_PATH)
        vp, i64, st = C.c_void_p, C.c_int64, C.c_int
        sig = {
            "engram_ctx_create": [C.POINTER(CtxDesc), vp, C.POINTER(vp)],
            "engram_ctx_destroy": [vp],
            "engram_layer_params": [vp, C.c_int, vp, vp, vp, vp],
            "engram_layer_set_multipliers": [vp, C.c_int, vp],
            "engram_layer_bind": [vp, C.c_int, C.POINTER(LayerWeights)],
            "engram_layer_info": [vp, C.c_int, C.POINTER(LayerInfo)],
            "engram_table_fill": [vp, C.c_uint64, vp, vp, C.c_uint64, C.c_uint64, vp],
            "engram_table_fill_bf16": [vp, C.c_uint64, vp, C.c_uint64, C.c_uint64, vp],
            "engram_session_create": [vp, C.POINTER(vp)],
            "engram_session_fork": [vp, C.POINTER(vp)],
            "engram_session_reset": [vp],
            "engram_session_destroy": [vp],
            "engram_session_append": [vp, vp, vp, i64, vp],
            "engram_batch_append": [vp, vp, vp, i64, vp],
            "engram_hash": [vp, C.c_int, vp, i64, vp, vp],
            "engram_gather_dequant": [vp, C.c_int, vp, i64, vp, vp],
            "engram_project": [vp, C.c_int, vp, i64, vp, vp],
            "engram_gate": [vp, C.c_int, vp, vp, i64, vp, vp, vp],
            "engram_forward": [vp, C.c_int, vp, i64, vp, vp, vp, vp],
            "engram_project_windows": [vp, C.c_int, vp, i64, vp, vp],
            "engram_prepass": [vp, C.c_int, vp, i64, vp, C.c_int, vp, vp],
            "engram_gate_bf16kv": [vp, C.c_int, vp, vp, i64, vp, vp, vp],
            "engram_forward_noalloc": [vp, C.c_int, vp, i64, vp, vp, vp],
            "engram_forward_staged": [vp, C.c_int, vp, i64, vp, vp, vp, vp],
            "engram_stage_rows": [vp, C.c_int, vp, i64, vp, vp],
            "engram_forward_staged_rows": [vp, C.c_int, vp, i64, vp, vp, vp, vp],
            "engram_sync": [vp, vp],
            "engram_ctx_set_wait_limit": [vp, i64],
            "engram_layer_bind_shard": [vp, C.c_int, C.POINTER(LayerWeights), C.c_uint64,
                                        C.c_uint32, C.c_uint32],
            "engram_scale_range": [vp, vp, C.c_uint64, C.POINTER(C.c_uint32),
                                   C.POINTER(C.c_uint32)],
            "engram_host_table_alloc": [C.c_uint64, C.POINTER(vp)],
            "engram_host_table_free": [vp, C.c_uint64],
            "engram_hash_by_bucket": [vp, C.c_int, vp, i64, vp, vp],
            "engram_shard_gather_raw": [vp, C.c_int, vp, i64, vp, vp],
            "engram_stage_raw_rows": [vp, C.c_int, vp, vp, i64, vp, vp],
            "engram_debug_starve_operand": [vp, C.c_int],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = st
        for name in ("engram_workspace_bytes", "engram_forward_staged_workspace_bytes"):
            getattr(L, name).argtypes = [vp, i64]
            getattr(L, name).restype = C.c_size_t
        L.engram_raw_row_bytes.argtypes = [vp]
        L.engram_raw_row_bytes.restype = C.c_size_t
        L.engram_last_error.argtypes = []
        L.engram_last_error.restype = C.c_char_p
        _lib = L
    return _lib


def engram_last_error() -> str:
    return lib().engram_last_error().decode()


def _check(status: int):
    if status != OK:
        raise EngramError(status, engram_last_error())


def _ptr(x):
    """Address of a buffer: int, None, torch tensor, numpy array or ctypes object."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"], "numpy buffers must be C-contiguous"
        return x.ctypes.data
    if isinstance(x, C.c_void_p):
        return x.value
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


# ---- context and layers ---------------------------------------------------------------

def engram_ctx_create(vocab, vc, token_map, layer_seeds, bucket_bases, *, min_n=2, max_n=4,
                      heads=8, row_dim=256, hc=4, d=5120, pad_cid=0, eps=1e-6):
    seeds = np.ascontiguousarray(layer_seeds, dtype=np.uint64)
    bases = np.ascontiguousarray(bucket_bases, dtype=np.uint64)
    tmap = np.ascontiguousarray(token_map, dtype=np.uint32)
    if tmap.size != vocab:
        raise EngramError(EINVAL, "token_map must have vocab entries")
    desc = CtxDesc(vocab, vc, min_n, max_n, heads, row_dim, hc, d, pad_cid, len(seeds), eps,
                   seeds.ctypes.data_as(C.POINTER(C.c_uint64)),
                   bases.ctypes.data_as(C.POINTER(C.c_uint64)))
    out = C.c_void_p()
    _check(lib().engram_ctx_create(C.byref(desc), tmap.ctypes.data, C.byref(out)))
    return out


def engram_ctx_destroy(ctx):
    _check(lib().engram_ctx_destroy(ctx))


def engram_layer_params(ctx, layer: int, nb: int):
    mult = np.zeros((nb, 4), np.uint64)
    prime = np.zeros(nb, np.uint64)
    offset = np.zeros(nb, np.uint64)
    rows = np.zeros(1, np.uint64)
    _check(lib().engram_layer_params(ctx, layer, mult.ctypes.data, prime.ctypes.data,
                                     offset.ctypes.data, rows.ctypes.data))
    return mult, prime, offset, int(rows[0])


def engram_layer_set_multipliers(ctx, layer: int, mult):
    m = np.ascontiguousarray(mult, dtype=np.uint64)
    _check(lib().engram_layer_set_multipliers(ctx, layer, m.ctypes.data))


def engram_layer_bind(ctx, layer: int, table, scales, rows: int, wkv, wq, wk, flags: int = 0):
    w = LayerWeights(_ptr(table), _ptr(scales), rows, _ptr(wkv), _ptr(wq), _ptr(wk), flags)
    _check(lib().engram_layer_bind(ctx, layer, C.byref(w)))


def engram_layer_info(ctx, layer: int) -> dict:
    info = LayerInfo()
    _check(lib().engram_layer_info(ctx, layer, C.byref(info)))
    return {name: getattr(info, name) for name, _ in LayerInfo._fields_}


def engram_table_fill(ctx, seed: int, data, scale, row_begin: int, row_end: int, stream=None):
    _check(lib().engram_table_fill(ctx, seed, _ptr(data), _ptr(scale), row_begin, row_end,
                                   _stream(stream)))


def engram_table_fill_bf16(ctx, seed: int, data, row_begin: int, row_end: int, stream=None):
    _check(lib().engram_table_fill_bf16(ctx, seed, _ptr(data), row_begin, row_end,
                                        _stream(stream)))


# ---- sessions -------------------------------------------------------------------------

def engram_session_create(ctx):
    out = C.c_void_p()
    _check(lib().engram_session_create(ctx, C.byref(out)))
    return out


def engram_session_fork(session):
    out = C.c_void_p()
    _check(lib().engram_session_fork(session, C.byref(out)))
    return out


def engram_session_reset(session):
    _check(lib().engram_session_reset(session))


def engram_session_destroy(session):
    _check(lib().engram_session_destroy(session))


def engram_session_append(session, tokens, is_image=None, windows_out=None):
    """Append tokens; returns the windows (uint32 [n][4], host)."""
    tk = np.ascontiguousarray(tokens, dtype=np.int32)
    im = None if is_image is None else np.ascontiguousarray(is_image, dtype=np.uint8)
    out = np.empty((tk.size, 4), np.uint32) if windows_out is None else windows_out
    _check(lib().engram_session_append(session, tk.ctypes.data,
                                       None if im is None else im.ctypes.data, tk.size,
                                       _ptr(out)))
    return out


def engram_batch_append(sessions, tokens, is_image=None, windows_out=None):
    """Append one token to each session; returns the windows (uint32 [n][4], host)."""
    arr = (C.c_void_p * len(sessions))(*[s.value if isinstance(s, C.c_void_p) else s
                                         for s in sessions])
    tk = np.ascontiguousarray(tokens, dtype=np.int32)
    im = None if is_image is None else np.ascontiguousarray(is_image, dtype=np.uint8)
    out = np.empty((len(sessions), 4), np.uint32) if windows_out is None else windows_out
    _check(lib().engram_batch_append(C.cast(arr, C.c_void_p), tk.ctypes.data,
                                     None if im is None else im.ctypes.data, len(sessions),
                                     _ptr(out)))
    return out


# ---- device steps -----------------------------------------------------------------------

def engram_workspace_bytes(ctx, T: int) -> int:
    return int(lib().engram_workspace_bytes(ctx, T))


def engram_hash(ctx, layer, d_windows, T, d_rows, stream=None):
    _check(lib().engram_hash(ctx, layer, _ptr(d_windows), T, _ptr(d_rows), _stream(stream)))


def engram_gather_dequant(ctx, layer, d_rows, T, d_emb, stream=None):
    _check(lib().engram_gather_dequant(ctx, layer, _ptr(d_rows), T, _ptr(d_emb), _stream(stream)))


def engram_project(ctx, layer, d_emb, T, d_kv, stream=None):
    _check(lib().engram_project(ctx, layer, _ptr(d_emb), T, _ptr(d_kv), _stream(stream)))


def engram_gate(ctx, layer, d_kv, d_windows, T, d_hidden, d_gates=None, stream=None):
    _check(lib().engram_gate(ctx, layer, _ptr(d_kv), _ptr(d_windows), T, _ptr(d_hidden),
                             _ptr(d_gates), _stream(stream)))


def engram_forward(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates=None, stream=None):
    _check(lib().engram_forward(ctx, layer, _ptr(d_windows), T, _ptr(d_hidden), _ptr(d_workspace),
                                _ptr(d_gates), _stream(stream)))


def engram_forward_staged_workspace_bytes(ctx, T: int) -> int:
    return int(lib().engram_forward_staged_workspace_bytes(ctx, T))


def engram_forward_staged(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates=None,
                          stream=None):
    _check(lib().engram_forward_staged(ctx, layer, _ptr(d_windows), T, _ptr(d_hidden),
                                       _ptr(d_workspace), _ptr(d_gates), _stream(stream)))


def engram_stage_rows(ctx, layer, d_windows, T, d_workspace, stream=None):
    _check(lib().engram_stage_rows(ctx, layer, _ptr(d_windows), T, _ptr(d_workspace),
                                   _stream(stream)))


def engram_forward_staged_rows(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates=None,
                               stream=None):
    _check(lib().engram_forward_staged_rows(ctx, layer, _ptr(d_windows), T, _ptr(d_hidden),
                                            _ptr(d_workspace), _ptr(d_gates), _stream(stream)))


def engram_forward_noalloc(ctx, layer, d_windows, T, d_hidden, d_gates=None, stream=None):
    """engram_forward without a workspace argument, for callers that cannot allocate:
    the scratch is the library's built-in 8 MiB device buffer (see include/engram.h)."""
    _check(lib().engram_forward_noalloc(ctx, layer, _ptr(d_windows), T, _ptr(d_hidden),
                                        _ptr(d_gates), _stream(stream)))


def engram_project_windows(ctx, layer, d_windows, T, d_kv, stream=None):
    _check(lib().engram_project_windows(ctx, layer, _ptr(d_windows), T, _ptr(d_kv),
                                        _stream(stream)))


def engram_prepass(ctx, layer, d_windows, T, d_kv, kv_format, d_workspace, stream=None):
    _check(lib().engram_prepass(ctx, layer, _ptr(d_windows), T, _ptr(d_kv), int(kv_format),
                                _ptr(d_workspace), _stream(stream)))


def engram_gate_bf16kv(ctx, layer, d_kv, d_windows, T, d_hidden, d_gates=None, stream=None):
    _check(lib().engram_gate_bf16kv(ctx, layer, _ptr(d_kv), _ptr(d_windows), T, _ptr(d_hidden),
                                    _ptr(d_gates), _stream(stream)))


def engram_layer_bind_shard(ctx, layer: int, table, scales, rows: int, wkv, wq, wk, row_lo: int,
                            scale_min: int, scale_max: int, flags: int = 0):
    w = LayerWeights(_ptr(table), _ptr(scales), rows, _ptr(wkv), _ptr(wq), _ptr(wk), flags)
    _check(lib().engram_layer_bind_shard(ctx, layer, C.byref(w), row_lo, scale_min, scale_max))


def engram_scale_range(ctx, scales, n: int):
    """(min, max) of n E8M0 bytes on the device (255, 0 for n = 0)."""
    lo, hi = C.c_uint32(), C.c_uint32()
    _check(lib().engram_scale_range(ctx, _ptr(scales), n, C.byref(lo), C.byref(hi)))
    return lo.value, hi.value


def engram_host_table_alloc(nbytes: int) -> int:
    """Registered, huge-page-advised host memory for a table read through UVA
    (see include/engram.h); returns its address (host and device)."""
    out = C.c_void_p()
    _check(lib().engram_host_table_alloc(nbytes, C.byref(out)))
    return out.value


def engram_host_table_free(ptr: int, nbytes: int):
    _check(lib().engram_host_table_free(ptr, nbytes))


def engram_hash_by_bucket(ctx, layer, d_windows, T, d_rows_bm, stream=None):
    _check(lib().engram_hash_by_bucket(ctx, layer, _ptr(d_windows), T, _ptr(d_rows_bm),
                                       _stream(stream)))


def engram_raw_row_bytes(ctx) -> int:
    return int(lib().engram_raw_row_bytes(ctx))


def engram_shard_gather_raw(ctx, layer, d_ids, n, d_raw, stream=None):
    _check(lib().engram_shard_gather_raw(ctx, layer, _ptr(d_ids), n, _ptr(d_raw), _stream(stream)))


def engram_stage_raw_rows(ctx, layer, d_rows_bm, d_raw_bm, T, d_workspace, stream=None):
    _check(lib().engram_stage_raw_rows(ctx, layer, _ptr(d_rows_bm), _ptr(d_raw_bm), T,
                                       _ptr(d_workspace), _stream(stream)))


def engram_ctx_set_wait_limit(ctx, ns: int):
    _check(lib().engram_ctx_set_wait_limit(ctx, ns))


def engram_debug_starve_operand(ctx, on: bool):
    _check(lib().engram_debug_starve_operand(ctx, 1 if on else 0))


def engram_sync(ctx, stream=None):
    _check(lib().engram_sync(ctx, _stream(stream)))
