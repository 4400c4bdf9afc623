"""ctypes front end of the C float64 oracle (``qsa_oracle.c``).

TEST INFRASTRUCTURE ONLY.  ``build()`` compiles the C file with the host's gcc
into ``oracle/_build/libqsa_oracle.so``; ``sparse_attention`` runs it on host
numpy arrays.  The arrays can come from any object carrying the
QSASparseAttentionRaggedPaged operands as attributes (``q``, ``kv_flat``,
``kv_shape``, ``page_stride``, ``input_row_offsets``, ``cache_lengths``,
``kv_lookup_table``, ``layer_idx``, ``token_indices``, ``counts``, ``scale``,
``group``, ``dtype``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libqsa_oracle.so")

ORACLE_DTYPES = {"f32": 0, "bf16": 1, "e4m3": 2}
_ERRORS = {1: "bad argument", 2: "index out of range", 3: "bad page", 4: "bad row", 5: "out of memory"}

_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int, row: int):
        super().__init__(f"oracle: {_ERRORS.get(code, code)} (row {row})")
        self.code = code
        self.row = row


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) if out of date."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.qsa_oracle_sparse_attention.restype = ctypes.c_int
        lib.qsa_oracle_sparse_attention.argtypes = [
            p, p, i64,
            p, ctypes.c_int, i64, i64, i64,
            p, i64,
            p, ctypes.c_int, i64, i64,
            i64, i64, i64,
            p, p, i64,
            i64, p, i64,
            p, ctypes.c_double, i64, ctypes.POINTER(i64),
        ]
        lib.qsa_oracle_msa_attention.restype = ctypes.c_int
        lib.qsa_oracle_msa_attention.argtypes = [
            p, p, i64,
            p, ctypes.c_int, i64, i64, i64,
            p, i64,
            p, i64, i64,
            i64, i64, i64,
            p, p, i64,
            i64, p, i64, ctypes.c_double, i64, ctypes.POINTER(i64),
        ]
        lib.qsa_oracle_compress_keys.restype = ctypes.c_int
        lib.qsa_oracle_compress_keys.argtypes = [
            p, i64, i64, i64,
            p, p, ctypes.c_int, i64,
            i64, p, p, ctypes.c_int,
            i64, i64, i64, i64,
            p, i64, i64, i64,
            ctypes.c_double,
        ]
        lib.qsa_oracle_latent_attention.restype = ctypes.c_int
        lib.qsa_oracle_latent_attention.argtypes = [
            p, p, i64,
            p, ctypes.c_int, i64, i64, i64,
            p, i64,
            p, i64, i64, i64, i64,
            p, p, i64,
            p, i64, i64, i64, i64,
            p, p, i64,
            i64, p, i64, p,
            i64, ctypes.c_double, ctypes.POINTER(i64),
        ]
        lib.qsa_oracle_decode.restype = None
        lib.qsa_oracle_decode.argtypes = [p, p, ctypes.c_int, i64]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def decode(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Raw storage (float32 / bf16 bits / e4m3 bits) -> exact float64."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.shape, dtype=np.float64)
    load().qsa_oracle_decode(_ptr(out), _ptr(raw), ORACLE_DTYPES[dtype], raw.size)
    return out


def sparse_attention(x, rows=None) -> np.ndarray:
    """float64 attention output for the query rows ``rows`` (all rows if None),
    shape ``[len(rows), num_q_heads, head_dim]``."""
    lib = load()
    total_q, nq, D = x.q.shape
    rows = np.arange(total_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, nq, D), dtype=np.float64)
    num_pages, two, L, P, nkv, Dk = x.kv_shape
    assert Dk == D and two == 2
    q = np.ascontiguousarray(x.q)
    kv = np.ascontiguousarray(x.kv_flat)
    off = np.ascontiguousarray(x.input_row_offsets, dtype=np.uint32)
    cl = np.ascontiguousarray(x.cache_lengths, dtype=np.uint32)
    tab = np.ascontiguousarray(x.kv_lookup_table, dtype=np.uint32)
    idx = np.ascontiguousarray(x.token_indices, dtype=np.int32)
    cnt = np.ascontiguousarray(x.counts, dtype=np.int32)
    bad = ctypes.c_int64(-1)
    code = lib.qsa_oracle_sparse_attention(
        _ptr(out), _ptr(rows), rows.size,
        _ptr(q), ORACLE_DTYPES[x.dtype], total_q, nq, D,
        _ptr(off), cl.size,
        _ptr(kv), ORACLE_DTYPES[x.dtype], num_pages, int(x.page_stride),
        L, P, nkv,
        _ptr(cl), _ptr(tab), tab.shape[1],
        int(x.layer_idx), _ptr(idx), idx.shape[1],
        _ptr(cnt), float(x.scale), int(x.group), ctypes.byref(bad),
    )
    if code != 0:
        raise OracleError(code, bad.value)
    return out


def msa_attention(x, rows=None) -> np.ndarray:
    """float64 block-sparse (MSA-style) attention output for the query rows
    ``rows`` (all if None): ``x`` also carries ``d_indices`` [nkv, total_q, topk]."""
    lib = load()
    total_q, nq, D = x.q.shape
    rows = np.arange(total_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, nq, D), dtype=np.float64)
    num_pages, two, L, P, nkv, Dk = x.kv_shape
    assert Dk == D and two == 2
    q = np.ascontiguousarray(x.q)
    kv = np.ascontiguousarray(x.kv_flat)
    off = np.ascontiguousarray(x.input_row_offsets, dtype=np.uint32)
    cl = np.ascontiguousarray(x.cache_lengths, dtype=np.uint32)
    tab = np.ascontiguousarray(x.kv_lookup_table, dtype=np.uint32)
    di = np.ascontiguousarray(x.d_indices, dtype=np.int32)
    assert di.shape[:2] == (nkv, total_q)
    bad = ctypes.c_int64(-1)
    code = lib.qsa_oracle_msa_attention(
        _ptr(out), _ptr(rows), rows.size,
        _ptr(q), ORACLE_DTYPES[x.dtype], total_q, nq, D,
        _ptr(off), cl.size,
        _ptr(kv), num_pages, int(x.page_stride),
        L, P, nkv,
        _ptr(cl), _ptr(tab), tab.shape[1],
        int(x.layer_idx), _ptr(di), di.shape[2], float(x.scale), int(x.group), ctypes.byref(bad),
    )
    if code != 0:
        raise OracleError(code, bad.value)
    return out


def compress_keys(x) -> np.ndarray:
    """float64 block keys [batch * max_blocks, head_dim] of a block-key
    compression call ``x`` (see qsa_oracle_compress_keys for the readings)."""
    lib = load()
    c = x.cache
    num_pages, two, L, P, nkv, D = c.kv_shape
    assert nkv == 1 and two == 2
    out = np.empty((x.batch * x.max_blocks, D), dtype=np.float64)
    kv = np.ascontiguousarray(c.kv_flat)
    tab = np.ascontiguousarray(c.kv_lookup_table, dtype=np.uint32)
    cnt = np.ascontiguousarray(x.key_counts, dtype=np.int32)
    gamma = np.ascontiguousarray(x.gamma)
    fr = np.ascontiguousarray(x.freqs_cis)
    code = lib.qsa_oracle_compress_keys(
        _ptr(out), x.batch, x.max_blocks, D,
        _ptr(gamma), _ptr(fr), ORACLE_DTYPES[x.freq_dtype], fr.shape[0],
        x.rotary_dim, _ptr(cnt), _ptr(kv), ORACLE_DTYPES[x.dtype],
        num_pages, int(c.page_stride), L, P,
        _ptr(tab), tab.shape[1], int(c.layer_idx), int(x.ratio),
        float(x.eps),
    )
    if code != 0:
        raise OracleError(code, -1)
    return out


def latent_attention(x, rows=None) -> np.ndarray:
    """float64 latent sparse attention (window + listed compressed entries +
    sinks) for the query rows ``rows`` (all if None)."""
    lib = load()
    a, c = x.swa, x.comp
    total_q, H, D = a.q.shape
    rows = np.arange(total_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, H, D), dtype=np.float64)
    keep = []

    def arr(v, dt=None):
        v = np.ascontiguousarray(v, dtype=dt) if dt is not None else np.ascontiguousarray(v)
        keep.append(v)
        return _ptr(v)

    ci = np.ascontiguousarray(x.comp_indices, dtype=np.int32)
    bad = ctypes.c_int64(-1)
    code = lib.qsa_oracle_latent_attention(
        _ptr(out), _ptr(rows), rows.size,
        arr(a.q), ORACLE_DTYPES[a.dtype], total_q, H, D,
        arr(a.input_row_offsets, np.uint32), a.batch,
        arr(a.kv_flat), a.kv_shape[0], int(a.page_stride), a.kv_shape[2], a.kv_shape[3],
        arr(a.cache_lengths, np.uint32), arr(a.kv_lookup_table, np.uint32), a.kv_lookup_table.shape[1],
        arr(c.kv_flat), c.kv_shape[0], int(c.page_stride), c.kv_shape[2], c.kv_shape[3],
        arr(c.cache_lengths, np.uint32), arr(c.kv_lookup_table, np.uint32), c.kv_lookup_table.shape[1],
        int(a.layer_idx), _ptr(ci), ci.shape[1], arr(x.attn_sink, np.float32),
        int(x.window), float(a.scale), ctypes.byref(bad),
    )
    if code != 0:
        raise OracleError(code, bad.value)
    return out
