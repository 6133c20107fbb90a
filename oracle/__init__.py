"""CPU oracle for the paged KV-cache attention step (fp64, plain loops).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The product library
never loads it and shares no code with it: the arithmetic lives in
``pkv_oracle.c`` (compiled with gcc by :func:`build`), and this module only
marshals numpy arrays into it.

Page sources and the readings taken where the pages are silent are listed in
the header of ``pkv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into a shared library with gcc (OpenMP if present).

    PKV_ORACLE_LIB names an already built library to load instead (the
    mutation tests use it to load a copy with a planted mistake).
    """
    override = os.environ.get("PKV_ORACLE_LIB")
    if override:
        return override
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    compile_to(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_to(src: str, out: str) -> None:
    """gcc -O2 -shared of one oracle source file (with OpenMP when gcc has it)."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_kv_store.argtypes = [_p, _i64, _i64, _i64, _i64, _i64, _i64, _p, _p,
                                          _i64, _p, _i64]
            L.oracle_decode_attn.argtypes = [_p, _i64, _i64, _i64, _i64, _i64, _i64, _p,
                                             _p, _i64, _p, _p, _i64, _i64, _dbl, _p, _p]
            L.oracle_extend_attn.argtypes = [_p, _i64, _i64, _i64, _i64, _i64, _i64, _p,
                                             _p, _p, _i64, _p, _p, _i64, _i64, _dbl, _p,
                                             _p]
            L.oracle_merge_lse.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p]
            L.oracle_set_threads.argtypes = [ctypes.c_int]
            L.oracle_max_threads.restype = ctypes.c_int
            for f in (L.oracle_kv_store, L.oracle_decode_attn, L.oracle_extend_attn,
                      L.oracle_merge_lse):
                f.restype = ctypes.c_int
            _lib = L
    return _lib


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: rejected its arguments (code {rc})")


def _pool_dims(pool: np.ndarray):
    if pool.dtype != np.uint16 or pool.ndim != 6 or pool.shape[0] != 2:
        raise ValueError("pool must be a uint16 (bf16 bits) array of shape "
                         "(2, layers, pages, page_size, kv_heads, head_dim)")
    if not pool.flags.c_contiguous:
        raise ValueError("pool must be C-contiguous")
    _, L, NP, P, Hkv, D = pool.shape
    return L, NP, P, Hkv, D


def kv_store(pool: np.ndarray, layer: int, k: np.ndarray, v: np.ndarray,
             out_loc: np.ndarray) -> None:
    """pool[0|1, layer, slot(out_loc[i])] = k[i] | v[i]; pool is updated in place.

    k, v: uint16 bf16 bits, [N, Hkv, D] (any row stride along N).
    """
    L, NP, P, Hkv, D = _pool_dims(pool)
    n = int(out_loc.shape[0])
    k2 = np.ascontiguousarray(k.reshape(n, Hkv * D), dtype=np.uint16)
    v2 = np.ascontiguousarray(v.reshape(n, Hkv * D), dtype=np.uint16)
    loc = _c(out_loc, np.int32)
    rc = lib().oracle_kv_store(_ptr(pool), L, NP, P, Hkv, D, int(layer), _ptr(k2),
                               _ptr(v2), Hkv * D, _ptr(loc), n)
    _check(rc, "kv_store")


def decode_attn(pool: np.ndarray, layer: int, q: np.ndarray, page_table: np.ndarray,
                seq_lens: np.ndarray, scale: float, table_idx: np.ndarray | None = None):
    """Decode attention. q: uint16 [B, Hq, D]. Returns (o [B,Hq,D], lse [B,Hq]) in fp64."""
    L, NP, P, Hkv, D = _pool_dims(pool)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim does not match the pool")
    qq = _c(q, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ti = _c(table_idx, np.int32)
    o = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib().oracle_decode_attn(_ptr(pool), L, NP, P, Hkv, D, int(layer), _ptr(qq),
                                  _ptr(pt), pt.shape[1], _ptr(ti), _ptr(sl), B, Hq,
                                  float(scale), _ptr(o), _ptr(lse))
    _check(rc, "decode_attn")
    return o, lse


def extend_attn(pool: np.ndarray, layer: int, q: np.ndarray, qo_indptr: np.ndarray,
                page_table: np.ndarray, seq_lens: np.ndarray, scale: float,
                table_idx: np.ndarray | None = None):
    """Extend attention. q: uint16 [T, Hq, D]. Returns (o [T,Hq,D], lse [T,Hq]) in fp64."""
    L, NP, P, Hkv, D = _pool_dims(pool)
    T, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim does not match the pool")
    B = int(seq_lens.shape[0])
    ind = _c(qo_indptr, np.int32)
    if ind.shape[0] != B + 1 or int(ind[-1]) != T:
        raise ValueError("qo_indptr must have batch+1 entries ending at total_q")
    qq = _c(q, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ti = _c(table_idx, np.int32)
    o = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    rc = lib().oracle_extend_attn(_ptr(pool), L, NP, P, Hkv, D, int(layer), _ptr(qq),
                                  _ptr(ind), _ptr(pt), pt.shape[1], _ptr(ti), _ptr(sl),
                                  B, Hq, float(scale), _ptr(o), _ptr(lse))
    _check(rc, "extend_attn")
    return o, lse


def merge_lse(o_a, lse_a, o_b, lse_b):
    """Merge two attention states. o_*: [rows, H, D], lse_*: [rows, H]; fp64 out."""
    o_a = _c(o_a, np.float64)
    o_b = _c(o_b, np.float64)
    lse_a = _c(lse_a, np.float64)
    lse_b = _c(lse_b, np.float64)
    rows, H, D = o_a.shape
    o = np.zeros_like(o_a)
    lse = np.zeros_like(lse_a)
    rc = lib().oracle_merge_lse(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, H,
                                D, _ptr(o), _ptr(lse))
    _check(rc, "merge_lse")
    return o, lse
