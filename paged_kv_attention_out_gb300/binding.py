"""Thin ctypes binding of the pkv C ABI (include/pkv.h), same names.

Argument marshalling only: every function takes torch tensors that already
live on the current CUDA device, checks their dtypes and shapes, and passes
raw pointers, sizes and the current stream to the C entry point of the same
name. All arithmetic runs in the library's CUDA kernels. If the library is
not built, importing this module's functions raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_c_int32 = ctypes.c_int32
_c_int64 = ctypes.c_int64
_p = ctypes.c_void_p


class PkvPool(ctypes.Structure):
    _fields_ = [("base", _p), ("num_layers", _c_int32), ("num_pages", _c_int64),
                ("page_size", _c_int32), ("num_kv_heads", _c_int32), ("head_dim", _c_int32)]


PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_WORKSPACE_TOO_SMALL", 4: "PKV_ERR_CUDA"}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libpkv.so (built by __graft_entry__.build()); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"pkv CUDA library not built ({path}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    pool_p = ctypes.POINTER(PkvPool)
    L.pkv_init.restype = ctypes.c_int
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_last_error.restype = ctypes.c_char_p
    L.pkv_kv_store.restype = ctypes.c_int
    L.pkv_kv_store.argtypes = [pool_p, _c_int32, _p, _p, _c_int64, _p, _c_int64, _p]
    L.pkv_decode_workspace_size.restype = ctypes.c_size_t
    L.pkv_decode_workspace_size.argtypes = [_c_int32] * 5
    L.pkv_paged_decode_attn.restype = ctypes.c_int
    L.pkv_paged_decode_attn.argtypes = [pool_p, _c_int32, _p, _p, _p, _p, _c_int64, _p, _p,
                                        _c_int32, _c_int32, ctypes.c_float, _c_int32, _p,
                                        ctypes.c_size_t, _p]
    L.pkv_paged_decode_attn_store.restype = ctypes.c_int
    L.pkv_paged_decode_attn_store.argtypes = [pool_p, _c_int32, _p, _p, _p, _c_int64, _p, _p, _p,
                                              _c_int64, _p, _p, _c_int32, _c_int32,
                                              ctypes.c_float, _c_int32, _p, ctypes.c_size_t, _p]
    L.pkv_paged_decode_attn_noalloc.restype = ctypes.c_int
    L.pkv_paged_decode_attn_noalloc.argtypes = [pool_p, _c_int32, _p, _p, _p, _p, _c_int64, _p,
                                                _p, _c_int32, _c_int32, ctypes.c_float,
                                                _c_int32, _p]
    L.pkv_extend_workspace_size.restype = ctypes.c_size_t
    L.pkv_extend_workspace_size.argtypes = [_c_int32] * 4 + [_c_int64]
    L.pkv_paged_extend_attn.restype = ctypes.c_int
    L.pkv_paged_extend_attn.argtypes = [pool_p, _c_int32, _p, _p, _p, _p, _p, _c_int64, _p, _p,
                                        _c_int32, _c_int32, _c_int32, ctypes.c_float,
                                        _c_int32, _c_int64, _p, ctypes.c_size_t, _p]
    L.pkv_paged_extend_attn_store.restype = ctypes.c_int
    L.pkv_paged_extend_attn_store.argtypes = [pool_p, _c_int32, _p, _p, _p, _c_int64, _p, _p, _p,
                                              _p, _c_int64, _p, _p, _c_int32, _c_int32,
                                              _c_int32, ctypes.c_float, _c_int32, _c_int64, _p,
                                              ctypes.c_size_t, _p]
    L.pkv_cascade_workspace_size.restype = ctypes.c_size_t
    L.pkv_cascade_workspace_size.argtypes = [_c_int32] * 7
    L.pkv_paged_cascade_decode_attn.restype = ctypes.c_int
    L.pkv_paged_cascade_decode_attn.argtypes = [pool_p, _c_int32, _p, _p, _p, _p, _c_int64, _p, _p,
                                                _p, _c_int32, _p, _c_int64, _p, _p, _c_int32,
                                                _c_int32, ctypes.c_float, _c_int32, _c_int32, _p,
                                                ctypes.c_size_t, _p]
    L.pkv_merge_lse.restype = ctypes.c_int
    L.pkv_merge_lse.argtypes = [_p, _p, _p, _p, _p, _c_int32, _p, _c_int64, _c_int32,
                                _c_int32, _p]
    L.pkv_read_device_errors.restype = ctypes.c_int
    L.pkv_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    _lib = L
    return L


def _check(status: int) -> None:
    if status != PKV_OK:
        msg = load().pkv_last_error().decode(errors="replace")
        raise PkvError(status, msg)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _want(t: torch.Tensor, dtype, name: str, ndim: int | None = None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _contig(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pool_struct(pool: torch.Tensor) -> PkvPool:
    """Descriptor of a (2, layers, pages, page_size, kv_heads, head_dim) bf16 pool."""
    _want(pool, torch.bfloat16, "pool", 6)
    _contig(pool, "pool")
    if pool.shape[0] != 2:
        raise ValueError("pool dim 0 must be 2 (K, V)")
    _, L, NP, P, H, D = pool.shape
    return PkvPool(pool.data_ptr(), L, NP, P, H, D)


def pkv_init() -> None:
    _check(load().pkv_init())


def pkv_kv_store(pool, layer: int, k, v, out_loc, stream=None) -> None:
    """pool[0|1, layer, out_loc[i]] = k[i] | v[i]; k, v [N, Hkv, D] bf16 (row stride free)."""
    ps = pool_struct(pool)
    _want(k, torch.bfloat16, "k", 3)
    _want(v, torch.bfloat16, "v", 3)
    _want(out_loc, torch.int32, "out_loc", 1)
    _contig(out_loc, "out_loc")
    n = out_loc.shape[0]
    if k.shape != v.shape or k.shape[0] != n:
        raise ValueError("k, v must be [N, Hkv, D] with N = len(out_loc)")
    if k.stride(0) != v.stride(0) or k.stride(1) != k.shape[2] or k.stride(2) != 1 \
            or v.stride(1) != v.shape[2] or v.stride(2) != 1:
        raise ValueError("k and v rows must share a row stride with heads/dims contiguous")
    _check(load().pkv_kv_store(ctypes.byref(ps), int(layer), _ptr(k), _ptr(v), k.stride(0),
                               _ptr(out_loc), n, _stream(stream)))


def pkv_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              max_seq_len_hint: int) -> int:
    return int(load().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                max_seq_len_hint))


def pkv_paged_decode_attn(pool, layer: int, q, o, lse, page_table, seq_lens, scale: float,
                          max_seq_len_hint: int, workspace=None, table_idx=None,
                          stream=None) -> None:
    """Decode attention; q, o [B, Hq, D] bf16; lse [B, Hq] fp32 or None."""
    ps = pool_struct(pool)
    _want(q, torch.bfloat16, "q", 3)
    _want(o, torch.bfloat16, "o", 3)
    _contig(q, "q")
    _contig(o, "o")
    _want(page_table, torch.int32, "page_table", 2)
    _contig(page_table, "page_table")
    _want(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    if o.shape != q.shape or seq_lens.shape[0] != B:
        raise ValueError("o must match q and seq_lens must have batch entries")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_decode_attn(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(o), _ptr(lse), _ptr(page_table),
        page_table.shape[1], _ptr(table_idx), _ptr(seq_lens), B, Hq, float(scale),
        int(max_seq_len_hint), _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_paged_decode_attn_store(pool, layer: int, q, k_new, v_new, o, lse, page_table, seq_lens,
                                scale: float, max_seq_len_hint: int, workspace=None,
                                table_idx=None, stream=None) -> None:
    """Decode step with store_kv fused: k_new, v_new [B, Hkv, D] bf16 go to key
    seq_lens[b] - 1 of each row, then decode as pkv_paged_decode_attn."""
    ps = pool_struct(pool)
    _want(q, torch.bfloat16, "q", 3)
    _want(o, torch.bfloat16, "o", 3)
    _contig(q, "q")
    _contig(o, "o")
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _want(t, torch.bfloat16, name, 3)
    if k_new.stride(0) != v_new.stride(0) or k_new.stride(1) != k_new.shape[2] \
            or k_new.stride(2) != 1 or v_new.stride(1) != v_new.shape[2] or v_new.stride(2) != 1:
        raise ValueError("k_new and v_new rows must share a row stride with heads/dims contiguous")
    _want(page_table, torch.int32, "page_table", 2)
    _contig(page_table, "page_table")
    _want(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    if o.shape != q.shape or seq_lens.shape[0] != B or k_new.shape[0] != B:
        raise ValueError("o must match q; seq_lens and k_new must have batch entries")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_decode_attn_store(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new), k_new.stride(0), _ptr(o),
        _ptr(lse), _ptr(page_table), page_table.shape[1], _ptr(table_idx), _ptr(seq_lens), B, Hq,
        float(scale), int(max_seq_len_hint), _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_paged_decode_attn_noalloc(pool, layer: int, q, o, lse, page_table, seq_lens,
                                  scale: float, max_seq_len_hint: int, table_idx=None,
                                  stream=None) -> None:
    """Decode attention with no workspace, for callers that cannot allocate.

    The split-KV scratch is a fixed library-owned device array (32 MiB), so
    nothing is allocated; calls whose kernels overlap on the GPU race on it.
    """
    ps = pool_struct(pool)
    _want(q, torch.bfloat16, "q", 3)
    _want(o, torch.bfloat16, "o", 3)
    _contig(q, "q")
    _contig(o, "o")
    _want(page_table, torch.int32, "page_table", 2)
    _contig(page_table, "page_table")
    _want(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    if o.shape != q.shape or seq_lens.shape[0] != B:
        raise ValueError("o must match q and seq_lens must have batch entries")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    _check(load().pkv_paged_decode_attn_noalloc(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(o), _ptr(lse), _ptr(page_table),
        page_table.shape[1], _ptr(table_idx), _ptr(seq_lens), B, Hq, float(scale),
        int(max_seq_len_hint), _stream(stream)))


def pkv_extend_workspace_size(batch: int, num_kv_heads: int, head_dim: int,
                              max_seq_len_hint: int, max_total_keys_hint: int = 0) -> int:
    """max_total_keys_hint: a bound on the sum of the call's seq_lens (0: none,
    batch x max_seq_len_hint is used)."""
    return int(load().pkv_extend_workspace_size(batch, num_kv_heads, head_dim,
                                                max_seq_len_hint, int(max_total_keys_hint)))


def pkv_paged_extend_attn(pool, layer: int, q, qo_indptr, o, lse, page_table, seq_lens,
                          scale: float, max_seq_len_hint: int, workspace, table_idx=None,
                          stream=None, max_total_keys_hint: int = 0) -> None:
    """Extend attention; q, o [T, Hq, D] bf16; qo_indptr [B+1]; lse [T, Hq] fp32 or None;
    workspace: device tensor of at least pkv_extend_workspace_size(...) bytes for the same
    hints."""
    ps = pool_struct(pool)
    _want(q, torch.bfloat16, "q", 3)
    _want(o, torch.bfloat16, "o", 3)
    _contig(q, "q")
    _contig(o, "o")
    _want(qo_indptr, torch.int32, "qo_indptr", 1)
    _want(page_table, torch.int32, "page_table", 2)
    _contig(page_table, "page_table")
    _want(seq_lens, torch.int32, "seq_lens", 1)
    T, Hq, D = q.shape
    B = seq_lens.shape[0]
    if o.shape != q.shape or qo_indptr.shape[0] != B + 1:
        raise ValueError("o must match q and qo_indptr must have batch+1 entries")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    if workspace is not None:
        _contig(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_extend_attn(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(qo_indptr), _ptr(o), _ptr(lse),
        _ptr(page_table), page_table.shape[1], _ptr(table_idx), _ptr(seq_lens), B, T, Hq,
        float(scale), int(max_seq_len_hint), int(max_total_keys_hint), _ptr(workspace), ws_bytes,
        _stream(stream)))


def pkv_paged_extend_attn_store(pool, layer: int, q, k_new, v_new, qo_indptr, o, lse,
                                page_table, seq_lens, scale: float, max_seq_len_hint: int,
                                workspace, table_idx=None, stream=None,
                                max_total_keys_hint: int = 0) -> None:
    """Extend step with store_kv fused: k_new, v_new [T, Hkv, D] bf16 (row t = query
    token t) go to the chunk's key positions of each row, then extend as
    pkv_paged_extend_attn."""
    ps = pool_struct(pool)
    _want(q, torch.bfloat16, "q", 3)
    _want(o, torch.bfloat16, "o", 3)
    _contig(q, "q")
    _contig(o, "o")
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _want(t, torch.bfloat16, name, 3)
    if k_new.stride(0) != v_new.stride(0) or k_new.stride(1) != k_new.shape[2] \
            or k_new.stride(2) != 1 or v_new.stride(1) != v_new.shape[2] or v_new.stride(2) != 1:
        raise ValueError("k_new and v_new rows must share a row stride with heads/dims contiguous")
    _want(qo_indptr, torch.int32, "qo_indptr", 1)
    _want(page_table, torch.int32, "page_table", 2)
    _contig(page_table, "page_table")
    _want(seq_lens, torch.int32, "seq_lens", 1)
    T, Hq, D = q.shape
    B = seq_lens.shape[0]
    if o.shape != q.shape or qo_indptr.shape[0] != B + 1:
        raise ValueError("o must match q and qo_indptr must have batch+1 entries")
    if k_new.shape[0] != T or v_new.shape[0] != T:
        raise ValueError("k_new and v_new must have total_q rows")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    if workspace is not None:
        _contig(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_extend_attn_store(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new), k_new.stride(0),
        _ptr(qo_indptr), _ptr(o), _ptr(lse), _ptr(page_table), page_table.shape[1],
        _ptr(table_idx), _ptr(seq_lens), B, T, Hq, float(scale), int(max_seq_len_hint),
        int(max_total_keys_hint), _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_cascade_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               num_groups: int, max_prefix_len_hint: int,
                               max_suffix_len_hint: int) -> int:
    return int(load().pkv_cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                 num_groups, max_prefix_len_hint,
                                                 max_suffix_len_hint))


def pkv_paged_cascade_decode_attn(pool, layer: int, q, o, lse, prefix_page_table, prefix_lens,
                                  member_indptr, members, page_table, seq_lens, scale: float,
                                  max_prefix_len_hint: int, max_suffix_len_hint: int, workspace,
                                  table_idx=None, stream=None) -> None:
    """Cascade decode: q, o [B, Hq, D] bf16; lse [B, Hq] fp32 or None; prefix_page_table
    [G, stride_p] and prefix_lens [G]; member_indptr [G+1] and members [B] partition the
    requests into groups; page_table rows and seq_lens [B] hold each request's suffix."""
    ps = pool_struct(pool)
    for t, name in ((q, "q"), (o, "o")):
        _want(t, torch.bfloat16, name, 3)
        _contig(t, name)
    for t, name, nd in ((prefix_page_table, "prefix_page_table", 2), (prefix_lens, "prefix_lens", 1),
                        (member_indptr, "member_indptr", 1), (members, "members", 1),
                        (page_table, "page_table", 2), (seq_lens, "seq_lens", 1)):
        _want(t, torch.int32, name, nd)
        _contig(t, name)
    B, Hq, D = q.shape
    G = prefix_lens.shape[0]
    if o.shape != q.shape or seq_lens.shape[0] != B or member_indptr.shape[0] != G + 1 \
            or prefix_page_table.shape[0] < G:
        raise ValueError("inconsistent cascade shapes")
    if lse is not None:
        _want(lse, torch.float32, "lse", 2)
        _contig(lse, "lse")
    if table_idx is not None:
        _want(table_idx, torch.int32, "table_idx", 1)
    if workspace is not None:
        _contig(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_cascade_decode_attn(
        ctypes.byref(ps), int(layer), _ptr(q), _ptr(o), _ptr(lse), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(prefix_lens), _ptr(member_indptr), _ptr(members), G,
        _ptr(page_table), page_table.shape[1], _ptr(table_idx), _ptr(seq_lens), B, Hq,
        float(scale), int(max_prefix_len_hint), int(max_suffix_len_hint), _ptr(workspace),
        ws_bytes, _stream(stream)))


def pkv_merge_lse(o_a, lse_a, o_b, lse_b, o_out, lse_out=None, stream=None) -> None:
    """Merge two states: o_* [rows, H, D] fp32, lse_* [rows, H] fp32; o_out bf16 or fp32."""
    for t, name in ((o_a, "o_a"), (o_b, "o_b")):
        _want(t, torch.float32, name, 3)
        _contig(t, name)
    for t, name in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _want(t, torch.float32, name, 2)
        _contig(t, name)
    if o_out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("o_out must be fp32 or bf16")
    _contig(o_out, "o_out")
    rows, H, D = o_a.shape
    if o_b.shape != o_a.shape or o_out.shape != o_a.shape or lse_a.shape != (rows, H) \
            or lse_b.shape != (rows, H):
        raise ValueError("shape mismatch")
    if lse_out is not None:
        _want(lse_out, torch.float32, "lse_out", 2)
    _check(load().pkv_merge_lse(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out),
                                1 if o_out.dtype == torch.bfloat16 else 0, _ptr(lse_out), rows,
                                H, D, _stream(stream)))


def pkv_read_device_errors() -> int:
    """Read and clear the device error word (synchronises the device)."""
    v = ctypes.c_uint32(0)
    _check(load().pkv_read_device_errors(ctypes.byref(v)))
    return int(v.value)
