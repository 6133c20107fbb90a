"""The C ABI: the library loads, exports every entry point include/pkv.h
declares, and rejects bad host-side arguments before touching the GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from paged_kv_attention_out_gb300 import binding
    return binding.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_extend_attn",
                 "pkv_merge_lse", "pkv_decode_workspace_size", "pkv_extend_workspace_size",
                 "pkv_status_string",
                 "pkv_last_error", "pkv_init", "pkv_read_device_errors"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in pkv.h but not exported: {missing}"


def test_python_binding_has_the_same_names(lib):
    import paged_kv_attention_out_gb300 as pkv
    for n in ("pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_extend_attn",
              "pkv_merge_lse", "pkv_decode_workspace_size", "pkv_extend_workspace_size",
              "pkv_init",
              "pkv_read_device_errors"):
        assert callable(getattr(pkv, n))


def test_status_strings(lib):
    f = lib.pkv_status_string
    assert [f(i).decode() for i in range(5)] == [
        "PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED",
        "PKV_ERR_WORKSPACE_TOO_SMALL", "PKV_ERR_CUDA"]


def test_bad_host_arguments_are_rejected_before_any_gpu_work(lib):
    from paged_kv_attention_out_gb300.binding import PkvPool
    # NULL pool
    assert lib.pkv_kv_store(None, 0, None, None, 0, None, 1, None) == 1
    assert b"pool" in lib.pkv_last_error()
    # head_dim 96 is unsupported, layer out of range is invalid
    pool = PkvPool(16, 2, 10, 1, 2, 96)
    assert lib.pkv_kv_store(ctypes.byref(pool), 0, 16, 16, 192, 16, 1, None) == 2
    pool = PkvPool(16, 2, 10, 1, 2, 128)
    assert lib.pkv_kv_store(ctypes.byref(pool), 2, 16, 16, 256, 16, 1, None) == 1
    # misaligned pool base
    pool = PkvPool(18, 2, 10, 1, 2, 128)
    assert lib.pkv_kv_store(ctypes.byref(pool), 0, 16, 16, 256, 16, 1, None) == 1
    # row stride below Hkv * D
    pool = PkvPool(16, 2, 10, 1, 2, 128)
    assert lib.pkv_kv_store(ctypes.byref(pool), 0, 16, 16, 128, 16, 1, None) == 1
    # decode: q heads not a multiple of kv heads; group above 8
    assert lib.pkv_paged_decode_attn(ctypes.byref(pool), 0, 16, 16, None, 16, 4, None, 16,
                                     1, 3, ctypes.c_float(1.0), 4, None, 0, None) == 1
    assert lib.pkv_paged_decode_attn(ctypes.byref(pool), 0, 16, 16, None, 16, 4, None, 16,
                                     1, 32, ctypes.c_float(1.0), 4, None, 0, None) == 2
    # merge: head_dim not a multiple of 4
    assert lib.pkv_merge_lse(16, 16, 16, 16, 16, 0, None, 1, 1, 6, None) == 1
    # empty work is a no-op success
    assert lib.pkv_merge_lse(None, None, None, None, None, 0, None, 0, 1, 4, None) == 0
    assert lib.pkv_kv_store(ctypes.byref(pool), 0, None, None, 256, None, 0, None) == 0
    # the workspace query refuses nonsense instead of guessing
    assert lib.pkv_decode_workspace_size(0, 32, 8, 128, 4096) == 0
    assert lib.pkv_decode_workspace_size(4, 30, 8, 128, 4096) == 0
    assert lib.pkv_extend_workspace_size(0, 8, 128, 4096, 0) == 0
    assert lib.pkv_cascade_workspace_size(4, 32, 8, 128, 0, 2048, 512) == 0
    assert lib.pkv_cascade_workspace_size(4, 30, 8, 128, 2, 2048, 512) == 0
    # fused store + decode: NULL or misaligned new rows, row stride below Hkv * D
    f = ctypes.c_float(1.0)
    assert lib.pkv_paged_decode_attn_store(ctypes.byref(pool), 0, 16, None, 16, 256, 16, None,
                                           16, 4, None, 16, 1, 4, f, 4, None, 0, None) == 1
    assert lib.pkv_paged_decode_attn_store(ctypes.byref(pool), 0, 16, 18, 16, 256, 16, None,
                                           16, 4, None, 16, 1, 4, f, 4, None, 0, None) == 1
    assert lib.pkv_paged_decode_attn_store(ctypes.byref(pool), 0, 16, 16, 16, 128, 16, None,
                                           16, 4, None, 16, 1, 4, f, 4, None, 0, None) == 1
    # fused store + extend: the same refusals
    assert lib.pkv_paged_extend_attn_store(ctypes.byref(pool), 0, 16, None, 16, 256, 16, 16,
                                           None, 16, 4, None, 16, 1, 8, 4, f, 8, 0, None, 0,
                                           None) == 1
    assert lib.pkv_paged_extend_attn_store(ctypes.byref(pool), 0, 16, 16, 34, 256, 16, 16,
                                           None, 16, 4, None, 16, 1, 8, 4, f, 8, 0, None, 0,
                                           None) == 1
    assert lib.pkv_paged_extend_attn_store(ctypes.byref(pool), 0, 16, 16, 16, 100, 16, 16,
                                           None, 16, 4, None, 16, 1, 8, 4, f, 8, 0, None, 0,
                                           None) == 1
    # cascade: group above 8; every request must be in a group; NULL member lists
    assert lib.pkv_paged_cascade_decode_attn(
        ctypes.byref(pool), 0, 16, 16, None, 16, 4, 16, 16, 16, 1, 16, 4, None, 16, 1, 32, f,
        64, 64, None, 0, None) == 2
    assert lib.pkv_paged_cascade_decode_attn(
        ctypes.byref(pool), 0, 16, 16, None, 16, 4, 16, 16, 16, 0, 16, 4, None, 16, 1, 4, f,
        64, 64, None, 0, None) == 1
    assert lib.pkv_paged_cascade_decode_attn(
        ctypes.byref(pool), 0, 16, 16, None, 16, 4, 16, None, None, 1, 16, 4, None, 16, 1, 4, f,
        64, 64, None, 0, None) == 1


def test_extend_workspace_follows_the_keys_present():
    """The extend workspace holds each request's keys rounded up to 128, back
    to back, so it is sized by a bound on their sum: 64 requests, one of 128k
    keys and 63 of at most 512, at 8 kv heads and head_dim 128, need under
    1 GB (batch x the longest would be 34 GB)."""
    from paged_kv_attention_out_gb300 import binding
    lib = binding.load()
    total = 131072 + 63 * 512
    keyed = lib.pkv_extend_workspace_size(64, 8, 128, 131072, total)
    longest = lib.pkv_extend_workspace_size(64, 8, 128, 131072, 0)
    kv = 2 * 8 * 128 * 2  # K and V bytes of one key, all kv heads
    assert total * kv <= keyed < (1 << 30)
    assert longest >= 64 * 131072 * kv > 30 * (1 << 30)
    # the bound covers the 127 rows of rounding per request
    assert keyed >= (total + 64 * 127) * kv


@pytest.mark.gpu
def test_gpu_argument_errors_raise():
    ensure_built()
    import paged_kv_attention_out_gb300 as pkv
    from paged_kv_attention_out_gb300 import workloads as W
    pkv.pkv_init()
    case = W.random_case(1, seq_lens=[300, 900], Hq=8, Hkv=2, D=128, P=1)
    pool = case.make_pool("cuda")
    q = case.q("cuda")
    o = torch.empty_like(q)
    t = case.device_tables("cuda")
    need = pkv.pkv_decode_workspace_size(2, 8, 2, 128, 900)
    assert need > 0
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_decode_attn(pool, 0, q, o, None, t["page_table"], t["seq_lens"],
                                  case.scale, 900, small)
    assert ei.value.status == 3
    with pytest.raises(pkv.PkvError):
        pkv.pkv_paged_decode_attn(pool, 0, q, o, None, t["page_table"], t["seq_lens"],
                                  float("nan"), 900, None)
    assert pkv.pkv_read_device_errors() == 0
