"""Decode with store_kv fused in (pkv_paged_decode_attn_store): the new key and
value rows land at key seq_len - 1 of each row and are attended in the same
launch; results equal store_kv + decode ("Code Notes: mini-sglang", Engine
Layer table, BaseKVCachePool and GraphRunner rows)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import (assert_every_row_written, compare, gpu_inputs, lse_compare, nan_outputs,
                     oracle_run, to_bits)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def fused_run(case, poison=True, hint=None, with_lse=True):
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case, poison)
    h = case.max_seq_len if hint is None else hint
    ws = torch.empty(max(pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, h), 256),
                     dtype=torch.uint8, device="cuda")
    o, lse = nan_outputs(q, with_lse)
    pkv.pkv_paged_decode_attn_store(pool, case.layer, q, k, v, o, lse, t["page_table"],
                                    t["seq_lens"], case.scale, h, ws, table_idx=t.get("table_idx"))
    torch.cuda.synchronize()
    return o, lse, pool


@pytest.mark.parametrize("kw", [
    dict(seq_lens=[1, 7, 16, 33], Hq=4, Hkv=2, D=64, P=1),
    dict(seq_lens=[300, 5, 1024, 77], Hq=8, Hkv=2, D=128, P=16, use_table_idx=True),
    dict(seq_lens=[4000, 17, 2500, 129, 1], Hq=32, Hkv=8, D=128, P=1),
    dict(seq_lens=[700, 64, 1500], Hq=8, Hkv=1, D=128, P=16),
])
def test_fused_store_decode_matches_oracle_and_pool_bits(kw):
    case = W.random_case(21, **kw)
    o, lse, pool = fused_run(case)
    assert_every_row_written(o, lse)
    want_o, want_lse, want_pool = oracle_run(case)
    compare(o.float().cpu().double().numpy(), want_o)
    lse_compare(lse.cpu().double().numpy(), want_lse)
    got_pool = to_bits(pool).reshape(case.pool_shape)
    assert np.array_equal(got_pool, want_pool), "pool bits differ from store_kv"


def test_fused_equals_separate_store_then_decode_bitwise():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(22, seq_lens=[900, 33, 2049, 400, 12, 1500], Hq=32, Hkv=8, D=128, P=16)
    o1, l1, p1 = fused_run(case)
    pool, k, v, q, t = gpu_inputs(case, True)
    h = case.max_seq_len
    ws = torch.empty(max(pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, h), 256),
                     dtype=torch.uint8, device="cuda")
    o2, l2 = nan_outputs(q)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    pkv.pkv_paged_decode_attn(pool, case.layer, q, o2, l2, t["page_table"], t["seq_lens"],
                              case.scale, h, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(p1.view(torch.int16), pool.view(torch.int16))


def test_llama8b_fused_full_size_every_request():
    case = W.llama8b_decode(0)
    o, lse, pool = fused_run(case)
    del pool
    torch.cuda.empty_cache()
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case.compact(list(range(case.B))))
    compare(o.float().cpu().double().numpy(), want_o)
    lse_compare(lse.cpu().double().numpy(), want_lse)
