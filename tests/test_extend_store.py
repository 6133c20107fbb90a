"""Extend with store_kv fused in (pkv_paged_extend_attn_store): the chunk's new
key and value rows land at the chunk's key positions of each row and are
attended in the same call; results equal store_kv + extend ("Code Notes:
mini-sglang", Engine Layer table, BaseKVCachePool row; Scheduler Layer table,
PrefillManager row)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import (assert_every_row_written, compare, gpu_inputs, lse_compare, nan_outputs,
                     oracle_inputs, oracle_run, to_bits)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def fused_run(case, poison=True):
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case, poison)
    h, total = case.max_seq_len, int(case.seq_lens.sum())
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h, total),
                     dtype=torch.uint8, device="cuda")
    o, lse = nan_outputs(q)
    pkv.pkv_paged_extend_attn_store(pool, case.layer, q, k, v, t["qo_indptr"], o, lse,
                                    t["page_table"], t["seq_lens"], case.scale, h, ws,
                                    table_idx=t.get("table_idx"), max_total_keys_hint=total)
    torch.cuda.synchronize()
    return o, lse, pool


def separate_run(case, poison=True):
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case, poison)
    h, total = case.max_seq_len, int(case.seq_lens.sum())
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h, total),
                     dtype=torch.uint8, device="cuda")
    o, lse = nan_outputs(q)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, lse, t["page_table"],
                              t["seq_lens"], case.scale, h, ws, table_idx=t.get("table_idx"),
                              max_total_keys_hint=total)
    torch.cuda.synchronize()
    return o, lse, pool


@pytest.mark.parametrize("kw", [
    dict(seq_lens=[1, 17, 80, 300, 129, 64], chunk_lens=[1, 17, 65, 100, 1, 64],
         Hq=4, Hkv=2, D=64, P=1),
    dict(seq_lens=[40, 9, 260, 33], chunk_lens=[12, 0, 190, 33], Hq=8, Hkv=2, D=128, P=16,
         use_table_idx=True),
    dict(seq_lens=[90, 200], chunk_lens=[70, 31], Hq=12, Hkv=2, D=128, P=1),
    dict(seq_lens=[700, 650, 600], chunk_lens=[100, 90, 80], Hq=32, Hkv=8, D=128, P=16,
         shared_prefix=480, group_size=3),
])
def test_fused_store_extend_matches_oracle_and_pool_bits(kw):
    case = W.random_case(61, kind="extend", **kw)
    o, lse, pool = fused_run(case)
    assert_every_row_written(o, lse)
    want_o, want_lse, want_pool = oracle_run(case)
    compare(o.float().cpu().double().numpy(), want_o)
    lse_compare(lse.cpu().double().numpy(), want_lse)
    got_pool = to_bits(pool).reshape(case.pool_shape)
    assert np.array_equal(got_pool, want_pool), "pool bits differ from store_kv"


def test_fused_equals_separate_store_then_extend_bitwise():
    case = W.random_case(62, kind="extend", seq_lens=[900, 33, 2049, 400, 12, 1500],
                         chunk_lens=[300, 33, 49, 400, 1, 256], Hq=32, Hkv=8, D=128, P=16)
    o1, l1, p1 = fused_run(case)
    o2, l2, p2 = separate_run(case)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(p1.view(torch.int16), p2.view(torch.int16))


def test_chunked_prefill_fused_full_size():
    """The 8-request, 8192-token chunked-prefill workload: bitwise equal to the
    separate calls (o, lse and the whole pool), and sampled rows against the
    oracle."""
    case = W.chunked_prefill_extend(0)
    o1, l1, p1 = fused_run(case)
    o2, l2, p2 = separate_run(case)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(p1.view(torch.int16), p2.view(torch.int16))
    assert_every_row_written(o1, l1)
    del p1, p2
    torch.cuda.empty_cache()
    o = o1.float().cpu().double().numpy()
    lse = l1.cpu().double().numpy()
    q_all = W.bf16_bits(case.q())
    rng = np.random.default_rng(2)
    for r in (0, case.B - 1):
        sub = case.compact([r])
        pool, k, v, _ = oracle_inputs(sub)
        oracle.kv_store(pool, 0, k, v, sub.out_loc)
        c = int(case.qo_indptr[r + 1] - case.qo_indptr[r])
        p = int(case.seq_lens[r]) - c
        for j in sorted({0, c - 1, *rng.integers(0, c, 2).tolist()}):
            t = int(case.qo_indptr[r]) + j
            want_o, want_l = oracle.decode_attn(pool, 0, q_all[t:t + 1], sub.page_table,
                                                np.array([p + j + 1], np.int32), case.scale)
            compare(o[t:t + 1], want_o)
            lse_compare(lse[t:t + 1], want_l)


def test_fused_bad_chunk_page_is_flagged_and_not_stored():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(63, kind="extend", seq_lens=[100, 60], chunk_lens=[40, 60],
                         Hq=8, Hkv=2, D=64, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    before = pool.clone()
    pt = t["page_table"].clone()
    pt[0, 70] = -3  # chunk key 70 of request 0 (chunk keys 60 .. 99)
    h, total = case.max_seq_len, int(case.seq_lens.sum())
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h, total),
                     dtype=torch.uint8, device="cuda")
    o, _ = nan_outputs(q, with_lse=False)
    pkv.pkv_read_device_errors()
    pkv.pkv_paged_extend_attn_store(pool, case.layer, q, k, v, t["qo_indptr"], o, None, pt,
                                    t["seq_lens"], case.scale, h, ws, max_total_keys_hint=total)
    assert pkv.pkv_read_device_errors() & 0x2
    want_o, _, want_pool = oracle_run(case)
    compare(o.float().cpu().double().numpy()[40:], want_o[40:])  # request 1 untouched
    got = to_bits(pool).reshape(case.pool_shape)
    old = to_bits(before).reshape(case.pool_shape)
    skipped = int(case.token_slots[0][70])
    assert np.array_equal(got[:, :, skipped], old[:, :, skipped]), "a bad slot was written"
    keep = np.ones(got.shape[2], bool)
    keep[skipped] = False
    assert np.array_equal(got[:, :, keep], want_pool[:, :, keep])
