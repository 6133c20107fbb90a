"""Device-side argument checks of the attention calls: values in device
memory that would index outside the pool, the tables or the workspace are
skipped on the device (never dereferenced) and reported in the device error
word (pkv_read_device_errors); requests not involved are computed as usual."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import compare, gpu_inputs, oracle_run
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PAGE, SEQ, INDPTR, TABLE_IDX = 0x2, 0x4, 0x8, 0x10


def _errors():
    import paged_kv_attention_out_gb300 as pkv
    torch.cuda.synchronize()
    return pkv.pkv_read_device_errors()


def _decode(case, pool, q, t, fused=None):
    import paged_kv_attention_out_gb300 as pkv
    h = case.max_seq_len
    ws = torch.empty(max(pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, h), 256),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    if fused is None:
        pkv.pkv_paged_decode_attn(pool, case.layer, q, o, None, t["page_table"], t["seq_lens"],
                                  case.scale, h, ws)
    else:
        k, v = fused
        pkv.pkv_paged_decode_attn_store(pool, case.layer, q, k, v, o, None, t["page_table"],
                                        t["seq_lens"], case.scale, h, ws)
    return o


@pytest.mark.parametrize("fused", [False, True])
def test_decode_page_id_out_of_range_is_flagged(fused):
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(31, seq_lens=[200, 90, 300], Hq=8, Hkv=2, D=128, P=16)
    pool, k, v, q, t = gpu_inputs(case)
    if not fused:
        pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    pt = t["page_table"].clone()
    pt[1, 2] = case.NP + 1000  # a page id past the pool in request 1's row
    pt[1, (90 - 1) // 16] = -7  # and its newest key's page (the fused store's target)
    _errors()
    o = _decode(case, pool, q, dict(t, page_table=pt), fused=(k, v) if fused else None)
    assert _errors() & PAGE
    want, _, _ = oracle_run(case)
    got = o.float().cpu().double().numpy()
    ok = [0, 2]
    compare(got[ok], want[ok])


def test_decode_seq_len_past_the_row_is_flagged():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(32, seq_lens=[64, 100, 33], Hq=4, Hkv=2, D=64, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    sl = t["seq_lens"].clone()
    sl[0] = case.page_table.shape[1] * case.P + 5
    _errors()
    o = _decode(case, pool, q, dict(t, seq_lens=sl))
    assert _errors() & SEQ
    want, _, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy()[1:], want[1:])


def test_extend_requests_past_the_key_bound_are_flagged_and_skipped():
    """Runs are laid out in request order, each seq_len rounded up to 128; with
    a bound of 300 keys the workspace holds 384 + 3 x 128 rows, so request 0
    (128 rows) fits and requests 1 (768) and 2 (128, starting past the end)
    do not: they are flagged and not computed, request 0 is."""
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(33, kind="extend", seq_lens=[100, 700, 60], chunk_lens=[40, 100, 60],
                         Hq=8, Hkv=2, D=128, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    hint, total = 700, 300
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, hint, total),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    _errors()
    pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, None, t["page_table"],
                              t["seq_lens"], case.scale, hint, ws, max_total_keys_hint=total)
    assert _errors() & SEQ
    want, _, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy()[0:40], want[0:40])


def test_extend_request_longer_than_the_length_hint_is_still_computed():
    """max_seq_len_hint only sizes the schedule's cost buckets: a longer request
    is computed (sorted as if it had the hint's length)."""
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(36, kind="extend", seq_lens=[100, 700, 60], chunk_lens=[40, 100, 60],
                         Hq=8, Hkv=2, D=128, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    hint = 200  # request 1 has 700 keys; no sum given: 3 x 256 rows of keys
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, hint, 0),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    _errors()
    pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, None, t["page_table"],
                              t["seq_lens"], case.scale, hint, ws)
    assert _errors() == 0
    want, _, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy(), want)


def test_extend_negative_table_idx_is_flagged():
    """A negative table_idx entry of a request other than the first (whose
    keys start in a later gather CTA) is reported; the other requests are
    computed as usual."""
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(37, kind="extend", seq_lens=[100, 300, 200, 50],
                         chunk_lens=[30, 64, 40, 50], Hq=8, Hkv=2, D=128, P=16,
                         use_table_idx=True)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    ti = t["table_idx"].clone()
    ti[2] = -3
    h = case.max_seq_len
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    _errors()
    pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, None, t["page_table"],
                              t["seq_lens"], case.scale, h, ws, table_idx=ti)
    assert _errors() & TABLE_IDX
    want, _, _ = oracle_run(case)
    got = o.float().cpu().double().numpy()
    qo = case.qo_indptr
    ok = np.r_[qo[0]:qo[2], qo[3]:qo[4]]  # requests 0, 1 and 3
    compare(got[ok], want[ok])


def test_extend_malformed_qo_indptr_is_flagged():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(34, kind="extend", seq_lens=[100, 120, 60], chunk_lens=[40, 50, 60],
                         Hq=8, Hkv=2, D=64, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    qo = t["qo_indptr"].clone()
    qo[2] = 10  # decreasing: request 1 would have a negative chunk
    h = case.max_seq_len
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h),
                     dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    _errors()
    pkv.pkv_paged_extend_attn(pool, case.layer, q, qo, o, None, t["page_table"], t["seq_lens"],
                              case.scale, h, ws)
    assert _errors() & INDPTR
    want, _, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy()[:40], want[:40])  # request 0 still computed


def test_cascade_member_out_of_range_is_flagged():
    import paged_kv_attention_out_gb300 as pkv
    case = W.cascade_case(35, group_sizes=[6, 3], prefix_lens=[64, 32], Hq=8, Hkv=2, D=64)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    ct = {n: torch.as_tensor(a, dtype=torch.int32, device="cuda")
          for n, a in W.cascade_tables(case).items()}
    members = ct["members"].clone()
    bad = int(members[0])
    members[0] = case.B + 50
    pmax, smax = 64, int(ct["seq_lens"].max())
    ws = torch.empty(pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, 2, pmax,
                                                    smax), dtype=torch.uint8, device="cuda")
    o = torch.full_like(q, float("nan"))
    _errors()
    pkv.pkv_paged_cascade_decode_attn(pool, case.layer, q, o, None, ct["prefix_page_table"],
                                      ct["prefix_lens"], ct["member_indptr"], members,
                                      ct["page_table"], ct["seq_lens"], case.scale, pmax, smax,
                                      ws)
    assert _errors() & INDPTR
    want, _, _ = oracle_run(case)
    ok = [b for b in range(case.B) if b != bad]
    compare(o.float().cpu().double().numpy()[ok], want[ok])
