"""Paged decode attention on the GPU against the fp64 oracle.

Tolerance on bf16 outputs: max|err| <= 2e-2 and mean|err| <= 2e-3; lse
(fp32) within 2e-3. Small cases run the whole oracle; the full-size named
workloads are checked on sampled requests, cut out into compact cases
whose pages are renumbered (the oracle's relocation pin makes that exact).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import (check_against_oracle, compare, gpu_attention, gpu_inputs, gpu_run,
                     lse_compare, oracle_run)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_tiny_decode_workload():
    check_against_oracle(W.tiny_decode(0))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("P", [1, 16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (8, 2), (32, 8), (32, 4), (8, 8), (16, 2)])
def test_decode_sweep(D, P, Hq, Hkv):
    seq = [1, 15, 16, 17, 33, 127, 128, 129, 700, 2049]
    case = W.random_case(41 + Hq + P + D, seq_lens=seq, Hq=Hq, Hkv=Hkv, D=D, P=P)
    check_against_oracle(case)


@pytest.mark.parametrize("hint", [1, 0, 100, 5000])
def test_decode_hint_changes_only_parallelism(hint):
    """A bound below the real seq_len (or none) is still computed correctly."""
    case = W.random_case(7, seq_lens=[2000, 37, 900, 1], Hq=16, Hkv=4, D=128, P=16)
    check_against_oracle(case, hint=hint)


def test_split_boundaries_exact_multiples():
    # keys exactly at, just below and just above multiples of the split size
    import paged_kv_attention_out_gb300 as pkv
    from paged_kv_attention_out_gb300 import build
    seq = [128 * k + e for k in (1, 2, 7) for e in (-1, 0, 1)]
    case = W.random_case(8, seq_lens=seq, Hq=8, Hkv=2, D=128, P=1)
    check_against_oracle(case, hint=1024)


def test_table_idx_indirection_and_poison():
    case = W.random_case(9, seq_lens=[300, 5, 1024, 77], Hq=8, Hkv=2, D=128, P=16,
                         use_table_idx=True)
    check_against_oracle(case)


def test_shared_prefix_rows():
    case = W.random_case(10, seq_lens=[600, 650, 700, 580, 611, 900], Hq=32, Hkv=8, D=128,
                         P=16, shared_prefix=512, group_size=3)
    check_against_oracle(case)


def test_empty_sequence_gives_zero_and_neg_inf():
    case = W.random_case(11, seq_lens=[50, 3], Hq=4, Hkv=2, D=64, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    import paged_kv_attention_out_gb300 as pkv
    pkv.pkv_kv_store(pool, 0, k, v, t["out_loc"])
    t["seq_lens"][0] = 0
    o, lse = gpu_attention(case, pool, q, t)
    torch.cuda.synchronize()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.isfinite(lse[1]).all()


def test_relocating_pages_gives_identical_bits():
    """The kernel's reduction order depends on logical key positions only."""
    case = W.random_case(12, seq_lens=[3000, 100, 1500], Hq=32, Hkv=8, D=128, P=16)
    o1, l1, pool = gpu_run(case)
    perm = torch.randperm(case.NP, generator=torch.Generator().manual_seed(0))
    pool2 = torch.empty_like(pool)
    pool2[:, :, perm.cuda()] = pool
    t = case.device_tables("cuda")
    t["page_table"] = perm.cuda()[t["page_table"].long()].to(torch.int32)
    o2, l2 = gpu_attention(case, pool2, case.q("cuda"), t)
    torch.cuda.synchronize()
    assert np.array_equal(o1, o2.float().cpu().double().numpy())
    assert np.array_equal(l1, l2.cpu().double().numpy())


def test_lse_is_optional():
    case = W.random_case(13, seq_lens=[900, 20], Hq=8, Hkv=2, D=128, P=1)
    pool, k, v, q, t = gpu_inputs(case)
    import paged_kv_attention_out_gb300 as pkv
    pkv.pkv_kv_store(pool, 0, k, v, t["out_loc"])
    o, _ = gpu_attention(case, pool, q, t, with_lse=False)
    want, _, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy(), want)


def _sampled_full_size(case, requests):
    """Runs the full case on the GPU; checks `requests` against the oracle."""
    o, lse, pool = gpu_run(case, poison=True)
    del pool
    torch.cuda.empty_cache()
    sub = case.compact(requests)
    want_o, want_lse, _ = oracle_run(sub)
    compare(o[requests], want_o)
    lse_compare(lse[requests], want_lse)
    assert np.isfinite(o).all()


def test_llama8b_decode_full_size_sampled():
    case = W.llama8b_decode(0)
    rng = np.random.default_rng(0)
    req = sorted({int(np.argmax(case.seq_lens)), int(np.argmin(case.seq_lens)),
                  *rng.choice(case.B, 4, replace=False).tolist()})
    _sampled_full_size(case, req)


@pytest.mark.parametrize("shuffled", [False, True])
def test_radix_shared_decode_full_size_sampled(shuffled):
    case = W.radix_shared_decode(0, shuffled=shuffled)
    groups = np.array(case.notes["group_of_request"])
    same = np.flatnonzero(groups == groups[0])[:3].tolist()
    other = np.flatnonzero(groups != groups[0])[:2].tolist()
    _sampled_full_size(case, sorted(same + other))


def test_long_context_decode_full_size_sampled():
    case = W.long_context_decode(0)
    req = sorted({int(np.argmax(case.seq_lens)), int(np.argmin(case.seq_lens))})
    _sampled_full_size(case, req)
