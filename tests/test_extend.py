"""Paged extend (chunked-prefill) attention on the GPU against the oracle.

Small cases run the whole oracle. The full-size chunked-prefill workload
(outputs NaN-filled before the call) must write every row, and two whole
requests, the one with the longest cached prefix and the one with the
longest chunk, are compared query by query and head by head against the
oracle on a compact cut of each request; the others on sampled queries
(query j of request r equals a decode over the first p_r + j + 1 keys of
its row, a pin of the oracle).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import (assert_every_row_written, check_against_oracle, compare, gpu_run,
                     lse_compare, oracle_inputs, oracle_run)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("P", [1, 16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (32, 8), (16, 2), (32, 2)])
def test_extend_sweep(D, P, Hq, Hkv):
    seq = [1, 17, 80, 300, 129, 64]
    chunks = [1, 17, 65, 100, 1, 64]  # prefix 0, 0, 15, 200, 128, 0
    case = W.random_case(51 + Hq + D + P, kind="extend", seq_lens=seq, chunk_lens=chunks,
                         Hq=Hq, Hkv=Hkv, D=D, P=P)
    check_against_oracle(case)


def test_extend_with_empty_chunk_and_table_idx():
    case = W.random_case(52, kind="extend", seq_lens=[40, 9, 260, 33],
                         chunk_lens=[12, 0, 190, 33], Hq=8, Hkv=2, D=128, P=16,
                         use_table_idx=True)
    check_against_oracle(case)


def test_extend_group_that_does_not_divide_the_tile():
    case = W.random_case(53, kind="extend", seq_lens=[90, 200], chunk_lens=[70, 31],
                         Hq=12, Hkv=2, D=128, P=1)
    check_against_oracle(case)


def test_extend_shared_prefix():
    case = W.random_case(54, kind="extend", seq_lens=[700, 650, 600], chunk_lens=[100, 90, 80],
                         Hq=32, Hkv=8, D=128, P=16, shared_prefix=480, group_size=3)
    check_against_oracle(case)


def test_mixed_prefill_and_decode_batch():
    """One extend call over a batch mixing prefill chunks with decode requests
    (chunk of one token after a long cached prefix): a decode row of an extend
    call is the decode of that request."""
    case = W.random_case(55, kind="extend", seq_lens=[513, 1, 2000, 37, 900, 4096, 2, 130],
                         chunk_lens=[1, 1, 300, 1, 128, 1, 2, 129], Hq=32, Hkv=8, D=128, P=16)
    check_against_oracle(case)


# The softmax scale is any finite number: negative (the largest scaled score
# comes from the smallest raw score), zero (every visible key weighs the
# same: o = mean(V), lse = log n) and large (scores spread over hundreds of
# log2 units, so the lazy rescale of O runs on most tiles).
@pytest.mark.parametrize("scale", [-0.0884, -1.0, 0.0, 1.0, 3.0])
@pytest.mark.parametrize("D", [64, 128])
def test_extend_any_finite_scale(scale, D):
    case = W.random_case(56, kind="extend", seq_lens=[300, 129, 700, 64],
                         chunk_lens=[170, 129, 256, 1], Hq=8, Hkv=2, D=D, P=16,
                         scale=scale)
    check_against_oracle(case)


def test_workspace_sized_by_keys_present():
    """64 requests, one with a 131,008-key cached prefix and a 64-token chunk,
    63 with short prefixes and chunks: the workspace from the sum of the
    seq_lens stays under 1 GB (159 MB; batch x the longest would be 8.6 GB
    here) and every query matches the oracle."""
    import paged_kv_attention_out_gb300 as pkv
    rng = np.random.default_rng(57)
    chunks = [64] + rng.integers(1, 65, size=63).tolist()
    seq = [131072] + (np.array(chunks[1:]) + rng.integers(0, 449, size=63)).tolist()
    case = W.random_case(57, kind="extend", seq_lens=seq, chunk_lens=chunks, Hq=8, Hkv=2, D=128,
                         P=16)
    total = int(case.seq_lens.sum())
    need = pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, case.max_seq_len, total)
    assert 0 < need < (1 << 30)
    assert pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, case.max_seq_len, 0) > 4 << 30
    o, lse, _ = gpu_run(case)
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case)
    compare(o, want_o)
    lse_compare(lse, want_lse)


def test_chunked_prefill_full_size():
    case = W.chunked_prefill_extend(0)
    o, lse, _ = gpu_run(case)
    torch.cuda.empty_cache()
    assert_every_row_written(o, lse)
    chunks = np.diff(case.qo_indptr)
    prefixes = case.seq_lens - chunks
    whole = sorted({int(np.argmax(prefixes)), int(np.argmax(chunks))})
    for r in whole:  # every chunk token, every head: every block and diagonal tile
        s, e = int(case.qo_indptr[r]), int(case.qo_indptr[r + 1])
        want_o, want_lse, _ = oracle_run(case.compact([r]))
        compare(o[s:e], want_o)
        lse_compare(lse[s:e], want_lse)
    rng = np.random.default_rng(0)
    q_all = W.bf16_bits(case.q())
    for r in sorted(set(range(case.B)) - set(whole)):
        sub = case.compact([r])
        pool, k, v, _ = oracle_inputs(sub)
        oracle.kv_store(pool, 0, k, v, sub.out_loc)
        c = int(case.qo_indptr[r + 1] - case.qo_indptr[r])
        p = int(case.seq_lens[r]) - c
        js = sorted({0, c - 1, *rng.integers(0, c, 3).tolist()})
        for j in js:
            t = int(case.qo_indptr[r]) + j
            want_o, want_l = oracle.decode_attn(pool, 0, q_all[t:t + 1], sub.page_table,
                                                np.array([p + j + 1], np.int32), case.scale)
            compare(o[t:t + 1], want_o)
            lse_compare(lse[t:t + 1], want_l)
