"""Batches past one round of the extend planner's 256-wide scans (many
requests, many cascade groups) and wide decode grids, against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import (assert_every_row_written, check_against_oracle, compare, gpu_inputs,
                     lse_compare, nan_outputs, oracle_run)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_extend_600_requests():
    rng = np.random.default_rng(71)
    chunks = rng.integers(1, 40, size=600)
    prefix = rng.integers(0, 60, size=600)
    case = W.random_case(71, kind="extend", seq_lens=(prefix + chunks).tolist(),
                         chunk_lens=chunks.tolist(), Hq=8, Hkv=2, D=64, P=1)
    check_against_oracle(case)


@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.125])
def test_extend_many_items_per_sm_any_scale(scale):
    """About seven (kv head, block) work items per SM for the persistent
    attention kernel, with chunk lengths spanning one and two query tiles
    (items whose second query tile is empty, and items whose second tile sees
    one key tile more), under a negative, zero and positive scale (the sign
    folded into each item's Q)."""
    rng = np.random.default_rng(74)
    chunks = rng.integers(1, 121, size=420)
    prefix = rng.integers(0, 300, size=420)
    case = W.random_case(74, kind="extend", seq_lens=(prefix + chunks).tolist(),
                         chunk_lens=chunks.tolist(), Hq=8, Hkv=2, D=64, P=16, scale=scale)
    check_against_oracle(case)


def test_decode_3000_requests():
    rng = np.random.default_rng(72)
    case = W.random_case(72, seq_lens=rng.integers(1, 90, size=3000).tolist(), Hq=8, Hkv=2,
                         D=64, P=16)
    check_against_oracle(case)


def test_cascade_300_groups():
    import paged_kv_attention_out_gb300 as pkv
    rng = np.random.default_rng(73)
    sizes = rng.integers(1, 4, size=300).tolist()
    prefixes = rng.integers(0, 70, size=300).tolist()
    case = W.cascade_case(73, group_sizes=sizes, prefix_lens=prefixes, Hq=8, Hkv=2, D=64,
                          suffix_lo=1, suffix_hi=40)
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    ct = {n: torch.as_tensor(a, dtype=torch.int32, device="cuda")
          for n, a in W.cascade_tables(case).items()}
    G = ct["prefix_lens"].shape[0]
    pmax = max(int(ct["prefix_lens"].max()), 1)
    smax = int(ct["seq_lens"].max())
    ws = torch.empty(pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, G, pmax,
                                                    smax), dtype=torch.uint8, device="cuda")
    o, lse = nan_outputs(q)
    pkv.pkv_read_device_errors()
    pkv.pkv_paged_cascade_decode_attn(pool, case.layer, q, o, lse, ct["prefix_page_table"],
                                      ct["prefix_lens"], ct["member_indptr"], ct["members"],
                                      ct["page_table"], ct["seq_lens"], case.scale, pmax, smax,
                                      ws)
    assert pkv.pkv_read_device_errors() == 0
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case)
    compare(o.float().cpu().double().numpy(), want_o)
    lse_compare(lse.cpu().double().numpy(), want_lse)
