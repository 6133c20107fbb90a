"""Cascade decode over shared prefixes (pkv_paged_cascade_decode_attn) against
the fp64 oracle evaluated on each request's full key list (prefix + suffix).

Grouped requests share their first keys, as a radix cache hit gives
("Introduction", Key Features, Radix Cache); the call attends each group's
prefix once for all members and merges it with every member's suffix.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import (assert_every_row_written, compare, gpu_inputs, lse_compare, nan_outputs,
                     oracle_run)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def cascade_run(case: W.Case, poison: bool = True, repeat: int = 1):
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case, poison)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    ct = {name: torch.as_tensor(a, dtype=torch.int32, device="cuda")
          for name, a in W.cascade_tables(case).items()}
    G = ct["prefix_lens"].shape[0]
    pmax = max(int(ct["prefix_lens"].max()), 1)
    smax = int(ct["seq_lens"].max())
    n = pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, G, pmax, smax)
    ws = torch.full((n,), 0x7F, dtype=torch.uint8, device="cuda")  # stale contents
    outs = []
    for _ in range(repeat):
        o, lse = nan_outputs(q)
        pkv.pkv_paged_cascade_decode_attn(
            pool, case.layer, q, o, lse, ct["prefix_page_table"], ct["prefix_lens"],
            ct["member_indptr"], ct["members"], ct["page_table"], ct["seq_lens"], case.scale,
            pmax, smax, ws)
        torch.cuda.synchronize()
        outs.append((o.float().cpu().double().numpy(), lse.cpu().double().numpy()))
    return outs


@pytest.mark.parametrize("P,Hq,Hkv,D,sizes,prefixes", [
    (1, 8, 2, 64, [5, 70, 1, 3], [40, 129, 0, 7]),     # several blocks in a group, empty prefix
    (16, 8, 2, 128, [3, 33, 2], [32, 256, 0]),          # whole-page prefixes
    (1, 8, 1, 128, [9, 1], [300, 5]),                   # 8 q heads per kv head
    (1, 4, 4, 64, [200, 2], [130, 0]),                  # one q head per kv head
    (1, 32, 8, 128, [40, 24], [2048, 513]),             # Llama-shaped heads
])
def test_cascade_matches_oracle(P, Hq, Hkv, D, sizes, prefixes):
    case = W.cascade_case(7, group_sizes=sizes, prefix_lens=prefixes, P=P, Hq=Hq, Hkv=Hkv,
                          D=D, suffix_lo=1, suffix_hi=150)
    (o, lse), = cascade_run(case)
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case)
    compare(o, want_o)
    lse_compare(lse, want_lse)


@pytest.mark.parametrize("scale", [-0.0884, -1.0, 0.0, 2.0])
def test_cascade_any_finite_scale(scale):
    """The shared-prefix attention runs on the extend kernel (non-causal, its
    last prefix tile masked): any finite scale, as for decode."""
    case = W.cascade_case(9, group_sizes=[40, 3], prefix_lens=[300, 129], P=1, Hq=32, Hkv=8,
                          D=128, suffix_lo=1, suffix_hi=200, scale=scale)
    (o, lse), = cascade_run(case)
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case)
    compare(o, want_o)
    lse_compare(lse, want_lse)


def test_cascade_repeat_is_bitwise_stable():
    case = W.cascade_case(3, group_sizes=[17, 4], prefix_lens=[200, 64], Hq=8, Hkv=2, D=128)
    (o1, l1), (o2, l2) = cascade_run(case, repeat=2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("shuffled", [False, True])
def test_radix_shared_cascade_full_size_every_request(shuffled):
    case = W.radix_shared_decode(0, shuffled=shuffled)
    (o, lse), = cascade_run(case)
    torch.cuda.empty_cache()
    assert_every_row_written(o, lse)
    want_o, want_lse, _ = oracle_run(case.compact(list(range(case.B))))
    compare(o, want_o)
    lse_compare(lse, want_lse)


def test_cascade_workspace_too_small_is_refused():
    import paged_kv_attention_out_gb300 as pkv
    case = W.cascade_case(1, group_sizes=[4], prefix_lens=[64], Hq=8, Hkv=2, D=64)
    pool, k, v, q, t = gpu_inputs(case, poison=False)
    ct = {name: torch.as_tensor(a, dtype=torch.int32, device="cuda")
          for name, a in W.cascade_tables(case).items()}
    n = pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, 1, 64,
                                       int(ct["seq_lens"].max()))
    ws = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_paged_cascade_decode_attn(
            pool, case.layer, q, o, None, ct["prefix_page_table"], ct["prefix_lens"],
            ct["member_indptr"], ct["members"], ct["page_table"], ct["seq_lens"], case.scale,
            64, int(ct["seq_lens"].max()), ws)
