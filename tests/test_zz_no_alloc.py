"""pkv_paged_decode_attn_noalloc: decode attention that allocates nothing.

Some callers cannot allocate device memory or hand the library a
workspace: a plugin inside a host framework that owns all device memory and
offers no allocation hook, or a serving loop that must never call cudaMalloc
because it can synchronise the device and fail with out-of-memory mid-step.
For them the library keeps the split-KV scratch in a fixed device array of
its own. These tests call that entry point through the C ABI and check it
bit for bit against pkv_paged_decode_attn with a caller workspace (the
same plan and kernels), and the first call also against the oracle, on two
calls in a row (the second call finds the first call's leftovers in the
shared scratch), and check that a plan larger than the array is refused.
"""
from __future__ import annotations

import pytest
import torch

from helpers import (assert_every_row_written, compare, ensure_built, gpu_attention, gpu_inputs,
                     lse_compare, nan_outputs, oracle_run)
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _noalloc_vs_workspace(case, against_oracle=False):
    """Both calls run the same split plan and kernels, so the scratch variant
    must give the workspace variant's bits exactly: a wrong scratch offset or
    a leftover of the previous call would change them."""
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    need = pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.max_seq_len)
    assert 0 < need <= SCRATCH_BYTES, "the case must exercise the split scratch"
    want_o, want_lse = gpu_attention(case, pool, q, t)  # caller-provided workspace
    o, lse = nan_outputs(q)
    pkv.pkv_paged_decode_attn_noalloc(pool, case.layer, q, o, lse, t["page_table"],
                                      t["seq_lens"], case.scale, case.max_seq_len,
                                      table_idx=t.get("table_idx"))
    torch.cuda.synchronize()
    assert_every_row_written(o, lse)
    assert torch.equal(o, want_o) and torch.equal(lse, want_lse)
    if against_oracle:
        oo, ol, _ = oracle_run(case)
        compare(o.double().cpu().numpy(), oo)
        lse_compare(lse.double().cpu().numpy(), ol)


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    ensure_built()
    first = W.random_case(71, seq_lens=[3000, 17, 1200, 4096, 640], Hq=32, Hkv=8, D=128,
                          P=1)
    second = W.random_case(72, seq_lens=[9000, 33, 2500], Hq=32, Hkv=4, D=128, P=16,
                           use_table_idx=True)
    _noalloc_vs_workspace(first, against_oracle=True)
    _noalloc_vs_workspace(second)


def test_noalloc_refuses_a_plan_larger_than_its_scratch():
    ensure_built()
    import paged_kv_attention_out_gb300 as pkv
    batch, need = None, 0
    for b in range(100, 8192, 100):
        need = pkv.pkv_decode_workspace_size(b, 32, 4, 128, 4096)
        if need > SCRATCH_BYTES:
            batch = b
            break
    assert batch is not None, "no batch size needs more scratch than the array holds"
    dev = "cuda"
    pool = torch.zeros(2, 1, 16, 16, 4, 128, dtype=torch.bfloat16, device=dev)
    q = torch.zeros(batch, 32, 128, dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    pt = torch.zeros(batch, 1, dtype=torch.int32, device=dev)
    sl = torch.ones(batch, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_decode_attn_noalloc(pool, 0, q, o, None, pt, sl, 0.1, 4096)
    assert ei.value.status == 3 and "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.all(o == 0)  # nothing was launched
