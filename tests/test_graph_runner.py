"""The decode graph harness (DecodeGraphRunner): fused store_kv + decode
captured at batch sizes 1, 2, 4, ..., 64 and replayed at the smallest
captured size >= the step's batch, with seq_len 0 padding rows ("Code Notes:
mini-sglang", Engine Layer table, GraphRunner row). Every real row is
checked against the oracle, every padding row gives o = 0 and lse = -inf,
rows past the padded size are left alone, and a replay gives the bits of
the same call run eagerly at the padded size."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import compare, ensure_built, lse_compare, oracle_run
from paged_kv_attention_out_gb300 import workloads as W
from paged_kv_attention_out_gb300.graph_runner import DecodeGraphRunner, default_sizes


def test_default_sizes_and_padded_size():
    assert default_sizes(64) == [1, 2, 4, 8, 16, 32, 64]
    assert default_sizes(48) == [1, 2, 4, 8, 16, 32, 48]
    assert default_sizes(1) == [1]
    r = DecodeGraphRunner.__new__(DecodeGraphRunner)
    r.sizes = default_sizes(64)
    assert [r.padded_size(b) for b in (1, 2, 3, 5, 16, 17, 33, 64)] == [1, 2, 4, 8, 16, 32,
                                                                         64, 64]
    with pytest.raises(ValueError):
        r.padded_size(65)


def _case():
    rng = np.random.default_rng(81)
    seq = rng.integers(1, 1500, size=64)
    return W.random_case(81, seq_lens=seq.tolist(), Hq=32, Hkv=8, D=128, P=16)


@pytest.mark.gpu
def test_padded_batches_match_the_oracle():
    ensure_built()
    case = _case()
    pool = case.make_pool("cuda", poison=True)
    k, v = case.new_kv("cuda")
    q = case.q("cuda")
    t = case.device_tables("cuda")
    runner = DecodeGraphRunner(pool, case.layer, case.Hq, 64, t["page_table"].shape[1],
                               case.max_seq_len, case.scale)
    assert runner.sizes == [1, 2, 4, 8, 16, 32, 64]
    # 64 first: its rows stay in the static buffers and become padding later
    for b in (64, 1, 3, 5, 8, 13, 33):
        n = runner.padded_size(b)
        runner.o.fill_(float("nan"))
        runner.lse.fill_(float("nan"))
        o, lse = runner.run(q[:b], k[:b], v[:b], t["page_table"][:b], t["seq_lens"][:b])
        torch.cuda.synchronize()
        want_o, want_lse, _ = oracle_run(case.compact(list(range(b))))
        compare(o.float().cpu().double().numpy(), want_o)
        lse_compare(lse.cpu().double().numpy(), want_lse)
        assert torch.all(runner.o[b:n] == 0) and torch.all(torch.isneginf(runner.lse[b:n]))
        assert torch.isnan(runner.o[n:].float()).all() and torch.isnan(runner.lse[n:]).all()


@pytest.mark.gpu
def test_replay_equals_the_eager_call_at_the_padded_size():
    ensure_built()
    import paged_kv_attention_out_gb300 as pkv
    case = _case()
    pool = case.make_pool("cuda", poison=True)
    k, v = case.new_kv("cuda")
    q = case.q("cuda")
    t = case.device_tables("cuda")
    runner = DecodeGraphRunner(pool, case.layer, case.Hq, 64, t["page_table"].shape[1],
                               case.max_seq_len, case.scale)
    b = 13
    n = runner.padded_size(b)
    o_g, l_g = runner.run(q[:b], k[:b], v[:b], t["page_table"][:b], t["seq_lens"][:b])
    torch.cuda.synchronize()
    o_g, l_g = runner.o[:n].clone(), runner.lse[:n].clone()
    sl = runner.seq_lens[:n].clone()  # b real rows, then padding
    o_e = torch.full_like(q[:n], float("nan"))
    l_e = torch.full((n, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(pkv.pkv_decode_workspace_size(n, case.Hq, case.Hkv, case.D,
                                                       case.max_seq_len), 256),
                     dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_decode_attn_store(pool, case.layer, runner.q[:n], runner.k_new[:n],
                                    runner.v_new[:n], o_e, l_e, runner.page_table[:n], sl,
                                    case.scale, case.max_seq_len, ws)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)
