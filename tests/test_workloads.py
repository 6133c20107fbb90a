"""The seeded input generator: determinism, recipes, and compact sub-cases."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import oracle_run
from paged_kv_attention_out_gb300 import workloads as W


def test_values_are_a_function_of_position_only():
    a = W.normal_tensor((3, 1000), 7, W.STREAM_Q)
    b = torch.empty(3000, dtype=torch.bfloat16)
    W.fill_normal_(b, 7, W.STREAM_Q, chunk=77)  # chunking does not matter
    assert torch.equal(a.view(-1), b)
    idx = torch.tensor([5, 1234, 2999])
    assert torch.equal(W.normal_bf16(7, W.STREAM_Q, idx), a.view(-1)[idx])
    # other seed or stream: different numbers
    assert not torch.equal(a, W.normal_tensor((3, 1000), 8, W.STREAM_Q))
    assert not torch.equal(a, W.normal_tensor((3, 1000), 7, W.STREAM_K_NEW))


def test_counter_hash_is_exact_past_32_bits():
    idx = torch.tensor([0, 2**32 - 1, 2**32, 2**33 + 5, 26 * 2**30], dtype=torch.int64)
    v = W.normal_bf16(0, W.STREAM_POOL, idx)
    assert v.dtype == torch.bfloat16 and torch.isfinite(v.float()).all()
    assert len(set(v.float().tolist())) > 1


def test_distribution_is_standard_normal():
    x = W.normal_tensor((1 << 20,), 1, W.STREAM_POOL).double()
    assert abs(float(x.mean())) < 5e-3
    assert abs(float(x.std()) - 1.0) < 5e-3
    assert float(x.abs().max()) < 4.5


def test_named_recipes_follow_their_descriptions():
    c = W.tiny_decode()
    assert list(c.seq_lens) == [1, 7, 16, 33] and (c.Hq, c.Hkv, c.D, c.P) == (4, 2, 64, 1)
    c = W.llama8b_decode()
    assert c.B == 64 and c.seq_lens.min() >= 512 and c.seq_lens.max() <= 4096
    assert (c.Hq, c.Hkv, c.D, c.P, c.L, c.NP) == (32, 8, 128, 1, 32, 400_000)
    assert len(np.unique(np.concatenate(c.token_slots))) == int(c.seq_lens.sum())
    c = W.radix_shared_decode()
    assert c.B == 256 and c.seq_lens.min() >= 2049 and c.seq_lens.max() <= 2560
    assert len(c.referenced_slots()) < int(c.seq_lens.sum())  # prefixes shared
    c = W.chunked_prefill_extend()
    ch = np.diff(c.qo_indptr)
    assert c.total_q == 8192 and ch.min() >= 512 and ch.max() <= 2048
    assert np.all(c.seq_lens - ch >= 0) and np.all(c.seq_lens - ch <= 8192)
    c = W.long_context_decode()
    assert c.P == 16 and c.seq_lens.min() >= 32768 and c.seq_lens.max() <= 131072
    assert c.NP == int(((c.seq_lens + 15) // 16).sum()) + 1024


def test_out_loc_is_the_newest_key_slot():
    c = W.random_case(3, seq_lens=[4, 9], P=4)
    assert [int(x) for x in c.out_loc] == [int(s[-1]) for s in c.token_slots]
    e = W.random_case(3, kind="extend", seq_lens=[7, 5], chunk_lens=[2, 5], P=2)
    want = np.concatenate([e.token_slots[0][5:], e.token_slots[1][0:]])
    assert np.array_equal(e.out_loc, want)


def test_poison_covers_everything_not_yet_written():
    c = W.random_case(4, seq_lens=[5, 3], P=4, extra_pages=3)
    pool = c.make_pool("cpu", poison=True)
    plane = pool[0, 0].reshape(c.NP * c.P, -1)
    finite = torch.isfinite(plane.float()).all(dim=1).nonzero().view(-1).numpy()
    assert np.array_equal(np.sort(finite), c.slots_before_store())


def test_compact_case_reproduces_the_full_case():
    """Oracle on a compact cut of requests == oracle on the full case, exactly."""
    for kind in ("decode", "extend"):
        seq = [40, 13, 77, 29, 51]
        chunks = [3, 5, 20, 1, 8] if kind == "extend" else None
        c = W.random_case(5, kind=kind, seq_lens=seq, chunk_lens=chunks, Hq=4, Hkv=2, D=16,
                          P=4, shared_prefix=8, group_size=2)
        o, lse, _ = oracle_run(c)
        keep = [3, 0]
        sub = c.compact(keep)
        so, slse, _ = oracle_run(sub)
        if kind == "decode":
            rows = keep
        else:
            rows = np.concatenate([np.arange(c.qo_indptr[b], c.qo_indptr[b + 1])
                                   for b in keep])
        assert np.array_equal(so, o[rows]) and np.array_equal(slse, lse[rows])


@pytest.mark.parametrize("P", [1, 16])
def test_cascade_tables_rebuild_every_key_list(P):
    """Prefix row + suffix row of each request name exactly its keys, in order."""
    case = W.cascade_case(5, group_sizes=[3, 70, 1], prefix_lens=[32, 64, 0], P=P, Hq=8, Hkv=2)
    t = W.cascade_tables(case)
    gof = np.asarray(case.notes["group_of_request"])
    for k in range(len(t["prefix_lens"])):
        mem = t["members"][t["member_indptr"][k]:t["member_indptr"][k + 1]]
        assert np.all(gof[mem] == k)
    assert sorted(t["members"].tolist()) == list(range(case.B))
    for b in range(case.B):
        g = gof[b]
        pre = [int(t["prefix_page_table"][g][i // P]) * P + i % P for i in range(t["prefix_lens"][g])]
        suf = [int(t["page_table"][b][i // P]) * P + i % P for i in range(t["seq_lens"][b])]
        assert pre + suf == [int(x) for x in case.token_slots[b]]


def test_cascade_tables_of_the_radix_workload():
    case = W.radix_shared_decode(0, shuffled=True)
    t = W.cascade_tables(case)
    assert t["prefix_lens"].tolist() == [2048] * 8
    assert np.all(t["seq_lens"] == case.seq_lens - 2048)
