"""The calls inside CUDA graphs: store_kv + decode, store_kv + extend and
store_kv + cascade decode captured once and replayed on new inputs give the
same bits as the same calls run eagerly ("Code Notes: mini-sglang", Engine
Layer table, GraphRunner row: decode steps are replayed from CUDA graphs).
The calls never allocate or synchronise, and every launch parameter comes
from host scalars, so a captured step stays valid while the buffers live."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import ensure_built
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _setup(case):
    ensure_built()
    dev = "cuda"
    pool = case.make_pool(dev, poison=True)
    k, v = case.new_kv(dev)
    q = case.q(dev)
    t = case.device_tables(dev)
    return pool, k, v, q, t


def _graph_vs_eager(case, call, inputs):
    """call(pool, k, v, q) enqueues one step; returns eager and replayed (o, lse)."""
    pool, k, v, q, t = inputs
    o_e, l_e = call(pool, k, v, q)  # eager (also initialises per-device state)
    torch.cuda.synchronize()
    o_e, l_e = o_e.clone(), l_e.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            o_g, l_g = call(pool, k, v, q)
    torch.cuda.current_stream().wait_stream(s)
    o_g.zero_()
    l_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)
    # new inputs in the captured buffers: the replay follows them
    q.copy_(torch.flip(q, dims=[0]))
    g.replay()
    o_e2, l_e2 = call(pool, k, v, q)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e2) and torch.equal(l_g, l_e2)
    return o_g


def test_decode_step_in_a_graph():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(11, seq_lens=np.arange(16) * 97 + 5, Hq=32, Hkv=8, D=128, P=16)
    inputs = _setup(case)
    t = inputs[4]
    h = case.max_seq_len
    ws = torch.empty(max(pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, h), 256),
                     dtype=torch.uint8, device="cuda")

    def call(pool, k, v, q):
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
        pkv.pkv_paged_decode_attn(pool, case.layer, q, o, lse, t["page_table"], t["seq_lens"],
                                  case.scale, h, ws)
        return o, lse

    o = _graph_vs_eager(case, call, inputs)
    assert np.isfinite(o.float().cpu().numpy()).all()


def test_extend_step_in_a_graph():
    import paged_kv_attention_out_gb300 as pkv
    case = W.random_case(12, kind="extend", seq_lens=[300, 77, 1024, 9],
                         chunk_lens=[100, 77, 200, 9], Hq=8, Hkv=2, D=128, P=1)
    inputs = _setup(case)
    t = inputs[4]
    h, total = case.max_seq_len, int(case.seq_lens.sum())
    ws = torch.empty(pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h, total),
                     dtype=torch.uint8, device="cuda")

    def call(pool, k, v, q):
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
        pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, lse, t["page_table"],
                                  t["seq_lens"], case.scale, h, ws, max_total_keys_hint=total)
        return o, lse

    _graph_vs_eager(case, call, inputs)


def test_cascade_step_in_a_graph():
    import paged_kv_attention_out_gb300 as pkv
    case = W.cascade_case(13, group_sizes=[20, 5, 1], prefix_lens=[512, 128, 0], Hq=32, Hkv=8,
                          D=128, suffix_hi=300)
    inputs = _setup(case)
    t = inputs[4]
    ct = {n: torch.as_tensor(a, dtype=torch.int32, device="cuda")
          for n, a in W.cascade_tables(case).items()}
    pmax, smax = max(int(ct["prefix_lens"].max()), 1), int(ct["seq_lens"].max())
    ws = torch.empty(pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, 3, pmax,
                                                    smax), dtype=torch.uint8, device="cuda")

    def call(pool, k, v, q):
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
        pkv.pkv_paged_cascade_decode_attn(
            pool, case.layer, q, o, lse, ct["prefix_page_table"], ct["prefix_lens"],
            ct["member_indptr"], ct["members"], ct["page_table"], ct["seq_lens"], case.scale,
            pmax, smax, ws)
        return o, lse

    _graph_vs_eager(case, call, inputs)
