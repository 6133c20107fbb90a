"""store_kv on the GPU: bit-exact against the oracle, nothing else touched."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built, oracle_inputs
from paged_kv_attention_out_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _store_both(case, k_dev=None, v_dev=None):
    import paged_kv_attention_out_gb300 as pkv
    ensure_built()
    pool = case.make_pool("cuda", poison=True)
    # other layers: a sentinel that must survive untouched
    for lyr in range(case.L):
        if lyr != case.layer:
            pool[:, lyr].view(torch.int16).fill_(0x1234)
    k, v = case.new_kv("cuda")
    if k_dev is not None:
        k, v = k_dev, v_dev
    t = case.device_tables("cuda")
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    torch.cuda.synchronize()
    hp, hk, hv, _ = oracle_inputs(case)
    for lyr in range(case.L):
        if lyr != case.layer:
            hp[:, lyr] = 0x1234
    oracle.kv_store(hp, case.layer, W.bf16_bits(k), W.bf16_bits(v), case.out_loc)
    return W.bf16_bits(pool).reshape(case.pool_shape), hp


@pytest.mark.parametrize("P", [1, 16])
@pytest.mark.parametrize("D,Hkv", [(64, 2), (128, 8), (128, 1)])
def test_store_is_bit_exact(P, D, Hkv):
    case = W.random_case(31, seq_lens=[3, 40, 17, 1, 64], Hq=Hkv, Hkv=Hkv, D=D, P=P, L=3,
                         layer=1)
    got, want = _store_both(case)
    assert np.array_equal(got, want)


def test_store_many_tokens_extend_style():
    case = W.random_case(32, kind="extend", seq_lens=[700, 1500, 333],
                         chunk_lens=[300, 1500, 200], Hq=8, Hkv=8, D=128, P=1)
    got, want = _store_both(case)
    assert np.array_equal(got, want)


def test_store_from_fused_qkv_rows():
    """k and v may be column slices of one [N, (Hq + 2 Hkv) * D] projection output."""
    case = W.random_case(33, seq_lens=[5, 9, 12, 30], Hq=8, Hkv=2, D=128, P=16)
    k, v = case.new_kv("cuda")
    n = case.n_new
    fused = torch.zeros(n, (8 + 4) * 128, dtype=torch.bfloat16, device="cuda")
    fused[:, 1024:1280] = k.reshape(n, -1)
    fused[:, 1280:1536] = v.reshape(n, -1)
    ks = fused[:, 1024:1280].view(n, 2, 128)
    vs = fused[:, 1280:1536].view(n, 2, 128)
    got, want = _store_both(case, ks, vs)
    assert np.array_equal(got, want)


def test_out_of_range_slot_is_dropped_and_reported():
    import paged_kv_attention_out_gb300 as pkv
    ensure_built()
    case = W.random_case(34, seq_lens=[4, 4], Hq=2, Hkv=2, D=64, P=1)
    pool = case.make_pool("cuda", poison=False)
    before = pool.clone()
    k, v = case.new_kv("cuda")
    bad = torch.tensor([case.NP * case.P, -1], dtype=torch.int32, device="cuda")
    pkv.pkv_read_device_errors()  # clear
    pkv.pkv_kv_store(pool, 0, k, v, bad)
    flags = pkv.pkv_read_device_errors()
    assert flags & 0x1
    assert torch.equal(pool.view(torch.int16), before.view(torch.int16))
