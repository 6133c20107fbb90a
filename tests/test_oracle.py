"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties the oracle to something fixed independently of its code: a
library routine for a special case (dense SDPA), closed forms, invariances
of the method (relocating pages, sharing a prefix, splitting the key set),
hand-derived golden values, or an independent brute-force restatement on
tiny inputs. A plausible slip in the oracle (a dropped key, a wrong GQA
index, a transposed page index, a misplaced causal edge, a wrong scale or
sign, a wrong lse) fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import bits_to_f64, f64_to_bits_exact, oracle_inputs, oracle_run
from paged_kv_attention_out_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _rand_bits(shape, seed, stream=W.STREAM_AUX):
    return W.bf16_bits(W.normal_tensor(shape, seed, stream))


def _identity_setup(seed, seq, Hq, Hkv, D):
    """P=1 pool where request b's keys sit at consecutive slots base_b + i."""
    NP = int(sum(seq)) + 7
    pool = _rand_bits((2, 1, NP, 1, Hkv, D), seed)
    q = _rand_bits((len(seq), Hq, D), seed, W.STREAM_Q)
    bases = np.concatenate([[3], 3 + np.cumsum(seq)[:-1]]).astype(np.int64)
    stride = max(seq)
    pt = np.zeros((len(seq), stride), np.int32)
    for b, n in enumerate(seq):
        pt[b, :n] = bases[b] + np.arange(n)
    return pool, q, pt, bases


def _dense_kv(pool, c, base, n):
    return torch.from_numpy(bits_to_f64(pool[c, 0, base:base + n, 0]))  # [n, Hkv, D]


@pytest.mark.parametrize("Hq,Hkv,D,scale", [(4, 2, 64, None), (8, 1, 32, 0.3),
                                            (6, 3, 16, None), (4, 4, 128, 0.05)])
def test_decode_identity_table_equals_dense_sdpa(Hq, Hkv, D, scale):
    """page_size 1 with identity rows is plain attention: torch SDPA, fp64."""
    seq = [1, 9, 37]
    scale = scale if scale is not None else 1.0 / math.sqrt(D)
    pool, q, pt, bases = _identity_setup(11, seq, Hq, Hkv, D)
    o, lse = oracle.decode_attn(pool, 0, q, pt, np.array(seq, np.int32), scale)
    g = Hq // Hkv
    for b, n in enumerate(seq):
        K = _dense_kv(pool, 0, bases[b], n).repeat_interleave(g, dim=1).transpose(0, 1)
        V = _dense_kv(pool, 1, bases[b], n).repeat_interleave(g, dim=1).transpose(0, 1)
        qq = torch.from_numpy(bits_to_f64(q[b]))[:, None, :]
        ref = F.scaled_dot_product_attention(qq, K, V, scale=scale)[:, 0, :]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("prefix,chunk", [(0, 5), (7, 1), (13, 6), (3, 17)])
def test_extend_identity_table_equals_sdpa_bottom_right_causal(prefix, chunk):
    """Extend over identity rows: SDPA with query j allowed keys i <= prefix + j."""
    Hq, Hkv, D = 4, 2, 32
    scale = 0.21
    n = prefix + chunk
    pool, _, pt, bases = _identity_setup(5, [n], Hq, Hkv, D)
    q = _rand_bits((chunk, Hq, D), 6, W.STREAM_Q)
    o, lse = oracle.extend_attn(pool, 0, q, np.array([0, chunk], np.int32), pt,
                                np.array([n], np.int32), scale)
    g = Hq // Hkv
    K = _dense_kv(pool, 0, bases[0], n).repeat_interleave(g, dim=1).transpose(0, 1)
    V = _dense_kv(pool, 1, bases[0], n).repeat_interleave(g, dim=1).transpose(0, 1)
    qq = torch.from_numpy(bits_to_f64(q)).transpose(0, 1)  # [Hq, chunk, D]
    allowed = torch.arange(n)[None, :] <= (prefix + torch.arange(chunk))[:, None]
    ref = F.scaled_dot_product_attention(qq, K, V, attn_mask=allowed, scale=scale)
    np.testing.assert_allclose(o, ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "log": math.log,
                                                     "exp": math.exp, "inf": math.inf}))


def _golden_pool(c, L=1):
    P, NP, Hkv, D = c["page_size"], c["num_pages"], c["kv_heads"], c["head_dim"]
    nan_bits = np.uint16(0x7FC0)
    pool = np.full((2, L, NP, P, Hkv, D), nan_bits, np.uint16)
    for which, key in ((0, "keys"), (1, "values")):
        for slot, rows in c[key].items():
            s = int(slot)
            pool[which, 0, s // P, s % P] = f64_to_bits_exact(rows)
    return pool


@pytest.mark.parametrize("idx", range(4))
def test_golden_closed_form_cases(idx):
    """Hand-derived values (golden file); unread slots hold NaN."""
    c = json.load(open(GOLDEN))["cases"][idx]
    pool = _golden_pool(c)
    q = f64_to_bits_exact(c["q"])
    pt = np.array(c["page_table"], np.int32)
    sl = np.array(c["seq_lens"], np.int32)
    if c["kind"] == "decode":
        o, lse = oracle.decode_attn(pool, 0, q, pt, sl, c["scale"])
    else:
        o, lse = oracle.extend_attn(pool, 0, q, np.array(c["qo_indptr"], np.int32), pt,
                                    sl, c["scale"])
    want_o = np.vectorize(_eval)(np.array(c["expect_o"], object)).astype(np.float64)
    want_lse = np.vectorize(_eval)(np.array(c["expect_lse"], object)).astype(np.float64)
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-14)


@pytest.mark.parametrize("idx", range(3))
def test_golden_merge_cases(idx):
    c = json.load(open(GOLDEN))["merge_cases"][idx]
    o, lse = oracle.merge_lse(np.array([[c["o_a"]]], float), np.array([[_eval(c["lse_a"])]]),
                              np.array([[c["o_b"]]], float), np.array([[_eval(c["lse_b"])]]))
    np.testing.assert_allclose(o[0, 0], [_eval(x) for x in c["expect_o"]], rtol=0, atol=1e-15)
    want = _eval(c["expect_lse"])
    if math.isinf(want):
        assert lse[0, 0] == want
    else:
        assert abs(lse[0, 0] - want) < 1e-15


def _relocated(pool, pt, P, NP, seed):
    """Move every physical page to pi(page); rewrite the table to match."""
    perm = np.random.default_rng(seed).permutation(NP)
    new = np.empty_like(pool)
    new[:, :, perm] = pool
    return new, perm[pt].astype(np.int32)


@pytest.mark.parametrize("P", [1, 4])
@pytest.mark.parametrize("kind", ["decode", "extend"])
def test_relocating_pages_changes_nothing(P, kind):
    seq = [5, 40, 23, 17]
    chunks = [5, 9, 1, 17] if kind == "extend" else None
    case = W.random_case(21, kind=kind, seq_lens=seq, chunk_lens=chunks, Hq=6, Hkv=2,
                         D=32, P=P)
    o1, l1, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    pool2, pt2 = _relocated(pool, case.page_table, P, case.NP, 3)
    if kind == "decode":
        o2, l2 = oracle.decode_attn(pool2, 0, q, pt2, case.seq_lens, case.scale)
    else:
        o2, l2 = oracle.extend_attn(pool2, 0, q, case.qo_indptr, pt2, case.seq_lens,
                                    case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("P", [1, 4])
def test_shared_prefix_equals_private_copies(P):
    """Rows that share prefix pages give exactly what private copies give."""
    seq = [44, 37, 52, 41, 60, 33]
    case = W.random_case(8, seq_lens=seq, Hq=4, Hkv=2, D=32, P=P, shared_prefix=32,
                         group_size=3, extra_pages=200)
    o1, l1, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    # give every request its own copy of the prefix pages, appended to the pool
    pt = case.page_table.copy()
    per = 32 // P
    pool2 = np.concatenate([pool, np.zeros(pool[:, :, :case.B * per].shape, pool.dtype)],
                           axis=2)
    dst = case.NP
    for b in range(case.B):
        for j in range(per):
            pool2[:, :, dst] = pool[:, :, int(pt[b, j])]
            pt[b, j] = dst
            dst += 1
    assert len(set(pt[:, 0])) == case.B  # prefixes are private now
    o2, l2 = oracle.decode_attn(pool2, 0, q, pt, case.seq_lens, case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_page_size_does_not_change_results():
    """The same logical keys stored in 8-token pages or in single slots agree."""
    seq = [19, 8, 33]
    case = W.random_case(4, seq_lens=seq, Hq=4, Hkv=2, D=16, P=8)
    o1, l1, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    n_tot = sum(seq)
    flat = np.zeros((2, 1, n_tot, 1, 2, 16), np.uint16)
    pt = np.zeros((3, max(seq)), np.int32)
    cur = 0
    for b, n in enumerate(seq):
        for i in range(n):
            s = int(case.token_slots[b][i])
            flat[:, 0, cur, 0] = pool[:, 0, s // 8, s % 8]
            pt[b, i] = cur
            cur += 1
    o2, l2 = oracle.decode_attn(flat, 0, q, pt, case.seq_lens, case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_single_key_returns_v():
    case = W.random_case(2, seq_lens=[1, 1, 1], Hq=4, Hkv=2, D=64, P=4)
    o, lse, pool = oracle_run(case)
    q = bits_to_f64(W.bf16_bits(case.q()))
    g = 2
    for b in range(3):
        s = int(case.out_loc[b])
        K = bits_to_f64(pool[0, 0, s // 4, s % 4])
        V = bits_to_f64(pool[1, 0, s // 4, s % 4])
        for h in range(4):
            assert np.array_equal(o[b, h], V[h // g])
            assert abs(lse[b, h] - case.scale * float(np.dot(q[b, h], K[h // g]))) < 1e-12


def test_zero_query_gives_mean_of_v():
    case = W.random_case(3, seq_lens=[1, 6, 29], Hq=4, Hkv=2, D=32, P=2)
    pool, k, v, q = oracle_inputs(case)
    oracle.kv_store(pool, 0, k, v, case.out_loc)
    q0 = np.zeros_like(q)
    o, lse = oracle.decode_attn(pool, 0, q0, case.page_table, case.seq_lens, case.scale)
    for b, n in enumerate(case.seq_lens):
        slots = case.token_slots[b]
        V = bits_to_f64(pool[1, 0, slots // 2, slots % 2])  # [n, Hkv, D]
        for h in range(4):
            np.testing.assert_allclose(o[b, h], V[:, h // 2].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[b, h] - math.log(n)) < 1e-13


@pytest.mark.parametrize("P", [1, 16])
def test_spike_key_dominates(P):
    """One key with a huge score returns that key's V; catches dropped or
    misrouted keys, which averaging over many N(0,1) keys would hide."""
    seq = [300, 77]
    case = W.random_case(9, seq_lens=seq, Hq=8, Hkv=2, D=64, P=P)
    pool, k, v, q = oracle_inputs(case)
    oracle.kv_store(pool, 0, k, v, case.out_loc)
    qf = bits_to_f64(q)
    rng = np.random.default_rng(1)
    for b in range(2):
        j = int(rng.integers(seq[b]))
        s = int(case.token_slots[b][j])
        # key j of kv head 0 := 8 * q of head 0 (exact in bf16)
        pool[0, 0, s // P, s % P, 0] = f64_to_bits_exact(8.0 * qf[b, 0])
        o, _ = oracle.decode_attn(pool, 0, q, case.page_table, case.seq_lens, case.scale)
        V = bits_to_f64(pool[1, 0, s // P, s % P, 0])
        np.testing.assert_allclose(o[b, 0], V, rtol=0, atol=1e-12)


def test_split_and_merge_equals_whole():
    """attention over [0,n) = merge(attention [0,k), attention [k,n)) for all k."""
    n = 57
    pool, q, pt, bases = _identity_setup(31, [n], 4, 2, 32)
    sl = np.array([n], np.int32)
    o, lse = oracle.decode_attn(pool, 0, q, pt, sl, 0.17)
    for k in range(0, n + 1):
        oa, la = oracle.decode_attn(pool, 0, q, pt[:, :max(k, 1)], np.array([k], np.int32), 0.17)
        rest = np.ascontiguousarray(pt[:, k:]) if k < n else pt[:, :1]
        ob, lb = oracle.decode_attn(pool, 0, q, rest, np.array([n - k], np.int32), 0.17)
        om, lm = oracle.merge_lse(oa, la, ob, lb)
        np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


def test_merge_is_associative_and_symmetric():
    rng = np.random.default_rng(0)
    o = [rng.standard_normal((5, 3, 8)) for _ in range(3)]
    lse = [rng.standard_normal((5, 3)) * 4 for _ in range(3)]
    lse[1][0, 0] = -np.inf
    ab = oracle.merge_lse(o[0], lse[0], o[1], lse[1])
    left = oracle.merge_lse(*ab, o[2], lse[2])
    bc = oracle.merge_lse(o[1], lse[1], o[2], lse[2])
    right = oracle.merge_lse(o[0], lse[0], *bc)
    np.testing.assert_allclose(left[0], right[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], rtol=0, atol=1e-12)
    ba = oracle.merge_lse(o[1], lse[1], o[0], lse[0])
    np.testing.assert_allclose(ab[0], ba[0], rtol=0, atol=1e-15)
    # merging a state with itself keeps o and adds log 2
    same = oracle.merge_lse(o[2], lse[2], o[2], lse[2])
    np.testing.assert_allclose(same[0], o[2], rtol=0, atol=1e-14)
    np.testing.assert_allclose(same[1], lse[2] + math.log(2), rtol=0, atol=1e-14)


def _brute(pool, q, rows, seq, Hkv, P, scale, causal_prefix=None):
    """Independent numpy restatement: gather whole K/V, softmax by np.exp."""
    out_o, out_l = [], []
    for t in range(q.shape[0]):
        n = seq[t]
        pages = np.asarray(rows[t])[np.arange(n) // P]
        offs = np.arange(n) % P
        K = bits_to_f64(pool[0, 0, pages, offs])  # [n, Hkv, D]
        V = bits_to_f64(pool[1, 0, pages, offs])
        qt = bits_to_f64(q[t])  # [Hq, D]
        g = qt.shape[0] // Hkv
        Kh = np.repeat(K, g, axis=1)  # [n, Hq, D]
        Vh = np.repeat(V, g, axis=1)
        s = scale * np.einsum("hd,nhd->hn", qt, Kh)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        z = w.sum(axis=1, keepdims=True)
        out_o.append(np.einsum("hn,nhd->hd", w / z, Vh))
        out_l.append(s.max(axis=1) + np.log(z[:, 0]))
    return np.array(out_o), np.array(out_l)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    P = int(rng.choice([1, 2, 4]))
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    seq = rng.integers(1, 9, size=B).tolist()
    case = W.random_case(200 + seed, seq_lens=seq, Hq=Hq, Hkv=Hkv, D=8, P=P,
                         use_table_idx=bool(seed % 2))
    o, lse, pool = oracle_run(case)
    rows = [case.page_table[case.table_idx[b] if case.table_idx is not None else b]
            for b in range(B)]
    bo, bl = _brute(pool, W.bf16_bits(case.q()), rows, seq, Hkv, P, case.scale)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_tiny_extend(seed):
    rng = np.random.default_rng(300 + seed)
    P = int(rng.choice([1, 2]))
    B = 2
    chunks = rng.integers(1, 5, size=B)
    seq = (chunks + rng.integers(0, 5, size=B)).tolist()
    case = W.random_case(400 + seed, kind="extend", seq_lens=seq, chunk_lens=chunks.tolist(),
                         Hq=4, Hkv=2, D=8, P=P)
    o, lse, pool = oracle_run(case)
    rows, n_keys = [], []
    for b in range(B):
        p = seq[b] - int(chunks[b])
        for j in range(int(chunks[b])):
            rows.append(case.page_table[b])
            n_keys.append(p + j + 1)
    bo, bl = _brute(pool, W.bf16_bits(case.q()), rows, n_keys, 2, P, case.scale)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_extend_query_equals_decode_at_its_position():
    """Chunk query j of request r is a decode over the first p_r + j + 1 keys."""
    case = W.random_case(12, kind="extend", seq_lens=[30, 12, 19], chunk_lens=[6, 12, 1],
                         Hq=4, Hkv=1, D=16, P=4)
    o, lse, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    t = 0
    for r in range(case.B):
        c = int(case.qo_indptr[r + 1] - case.qo_indptr[r])
        p = int(case.seq_lens[r]) - c
        for j in range(c):
            od, ld = oracle.decode_attn(pool, 0, q[t:t + 1], case.page_table[r:r + 1],
                                        np.array([p + j + 1], np.int32), case.scale)
            assert np.array_equal(od[0], o[t]) and np.array_equal(ld[0], lse[t])
            t += 1


def test_table_idx_selects_rows():
    case = W.random_case(14, seq_lens=[9, 3, 27, 14], Hq=4, Hkv=2, D=16, P=2,
                         use_table_idx=True)
    o1, l1, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    direct = case.page_table[case.table_idx]
    o2, l2 = oracle.decode_attn(pool, 0, q, direct, case.seq_lens, case.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_empty_sequence_gives_zero_and_neg_inf():
    case = W.random_case(15, seq_lens=[4, 2], Hq=2, Hkv=1, D=8, P=1)
    pool, k, v, q = oracle_inputs(case)
    oracle.kv_store(pool, 0, k, v, case.out_loc)
    o, lse = oracle.decode_attn(pool, 0, q, case.page_table, np.array([0, 2], np.int32),
                                case.scale)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("P", [1, 4])
def test_kv_store_is_a_bit_copy_to_out_loc(P):
    case = W.random_case(16, seq_lens=[5, 11, 2], Hq=4, Hkv=2, D=16, P=P, L=3, layer=1)
    pool, k, v, q = oracle_inputs(case)
    pool[:, [0, 2]] = 0x1234  # other layers: a sentinel that must survive
    before = pool.copy()
    oracle.kv_store(pool, 1, k, v, case.out_loc)
    want = before.copy()
    for i, s in enumerate(case.out_loc):
        want[0, 1, s // P, s % P] = k[i]
        want[1, 1, s // P, s % P] = v[i]
    assert np.array_equal(pool, want)
    assert np.all(pool[:, [0, 2]] == 0x1234)


def test_oracle_rejects_bad_arguments():
    case = W.random_case(17, seq_lens=[5], Hq=4, Hkv=2, D=16, P=1)
    pool, k, v, q = oracle_inputs(case)
    with pytest.raises(ValueError):
        oracle.decode_attn(pool, 1, q, case.page_table, case.seq_lens, case.scale)  # layer
    bad = case.page_table.copy()
    bad[0, 0] = case.NP + 5
    with pytest.raises(ValueError):
        oracle.decode_attn(pool, 0, q, bad, case.seq_lens, case.scale)
    with pytest.raises(ValueError):
        oracle.kv_store(pool, 0, k, v, np.array([case.NP * case.P], np.int32))


@pytest.mark.parametrize("P", [1, 8])
def test_cascade_decomposition_of_shared_prefix_decode(P):
    """Reading R11: a request of a shared-prefix group attends to its group's
    prefix keys followed by its own suffix keys, so its attention is the
    log-sum-exp merge of attention over the prefix row and attention over the
    suffix row (the merge invariant, pinned above, applied to the cascade
    tables); an empty prefix leaves the suffix state unchanged."""
    case = W.cascade_case(4, group_sizes=[3, 5, 2], prefix_lens=[16, 40, 0], P=P, Hq=4, Hkv=2,
                          D=32, suffix_lo=1, suffix_hi=30)
    want_o, want_lse, pool = oracle_run(case)
    q = W.bf16_bits(case.q())
    t = W.cascade_tables(case)
    gof = np.asarray(case.notes["group_of_request"])
    # the prefix state of each request: its group's prefix row
    pre_pt = t["prefix_page_table"][gof]
    pre_len = t["prefix_lens"][gof]
    o_p, l_p = oracle.decode_attn(pool, case.layer, q, pre_pt, pre_len, case.scale)
    o_s, l_s = oracle.decode_attn(pool, case.layer, q, t["page_table"], t["seq_lens"], case.scale)
    o, lse = oracle.merge_lse(o_p, l_p, o_s, l_s)
    assert np.allclose(o, want_o, atol=1e-12, rtol=0) and np.allclose(lse, want_lse, atol=1e-12)
    empty = pre_len == 0
    assert empty.any()
    assert np.array_equal(o[empty], o_s[empty]) and np.array_equal(lse[empty], l_s[empty])
