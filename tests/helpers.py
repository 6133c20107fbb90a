"""Shared helpers for the tests: run the oracle on a seeded case, compare results."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_attention_out_gb300 import workloads as W

# Attention tolerance on bf16 outputs against the fp64 oracle (both must hold).
MAX_ABS_TOL = 2e-2
MEAN_ABS_TOL = 2e-3
# lse is an fp32 output: its error is dominated by fp32 score accumulation.
LSE_ABS_TOL = 2e-3


def oracle_inputs(case: W.Case):
    """Host inputs of a case as the oracle takes them (uint16 bf16 bits)."""
    pool = W.bf16_bits(case.make_pool("cpu", poison=True)).reshape(case.pool_shape).copy()
    k, v = case.new_kv("cpu")
    q = case.q("cpu")
    return pool, W.bf16_bits(k), W.bf16_bits(v), W.bf16_bits(q)


def oracle_run(case: W.Case):
    """store_kv of the case's new tokens, then its attention, all on the oracle.

    Returns (o fp64, lse fp64, pool after store as uint16 bits).
    """
    pool, k, v, q = oracle_inputs(case)
    oracle.kv_store(pool, case.layer, k, v, case.out_loc)
    if case.kind == "decode":
        o, lse = oracle.decode_attn(pool, case.layer, q, case.page_table, case.seq_lens,
                                    case.scale, case.table_idx)
    else:
        o, lse = oracle.extend_attn(pool, case.layer, q, case.qo_indptr, case.page_table,
                                    case.seq_lens, case.scale, case.table_idx)
    return o, lse, pool


def compare(got: np.ndarray, want: np.ndarray, max_tol=MAX_ABS_TOL, mean_tol=MEAN_ABS_TOL,
            what="o", rel_rms_tol=None):
    """Element-wise check of bf16 outputs against the oracle: max and mean
    absolute error, and (rel_rms_tol) the error's RMS relative to the
    result's RMS, which is the tighter gate where |o| is small (long rows of
    N(0,1) values average to |o| ~ 1/sqrt(n))."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values in the result"
    err = np.abs(got - want)
    max_err = float(err.max()) if err.size else 0.0
    mean_err = float(err.mean()) if err.size else 0.0
    rms = float(np.sqrt((want ** 2).mean())) if want.size else 0.0
    rel_rms = float(np.sqrt((err ** 2).mean()) / rms) if rms > 0 else 0.0
    msg = (f"{what}: max|err| {max_err:.3e} (tol {max_tol}), mean|err| {mean_err:.3e} "
           f"(tol {mean_tol}), rel-rms {rel_rms:.3e}")
    assert max_err <= max_tol and mean_err <= mean_tol, msg
    if rel_rms_tol is not None:
        assert rel_rms <= rel_rms_tol, msg + f" (rel-rms tol {rel_rms_tol})"
    return max_err, mean_err


def lse_compare(got, want, tol=LSE_ABS_TOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    inf = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), inf), "lse: -inf positions differ"
    if (~inf).any():
        err = np.abs(got[~inf] - want[~inf])
        assert err.max() <= tol, f"lse: max|err| {err.max():.3e} (tol {tol})"


def to_bits(t: torch.Tensor) -> np.ndarray:
    return W.bf16_bits(t)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bits_exact(x) -> np.ndarray:
    """Values that are exact in bf16 -> bits (asserts exactness)."""
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# GPU side: the same case through the C ABI (pkv_* bindings)
# ---------------------------------------------------------------------------
_BUILT = False


def ensure_built():
    global _BUILT
    if not _BUILT:
        import __graft_entry__
        __graft_entry__.build()
        _BUILT = True


def gpu_inputs(case: W.Case, poison: bool = True, device="cuda"):
    ensure_built()
    pool = case.make_pool(device, poison=poison)
    k, v = case.new_kv(device)
    q = case.q(device)
    return pool, k, v, q, case.device_tables(device)


def nan_outputs(q: torch.Tensor, with_lse: bool = True):
    """o and lse buffers filled with NaN, so that any element a call fails to
    write stays NaN and shows up, instead of a stale finite value left in
    reused allocator memory."""
    o = torch.full_like(q, float("nan"))
    lse = (torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=q.device)
           if with_lse else None)
    return o, lse


def assert_every_row_written(o, lse=None, empty_rows=()):
    """After a call on NaN-filled outputs: every element of o is finite, and
    lse is finite on every row except the listed empty ones (-inf there)."""
    o = np.asarray(o.float().cpu() if isinstance(o, torch.Tensor) else o, np.float64)
    bad = ~np.isfinite(o)
    assert not bad.any(), f"o: {int(bad.sum())} elements unwritten or non-finite, first at " \
                          f"{np.argwhere(bad)[0].tolist()}"
    if lse is not None:
        lse = np.asarray(lse.cpu() if isinstance(lse, torch.Tensor) else lse, np.float64)
        want_inf = np.zeros(lse.shape, bool)
        for r in empty_rows:
            want_inf[r] = True
        assert np.all(np.isneginf(lse[want_inf])), "lse: an empty row is not -inf"
        ok = np.isfinite(lse[~want_inf])
        assert ok.all(), f"lse: {int((~ok).sum())} entries unwritten or non-finite"


def gpu_attention(case: W.Case, pool, q, t, hint=None, with_lse=True, table_idx=True):
    """Runs the case's attention call on the GPU on NaN-filled outputs;
    returns (o, lse) tensors."""
    import paged_kv_attention_out_gb300 as pkv
    o, lse = nan_outputs(q, with_lse)
    ti = t.get("table_idx") if table_idx else None
    if case.kind == "decode":
        h = case.max_seq_len if hint is None else hint
        n = pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, h)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
        pkv.pkv_paged_decode_attn(pool, case.layer, q, o, lse, t["page_table"], t["seq_lens"],
                                  case.scale, h, ws, table_idx=ti)
    else:
        h = case.max_seq_len if hint is None else hint
        total = int(case.seq_lens.sum())  # the workspace follows the keys present
        n = pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, h, total)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
        pkv.pkv_paged_extend_attn(pool, case.layer, q, t["qo_indptr"], o, lse, t["page_table"],
                                  t["seq_lens"], case.scale, h, ws, table_idx=ti,
                                  max_total_keys_hint=total)
    return o, lse


def gpu_run(case: W.Case, poison: bool = True, hint=None):
    """store_kv then attention on the GPU. Returns host fp64 (o, lse) and the pool."""
    import paged_kv_attention_out_gb300 as pkv
    pool, k, v, q, t = gpu_inputs(case, poison)
    pkv.pkv_kv_store(pool, case.layer, k, v, t["out_loc"])
    o, lse = gpu_attention(case, pool, q, t, hint=hint)
    torch.cuda.synchronize()
    return (o.float().cpu().double().numpy(), lse.cpu().double().numpy(), pool)


def check_against_oracle(case: W.Case, hint=None):
    o, lse, _ = gpu_run(case, hint=hint)
    want_o, want_lse, _ = oracle_run(case)
    compare(o, want_o)
    lse_compare(lse, want_lse)
    return o, lse
