"""pkv_merge_lse on the GPU against the oracle's closed-form merge."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built

pytestmark = pytest.mark.gpu


def _states(rows, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    o_a = torch.randn(rows, H, D, generator=g)
    o_b = torch.randn(rows, H, D, generator=g)
    l_a = torch.randn(rows, H, generator=g) * 5
    l_b = torch.randn(rows, H, generator=g) * 5
    l_a[0, 0] = -float("inf")
    l_b[1 % rows, 0] = -float("inf")
    l_a[2 % rows, H - 1] = -float("inf")
    l_b[2 % rows, H - 1] = -float("inf")
    return o_a, l_a, o_b, l_b


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,H,D", [(3, 4, 64), (257, 32, 128), (5, 3, 12)])
def test_merge_matches_oracle(out_dtype, rows, H, D):
    ensure_built()
    import paged_kv_attention_out_gb300 as pkv
    o_a, l_a, o_b, l_b = _states(rows, H, D, rows)
    want_o, want_l = oracle.merge_lse(o_a.double().numpy(), l_a.double().numpy(),
                                      o_b.double().numpy(), l_b.double().numpy())
    d = [x.cuda() for x in (o_a, l_a, o_b, l_b)]
    out = torch.full((rows, H, D), float("nan"), dtype=out_dtype, device="cuda")
    lse = torch.full((rows, H), float("nan"), device="cuda")
    pkv.pkv_merge_lse(*d, out, lse)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    tol = 1e-5 if out_dtype == torch.float32 else 2e-2
    np.testing.assert_allclose(got, want_o, rtol=0, atol=tol * max(1.0, np.abs(want_o).max()))
    gl = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(want_l))
    fin = ~np.isneginf(want_l)
    np.testing.assert_allclose(gl[fin], want_l[fin], rtol=0, atol=1e-5)


def test_merge_in_place():
    """o_out may alias o_a and lse_out may alias lse_a."""
    ensure_built()
    import paged_kv_attention_out_gb300 as pkv
    o_a, l_a, o_b, l_b = _states(64, 8, 128, 3)
    want_o, want_l = oracle.merge_lse(o_a.double().numpy(), l_a.double().numpy(),
                                      o_b.double().numpy(), l_b.double().numpy())
    a, la, b, lb = (x.cuda() for x in (o_a, l_a, o_b, l_b))
    pkv.pkv_merge_lse(a, la, b, lb, a, la)
    torch.cuda.synchronize()
    np.testing.assert_allclose(a.double().cpu().numpy(), want_o, rtol=0, atol=1e-4)
    fin = ~np.isneginf(want_l)
    np.testing.assert_allclose(la.double().cpu().numpy()[fin], want_l[fin], rtol=0, atol=1e-5)
