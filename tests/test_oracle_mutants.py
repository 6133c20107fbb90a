"""The oracle's pins catch plausible slips.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs the pin suite
(test_oracle.py) against that copy in a subprocess. The suite must fail for
every mutant; the unmodified copy must pass.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

# (name, text in pkv_oracle.c, replacement)
MUTANTS = [
    ("gqa-head-map-modulo", "attend(pool, g, layer, h / group, q + bh * D",
     "attend(pool, g, layer, h % Hkv, q + bh * D"),
    ("last-key-dropped", "    s[i] = scale * acc;",
     "    s[i] = (i == n - 1 && n > 1) ? -INFINITY : scale * acc;"),
    ("causal-edge-off-by-one", "p + j + 1, scale, s,", "p + j, scale, s,"),
    ("page-offset-reversed", "  *off = i % P;", "  *off = (P - 1) - i % P;"),
    ("scale-not-applied", "    s[i] = scale * acc;", "    s[i] = acc;"),
    ("lse-base-2", "  *lse = m + log(z);", "  *lse = m + log2(z);"),
    ("v-read-from-k-plane", "w * widen(pool[pool_pos(g, 1, layer, page, off, kvh, d)])",
     "w * widen(pool[pool_pos(g, 0, layer, page, off, kvh, d)])"),
    ("store-v-from-k", "pool[pool_pos(g, 1, layer, page, off, h, d)] = v[",
     "pool[pool_pos(g, 1, layer, page, off, h, d)] = k["),
    ("layer-ignored", "((((c * g.L + layer) * g.NP", "((((c * g.L + 0) * g.NP"),
    ("table-idx-ignored",
     "page_table + (table_idx ? (int64_t)table_idx[b] : b) * table_stride;\n      attend",
     "page_table + b * table_stride;\n      attend"),
    ("merge-weight-sign", "wb = exp(lb - m);", "wb = exp(m - lb);"),
    ("softmax-missing-normaliser", "    double w = exp(s[i] - m) / z;",
     "    double w = exp(s[i] - m);"),
]


def _run_pins(lib_path: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, PKV_ORACLE_LIB=lib_path)
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _build_variant(tmp_path, name, text, repl):
    src = open(SRC).read()
    if text is not None:
        assert src.count(text) >= 1, f"mutation site for {name} not found"
        src = src.replace(text, repl, 1)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    out = str(tmp_path / f"lib{name}.so")
    oracle.compile_to(str(path), out)
    return out


def test_unmodified_copy_passes(tmp_path):
    r = _run_pins(_build_variant(tmp_path, "clean", None, None))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,text,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_fail_on_mutant(tmp_path, name, text, repl):
    r = _run_pins(_build_variant(tmp_path, name, text, repl))
    assert r.returncode != 0, f"mutant {name} passed every pin"
