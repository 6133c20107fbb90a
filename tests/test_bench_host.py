"""Host-side logic of bench.py: work formulas, rank aggregation (gloo,
world size 2), and the reference arm (the oracle), all on the CPU."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from paged_kv_attention_out_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_formulas_match_the_workload_descriptions():
    c2 = W.llama8b_decode(0)
    assert abs(bench.decode_bytes(c2) - int(c2.seq_lens.sum()) * 4100) < 2e6
    c4 = W.chunked_prefill_extend(0)
    c = np.diff(c4.qo_indptr)
    p = c4.seq_lens - c
    brute = 0
    for r in range(c4.B):  # count allowed (query, key) pairs one query at a time
        brute += sum(int(p[r]) + j + 1 for j in range(int(c[r])))
    assert bench.extend_flops(c4) == pytest.approx(4 * 128 * 32 * brute, rel=1e-12)
    c3 = W.radix_shared_decode(0)
    assert bench.decode_bytes(c3, unique=True) < bench.decode_bytes(c3) / 5
    c5 = W.long_context_decode(0)
    assert 2.0e9 < bench.decode_bytes(c5) < 3.5e9


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r reports 10 + r ms for 5 units each
    t, u = bench.aggregate_ranks(10.0 + rank, 5.0, world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_rank_aggregation_takes_max_time_and_total_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 11.0, 10.0), (1, 11.0, 10.0)]


def test_single_rank_aggregation_is_identity():
    assert bench.aggregate_ranks(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_gpus_must_match_the_running_ranks():
    """`--gpus 2` without a second rank exits non-zero instead of measuring one
    GPU under an n_gpus of 1."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300, env=env)
    assert r.returncode != 0 and "--gpus 2" in r.stderr and r.stdout.strip() == ""


def _bench_rank(rank, world, port, q):
    """One rank of `bench.py --impl reference --gpus 2` under a gloo world."""
    import contextlib
    import io
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "1",
                    "--warmup", "3"])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out.getvalue()))


def test_world_of_two_reports_n_gpus_equal_to_the_world_size():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30000 + os.getpid() % 1000
    procs = [ctx.Process(target=_bench_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[1].strip() == ""  # only rank 0 prints
    lines = [x for x in out[0].splitlines() if x.strip()]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_e2e_staging_buffer_round_trips_every_tensor(monkeypatch):
    """The e2e step moves its inputs in one copy: every tensor's view of the
    staging buffer holds exactly its bytes, at a 256-byte aligned offset."""
    import torch
    import bench
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)  # no CUDA here
    x = {"q": torch.randn(3, 4, 8).to(torch.bfloat16), "t": torch.arange(11, dtype=torch.int32),
         "l": torch.randn(5, 3)}
    host, dev, views = bench._staging(x, "cpu")
    assert host.numel() == 256 * 3
    dev.copy_(host)
    for name, t in x.items():
        assert views[name].dtype == t.dtype and views[name].shape == t.shape
        assert torch.equal(views[name], t)
        assert (views[name].data_ptr() - dev.data_ptr()) % 256 == 0
