#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention step on GB300 (sm_103a).

One step = one pass of the decode hot path over one batch of the
Llama-3-8B-shaped workload (64 requests, 32 q / 8 kv heads, head_dim 128,
page_size 1, seq_len uniform in [512, 4096], a 400k-slot pool of 32
layers): store_kv of the 64 new tokens (fused into the decode launch),
split-KV decode attention through the page table, and the cross-split
log-sum-exp merge. `value` is decode
attention KV throughput in GB/s (algorithmic bytes: every K/V byte of every
key, the page-table entries, q and o) over whole-step device time, inputs
resident in HBM, L2 flushed between steps (a 320 MB write, then a 256 MB
read, so no input line is in L2 and the flush's own dirty lines are not
written back inside the timed region). The other named workloads
(chunked-prefill extend in TFLOP/s, long-context and radix-shared decode in
GB/s, the tiny decode in microseconds) are measured in the same run and
reported under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

--impl reference times the fp64 CPU oracle (the correctness reference) on a
bounded sample of the same workload on this machine's host cores. With
torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling); rank 0 prints the one JSON line.
"""
from __future__ import annotations

import argparse
import copy
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_attention_out_gb300 import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 320 << 20  # > 2x the 129 MB L2
L2_CLEAN_BYTES = 256 << 20  # read after the flush write (see L2Flush)
CSRC = os.path.join(ROOT, "paged_kv_attention_out_gb300", "csrc")

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per call, summed
# over the call's launches, from one ncu capture of each call. Each entry
# holds the SHA-256 of the kernel sources it was taken on; the bench reports
# it only while those sources are unchanged (else null).
MEASURED_TRAFFIC = {
    # decode_kernel + decode_merge_kernel, Llama-3-8B-shaped decode
    "decode": {"sources": ['decode.cu', 'decode_common.cuh', 'pkv_common.cuh'],
               "sha256": "1946f3ac4ab631093fbc25b82b65651fec5fd69a755e14f8055eb573eab8ac9f",
               "bytes": 625499392},
    # extend_gather_kernel + extend_tc_persistent_kernel, chunked-prefill extend
    "extend": {"sources": ['extend.cu', 'tc_common.cuh', 'pkv_common.cuh'],
               "sha256": "603ff433c0bcf92b10475c79a715087cc51e548d1834ee93f00ce253edbfd45c",
               "bytes": 489539904},
    # cascade_prefix_kernel + decode_kernel (suffix) + decode_merge_narrow_kernel,
    # radix-shared decode through cascade decode
    "cascade": {"sources": ['cascade.cu', 'decode.cu', 'decode_common.cuh', 'tc_common.cuh', 'pkv_common.cuh'],
                "sha256": "3e5d0f458ab7b66880974acc5521cb2eb68108f6736d1a82d0963b3ff761b592",
                "bytes": 372296352},
}


def sources_sha256(names) -> str:
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(CSRC, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kind: str, override=None):
    """Captured DRAM bytes per call for `kind`, or None if the kernels changed since."""
    if override is not None:
        return override
    e = MEASURED_TRAFFIC[kind]
    if e["sha256"] is None or sources_sha256(e["sources"]) != e["sha256"]:
        return None
    return e["bytes"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "paged decode attn KV GB/s"


# ---------------------------------------------------------------------------
# ranks (replicas only: the path has no exchange step)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def aggregate_ranks(elapsed_ms: float, units: float, world: int):
    """Max step time and total units over ranks (control-plane collectives only)."""
    if world <= 1:
        return elapsed_ms, units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def decode_bytes(case: W.Case, unique: bool = False) -> int:
    """Bytes decode attention must move: K and V of every key (all kv heads),
    the page-table entries and seq_lens it reads, q in and o + lse out."""
    kv_row = 2 * case.Hkv * case.D * 2  # K + V of one token, bytes
    keys = len(case.referenced_slots()) if unique else int(case.seq_lens.sum())
    table = int(((case.seq_lens + case.P - 1) // case.P).sum()) * 4 + case.B * 4
    qo = 2 * case.B * case.Hq * case.D * 2 + case.B * case.Hq * 4
    return keys * kv_row + table + qo


def store_bytes(case: W.Case) -> int:
    return case.n_new * (2 * case.Hkv * case.D * 2 * 2 + 4)


def extend_flops(case: W.Case) -> float:
    """4 D Hq sum_r [c_r p_r + c_r (c_r + 1) / 2]: QK^T and PV over exactly the
    (query, key) pairs the causal rule allows."""
    c = np.diff(case.qo_indptr).astype(np.float64)
    p = case.seq_lens.astype(np.float64) - c
    return 4.0 * case.D * case.Hq * float((c * p + c * (c + 1) / 2).sum())


def extend_bytes(case: W.Case) -> int:
    kv = int(case.seq_lens.sum()) * 2 * case.Hkv * case.D * 2
    qo = 2 * case.total_q * case.Hq * case.D * 2 + case.total_q * case.Hq * 4
    return kv + qo


# ---------------------------------------------------------------------------
# peaks and clocks
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples, each stamped on arrival."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int | None, interval_ms: int = 50):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               f"--loop-ms={interval_ms}"]
        if gpu_index is not None:
            cmd.insert(1, f"--id={gpu_index}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1 and len(s) >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def gpu_index_for(dev: int):
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        out = subprocess.run(["nvidia-smi", "--query-gpu=index,uuid", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout
        for line in out.strip().splitlines():
            idx, u = [x.strip() for x in line.split(",")]
            if uuid.replace("GPU-", "") in u:
                return int(idx)
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# the pkv arm
# ---------------------------------------------------------------------------

class Workload:
    """Device-resident inputs of one case plus the calls of one step."""

    def __init__(self, case: W.Case, dev, pool_layers: int | None = None):
        import paged_kv_attention_out_gb300 as pkv
        self.pkv = pkv
        self.case = case
        if pool_layers is not None and pool_layers != case.L:
            case.L = pool_layers
            case.layer = min(case.layer, pool_layers - 1)
        self.pool = case.make_pool(dev, poison=False)
        self.k, self.v = case.new_kv(dev)
        self.q = case.q(dev)
        self.t = case.device_tables(dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=dev)
        self.hint = case.max_seq_len
        self.total_keys = int(case.seq_lens.sum())  # the scheduler knows it on the host
        self.ws = None
        if case.kind == "decode":
            n = pkv.pkv_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, self.hint)
        else:
            n = pkv.pkv_extend_workspace_size(case.B, case.Hkv, case.D, self.hint,
                                              self.total_keys)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        self.launches_per_step = None

    def store(self):
        c = self.case
        self.pkv.pkv_kv_store(self.pool, c.layer, self.k, self.v, self.t["out_loc"])

    def attention(self):
        c, t = self.case, self.t
        if c.kind == "decode":
            self.pkv.pkv_paged_decode_attn(self.pool, c.layer, self.q, self.o, self.lse,
                                           t["page_table"], t["seq_lens"], c.scale, self.hint,
                                           self.ws, table_idx=t.get("table_idx"))
        else:
            self.pkv.pkv_paged_extend_attn(self.pool, c.layer, self.q, t["qo_indptr"], self.o,
                                           self.lse, t["page_table"], t["seq_lens"], c.scale,
                                           self.hint, self.ws, table_idx=t.get("table_idx"),
                                           max_total_keys_hint=self.total_keys)

    def kernels_per_step(self) -> int:
        c = self.case
        if c.kind == "extend":
            return 3  # store, gather, attention
        from paged_kv_attention_out_gb300.binding import load
        split = load().pkv_decode_workspace_size(
            c.B, c.Hq, c.Hkv, c.D, self.hint) > 0
        return 3 if split else 2


class FusedDecodeWorkload(Workload):
    """The decode step through pkv_paged_decode_attn_store: store_kv of the new
    tokens fused into the decode launch (one launch fewer per step). Shares
    the device tensors of an existing decode Workload."""

    def __init__(self, base: Workload):  # noqa: super().__init__ would rebuild the inputs
        self.__dict__.update(base.__dict__)

    def store(self):
        pass

    def attention(self):
        c, t = self.case, self.t
        self.pkv.pkv_paged_decode_attn_store(self.pool, c.layer, self.q, self.k, self.v, self.o,
                                             self.lse, t["page_table"], t["seq_lens"], c.scale,
                                             self.hint, self.ws, table_idx=t.get("table_idx"))

    def kernels_per_step(self) -> int:
        return super().kernels_per_step() - 1


class FusedExtendWorkload(Workload):
    """The extend step through pkv_paged_extend_attn_store: store_kv of the
    chunk's tokens fused into the gather launch. Shares the device tensors of
    an existing extend Workload."""

    def __init__(self, base: Workload):  # noqa: super().__init__ would rebuild the inputs
        self.__dict__.update(base.__dict__)

    def store(self):
        pass

    def attention(self):
        c, t = self.case, self.t
        self.pkv.pkv_paged_extend_attn_store(self.pool, c.layer, self.q, self.k, self.v,
                                             t["qo_indptr"], self.o, self.lse, t["page_table"],
                                             t["seq_lens"], c.scale, self.hint, self.ws,
                                             table_idx=t.get("table_idx"),
                                             max_total_keys_hint=self.total_keys)

    def kernels_per_step(self) -> int:
        return 2  # gather (with the store), attention


class CascadeWorkload(Workload):
    """The radix-shared case through pkv_paged_cascade_decode_attn: each
    group's prefix attended once (tensor cores), merged with every member's
    suffix decode."""

    def __init__(self, case: W.Case, dev):
        super().__init__(case, dev)
        self.ct = {n: torch.as_tensor(a, dtype=torch.int32, device=dev)
                   for n, a in W.cascade_tables(case).items()}
        self.pmax = max(int(self.ct["prefix_lens"].max()), 1)
        self.smax = int(self.ct["seq_lens"].max())
        G = self.ct["prefix_lens"].shape[0]
        n = self.pkv.pkv_cascade_workspace_size(case.B, case.Hq, case.Hkv, case.D, G, self.pmax,
                                                self.smax)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    def attention(self):
        c, ct = self.case, self.ct
        self.pkv.pkv_paged_cascade_decode_attn(
            self.pool, c.layer, self.q, self.o, self.lse, ct["prefix_page_table"],
            ct["prefix_lens"], ct["member_indptr"], ct["members"], ct["page_table"],
            ct["seq_lens"], c.scale, self.pmax, self.smax, self.ws)

    def kernels_per_step(self) -> int:
        return 5  # store, suffix decode, prefix gather, prefix attention, merge


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (no input line
    survives), then read another buffer larger than L2, so the write's own
    dirty lines are written back before the timed region instead of inside
    it; a step then starts with L2 holding clean, unrelated lines (as after
    the weight-reading GEMMs of a model layer). write_only=True keeps the
    plain write flush, reported beside it for comparison."""

    def __init__(self, dev, write_only: bool = False):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = None if write_only else torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32,
                                                    device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        if self.r is not None:
            torch.sum(self.r, dim=(0,), out=self.acc)


def time_steps(wl: Workload, steps: int, warmup: int, flush: L2Flush):
    """Per-step CUDA-event times (ms) of store + attention, and of attention alone."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        wl.store()
        wl.attention()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        wl.store()
        ev[i][1].record(stream)
        wl.attention()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step = [e[0].elapsed_time(e[2]) for e in ev]
    attn = [e[1].elapsed_time(e[2]) for e in ev]
    return step, attn


def _staging(tensors: dict, device):
    """One pinned host byte buffer and one device byte buffer holding every
    tensor at a 256-byte aligned offset, plus dtype/shape views of the device
    buffer (so a step moves its inputs, or its results, in one copy)."""
    offs, n = {}, 0
    for name, x in tensors.items():
        offs[name] = n
        n += -(-x.numel() * x.element_size() // 256) * 256
    host = torch.empty(max(n, 256), dtype=torch.uint8).pin_memory()
    devb = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    views = {}
    for name, x in tensors.items():
        nb = x.numel() * x.element_size()
        host[offs[name]:offs[name] + nb].copy_(x.detach().contiguous().reshape(-1)
                                               .view(torch.uint8).cpu())
        views[name] = devb[offs[name]:offs[name] + nb].view(x.dtype).view(x.shape)
    return host, devb, views


def time_e2e(wl: Workload, steps: int, warmup: int, flush: L2Flush):
    """Same step through the public API from pinned host memory: H2D of the
    step's inputs (q, new k/v, out_loc, page_table, seq_lens), the calls, and
    D2H of the result (o, lse), all inside the timed region. The inputs sit
    in one pinned staging buffer and travel in one copy; o and lse come back
    in one copy (the calls read and write views of the device staging
    buffers)."""
    ins = {"q": wl.q, "k": wl.k, "v": wl.v, **wl.t}
    in_h, in_d, iv = _staging(ins, wl.q.device)
    out_h, out_d, ov = _staging({"o": wl.o, "lse": wl.lse}, wl.q.device)
    ew = copy.copy(wl)
    ew.q, ew.k, ew.v = iv["q"], iv["k"], iv["v"]
    ew.t = {n: iv[n] for n in wl.t}
    ew.o, ew.lse = ov["o"], ov["lse"]
    h2d = in_h.numel()
    d2h = out_h.numel()
    stream = torch.cuda.current_stream()

    def one():
        in_d.copy_(in_h, non_blocking=True)
        ew.store()
        ew.attention()
        out_h.copy_(out_d, non_blocking=True)

    for _ in range(warmup):
        flush()
        one()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        one()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    return ms, h2d, d2h


def roofline(kind: str, work: float, ms: float, peaks, peak_src: str, traffic=None,
             sustained: bool = False):
    if kind == "hbm":
        achieved = work / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    else:
        achieved = work / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        unit = "TFLOP/s"
    return {"bound": kind, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{peak_src} ({'sustained' if sustained else 'burst'})"
            if kind == "tensor" else peak_src}


def cpu_baseline(case: W.Case, budget_s: float, every: int = 4):
    """The oracle (as it stands) on a sample of the workload: every `every`-th
    request, store_kv + decode, repeated until `budget_s` of CPU time."""
    import oracle
    req = list(range(0, case.B, every))
    sub = case.compact(req)
    pool = W.bf16_bits(sub.make_pool("cpu", poison=True)).reshape(sub.pool_shape).copy()
    k, v = sub.new_kv("cpu")
    kb, vb, qb = W.bf16_bits(k), W.bf16_bits(v), W.bf16_bits(sub.q("cpu"))
    threads = oracle.max_threads()
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.kv_store(pool, 0, kb, vb, sub.out_loc)
        oracle.decode_attn(pool, 0, qb, sub.page_table, sub.seq_lens, sub.scale)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = decode_bytes(sub) * reps / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(req)} of {case.B} requests (every {every}th), store_kv + decode, "
                      f"{reps} repetitions in {el:.1f} s, fp64"}, el / reps, decode_bytes(sub)


def run_pkv(args):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_attention_out_gb300 as pkv
    pkv.pkv_init()
    peaks, peak_src = load_peaks()
    flush = L2Flush(dev)
    if args.only not in (None, "llama3-8b-decode"):
        # one named workload alone (used for profiling): prints its JSON object
        if rank == 0:
            print(json.dumps(other_workloads(args, dev, peaks, peak_src, flush, args.only)),
                  flush=True)
        return

    # ---- main workload: Llama-3-8B-shaped decode -----------------------------
    case = W.llama8b_decode(args.seed + rank)
    wl_sep = Workload(case, dev, pool_layers=args.pool_layers)
    # the step as two calls (store_kv, then decode): the decode call alone is
    # the roofline's timed kernel pair
    sep_step_ms, sep_attn_ms = time_steps(wl_sep, max(3, min(args.steps, 200)), args.warmup, flush)
    # the step as timed: store_kv fused into the decode launch
    wl = FusedDecodeWorkload(wl_sep)
    sampler = ClockSampler(gpu_index_for(dev.index)) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    t_start = time.monotonic()
    step_ms, attn_ms = time_steps(wl, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    barrier(world)
    t_end = time.monotonic()
    # keep the GPU under the same load until clocks have been sampled for ~1.5 s
    while time.monotonic() - t_start < 1.5 and sampler is not None:
        time_steps(wl, 50, 0, flush)
    t_load_end = time.monotonic()
    if sampler:
        sampler.stop()
    units = decode_bytes(case)
    total_ms = float(sum(step_ms))
    max_ms, all_units = aggregate_ranks(total_ms, units * args.steps, world)
    value = all_units / (max_ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_e2e(wl, max(3, min(args.steps, 200)), args.warmup, flush)
    # the same step after the plain write flush (its dirty lines written back
    # inside the timed region), for comparison
    wo_ms, _ = time_steps(wl, max(3, min(args.steps, 200)), args.warmup,
                          L2Flush(dev, write_only=True))
    e2e_value = units / (statistics.mean(e2e_ms) * 1e-3) / 1e9
    kernels = wl.kernels_per_step()
    sep_attn = statistics.mean(sep_attn_ms)
    main = {
        "roofline": roofline("hbm", units, sep_attn, peaks, peak_src),
        "fused_step_ms": round(statistics.mean(step_ms), 5),
        "attn_ms": round(sep_attn, 5),
        "store_ms": round(statistics.mean(s - a for s, a in zip(sep_step_ms, sep_attn_ms)), 5),
        "unfused_step_ms": round(statistics.mean(sep_step_ms), 5),
    }
    main["roofline"]["kernel"] = ("pkv_paged_decode_attn: decode_kernel + decode_merge_kernel "
                                  "(both launches inside the timed duration)")
    main["roofline"]["traffic"] = measured_traffic("decode", args.decode_traffic)
    del wl, wl_sep
    torch.cuda.empty_cache()

    clocks = sampler.summary(t_start, t_load_end) if sampler else None
    if clocks is not None:
        clocks["window"] = ("timed region" if t_end - t_start >= 1.0 else
                            "timed region + identical untimed steps to 1.5 s")

    # ---- the other named workloads -----------------------------------------
    workloads = {}
    if rank == 0 and not args.main_only:
        workloads = other_workloads(args, dev, peaks, peak_src, flush)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu, _, _ = cpu_baseline(case, args.cpu_budget)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based N(0,1) bf16 values and seeded page tables)",
        "config": {"workload": "llama3-8b-decode", "batch": case.B, "q_heads": case.Hq,
                   "kv_heads": case.Hkv, "head_dim": case.D, "page_size": case.P,
                   "seq_len": "uniform [512, 4096]", "sum_seq_len": int(case.seq_lens.sum()),
                   "pool": f"{case.NP} slots x {case.L} layers", "seed": args.seed,
                   "step": ("kv_store fused into split-KV decode (pkv_paged_decode_attn_store) "
                            "+ split merge"),
                   "algorithmic_bytes_per_step": units,
                   "l2": ("flushed between steps: a 320 MB write, then a 256 MB read so the "
                          "write's dirty lines are written back before the timed region"),
                   "parallelism": f"replicas x{world}"},
        "roofline": main["roofline"],
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": round(statistics.mean(e2e_ms), 5)},
        "gpu_launches": kernels * args.steps,
        "clocks": clocks,
        "detail": {"fused_step_ms": main["fused_step_ms"],
                   "unfused_step_ms": main["unfused_step_ms"],
                   "decode_call_ms": main["attn_ms"], "kv_store_ms": main["store_ms"],
                   "kernels_per_step": kernels,
                   "fused_step_ms_write_only_flush": round(statistics.mean(wo_ms), 5),
                   "value_write_only_flush": round(units / (statistics.mean(wo_ms) * 1e-3) / 1e9,
                                                   2)},
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _measure(wl: Workload, steps: int, warmup: int, flush):
    step_ms, attn_ms = time_steps(wl, steps, warmup, flush)
    return statistics.mean(step_ms), statistics.mean(attn_ms)


def other_workloads(args, dev, peaks, peak_src, flush, only=None):
    out = {}
    steps = max(5, min(args.steps, 100)) if only is None else args.steps
    warm = max(3, args.warmup)
    want = (lambda name: only is None or only == name)
    if want("chunked-prefill-extend"):
        out.update(_extend_workload(args, dev, peaks, peak_src, flush, steps, warm))
    if want("long-context-decode"):
        out.update(_long_workload(args, dev, peaks, peak_src, flush, steps, warm))
    if want("radix-shared-decode"):
        out.update(_radix_workload(args, dev, peaks, peak_src, flush, steps, warm))
    if want("tiny-decode"):
        out.update(_tiny_workload(args, dev, flush, steps, warm))
    if want("decode-graph-batches"):
        out.update(_graph_batches_workload(args, dev, flush, steps, warm))
    return out


def _extend_workload(args, dev, peaks, peak_src, flush, steps, warm):
    out = {}
    case = W.chunked_prefill_extend(args.seed)
    wl = Workload(case, dev)
    st, at = _measure(wl, steps, warm, flush)
    _, ft = _measure(FusedExtendWorkload(wl), steps, warm, flush)
    fl = extend_flops(case)
    out["chunked-prefill-extend"] = {
        "metric": "extend attn TFLOP/s", "value": round(fl / (at * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "ms_attention": round(at, 4), "ms_step_with_store": round(st, 4),
        "ms_step_fused_store": round(ft, 4),
        "flops": fl, "tokens_per_s": round(case.total_q / (min(st, ft) * 1e-3), 1),
        "roofline": {**roofline("tensor", fl, at, peaks, peak_src),
                     "kernel": ("pkv_paged_extend_attn: extend_gather_kernel + extend_tc_persistent_kernel "
                                "(both launches inside the timed duration)"),
                     "traffic": measured_traffic("extend", args.extend_traffic),
                     "algorithmic_bytes": extend_bytes(case)}}
    del wl
    torch.cuda.empty_cache()
    return out


def _long_workload(args, dev, peaks, peak_src, flush, steps, warm):
    out = {}
    case = W.long_context_decode(args.seed)
    wl = Workload(case, dev)
    st, at = _measure(wl, steps, warm, flush)
    by = decode_bytes(case)
    out["long-context-decode"] = {
        "metric": METRIC, "value": round(by / (at * 1e-3) / 1e9, 2), "unit": "GB/s",
        "ms_attention": round(at, 4), "ms_step_with_store": round(st, 4),
        "algorithmic_bytes": by, "tokens_per_s": round(case.B / (st * 1e-3), 1),
        "roofline": {**roofline("hbm", by, at, peaks, peak_src),
                     "kernel": "decode_kernel + decode_merge_kernel"}}
    del wl
    torch.cuda.empty_cache()
    return out


def _radix_workload(args, dev, peaks, peak_src, flush, steps, warm):
    """Radix-shared-prefix decode: unique bytes (roofline) and logical bytes."""
    out = {}
    case = W.radix_shared_decode(args.seed)
    wl = Workload(case, dev)
    st, at = _measure(wl, steps, warm, flush)
    uniq, logical = decode_bytes(case, unique=True), decode_bytes(case)
    out["radix-shared-decode"] = {
        "metric": METRIC + " (unique bytes)", "value": round(uniq / (at * 1e-3) / 1e9, 2),
        "unit": "GB/s", "logical_gbs": round(logical / (at * 1e-3) / 1e9, 2),
        "ms_attention": round(at, 4), "ms_step_with_store": round(st, 4),
        "unique_bytes": uniq, "logical_bytes": logical,
        "roofline": {**roofline("hbm", uniq, at, peaks, peak_src),
                     "kernel": "decode_kernel + decode_merge_kernel"}}
    del wl
    torch.cuda.empty_cache()
    wl = CascadeWorkload(case, dev)
    st, at = _measure(wl, steps, warm, flush)
    out["radix-shared-decode-cascade"] = {
        "metric": METRIC + " (unique bytes)", "value": round(uniq / (at * 1e-3) / 1e9, 2),
        "unit": "GB/s", "logical_gbs": round(logical / (at * 1e-3) / 1e9, 2),
        "ms_attention": round(at, 4), "ms_step_with_store": round(st, 4),
        "unique_bytes": uniq, "logical_bytes": logical,
        "roofline": {**roofline("hbm", uniq, at, peaks, peak_src),
                     "kernel": ("pkv_paged_cascade_decode_attn: cascade_prefix_kernel + "
                                "suffix decode_kernel + decode_merge_narrow_kernel, all inside "
                                "the timed duration"),
                     "traffic": measured_traffic("cascade")}}
    del wl
    torch.cuda.empty_cache()
    return out


def _tiny_workload(args, dev, flush, steps, warm):
    out = {}
    case = W.tiny_decode(args.seed)
    wl = Workload(case, dev)
    st, at = _measure(wl, steps, warm, flush)
    wf = FusedDecodeWorkload(wl)
    fst, _ = _measure(wf, steps, warm, flush)
    out["tiny-decode"] = {"metric": "step latency", "value": round(fst * 1e3, 2), "unit": "us",
                          "step": "store_kv fused into decode (one launch)",
                          "unfused_step_us": round(st * 1e3, 2),
                          "attention_us": round(at * 1e3, 2),
                          "graph_replay_us": round(_graph_replay_us(wf, steps, warm), 2),
                          "unfused_graph_replay_us": round(_graph_replay_us(wl, steps, warm), 2)}
    del wf
    del wl
    torch.cuda.empty_cache()
    return out


def _graph_batches_workload(args, dev, flush, steps, warm):
    """Small-batch decode latency through the graph harness: the fused
    store_kv + decode step of the Llama-3-8B-shaped workload captured at
    batch sizes 1, 2, 4, ..., 64 (DecodeGraphRunner) and replayed at each
    size on that many of its requests; per size the replay time (L2 flushed
    before each replay, CUDA events around the replay alone) and the same
    step as an eager call. The pool holds one layer (the attended data are
    the same as in the 32-layer pool)."""
    from paged_kv_attention_out_gb300.graph_runner import DecodeGraphRunner
    import paged_kv_attention_out_gb300 as pkv
    case = W.llama8b_decode(args.seed)
    case.L, case.layer = 1, 0
    pool = case.make_pool(dev, poison=False)
    k, v = case.new_kv(dev)
    q = case.q(dev)
    t = case.device_tables(dev)
    runner = DecodeGraphRunner(pool, 0, case.Hq, case.B, t["page_table"].shape[1],
                               case.max_seq_len, case.scale)
    stream = torch.cuda.current_stream()
    reps = max(10, min(steps, 50))
    rows = {"batch": [], "replay_us": [], "eager_us": [], "replay_gbs": []}
    for n in runner.sizes:
        runner.stage(q[:n], k[:n], v[:n], t["page_table"][:n], t["seq_lens"][:n])
        ws = torch.empty(max(pkv.pkv_decode_workspace_size(n, case.Hq, case.Hkv, case.D,
                                                           case.max_seq_len), 256),
                         dtype=torch.uint8, device=dev)
        o = torch.empty_like(q[:n])
        lse = torch.empty(n, case.Hq, dtype=torch.float32, device=dev)

        def eager():
            pkv.pkv_paged_decode_attn_store(pool, 0, q[:n], k[:n], v[:n], o, lse,
                                            t["page_table"][:n], t["seq_lens"][:n],
                                            case.scale, case.max_seq_len, ws)

        def replay():
            runner.replay(n)

        times = {}
        for name, fn in (("replay", replay), ("eager", eager)):
            for _ in range(warm):
                flush()
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for e0, e1 in ev:
                flush()
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize()
            times[name] = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
        by = decode_bytes(case.compact(list(range(n))))
        rows["batch"].append(n)
        rows["replay_us"].append(round(times["replay"], 2))
        rows["eager_us"].append(round(times["eager"], 2))
        rows["replay_gbs"].append(round(by / (times["replay"] * 1e-6) / 1e9, 1))
    del runner, pool
    torch.cuda.empty_cache()
    return {"decode-graph-batches": {
        "metric": "decode step latency (graph replay)", "unit": "us",
        "step": "store_kv fused into decode + split merge, Llama-3-8B-shaped requests "
                "(first n of the 64), replayed from the graph captured at n",
        **rows}}


def _graph_replay_us(wl: Workload, steps: int, warm: int) -> float:
    """Mean device time of one store_kv + attention step captured in a CUDA
    graph and replayed back to back (the serving engine replays decode steps
    from graphs): launch overhead out of the picture."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        wl.store()
        wl.attention()
        with torch.cuda.graph(g, stream=s):
            wl.store()
            wl.attention()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    reps = max(steps, 20)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


# ---------------------------------------------------------------------------
# the reference arm: the fp64 CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    case = W.llama8b_decode(args.seed)
    every = 8
    req = list(range(0, case.B, every))
    sub = case.compact(req)
    pool = W.bf16_bits(sub.make_pool("cpu", poison=True)).reshape(sub.pool_shape).copy()
    k, v = sub.new_kv("cpu")
    kb, vb, qb = W.bf16_bits(k), W.bf16_bits(v), W.bf16_bits(sub.q("cpu"))

    def step():
        oracle.kv_store(pool, 0, kb, vb, sub.out_loc)
        oracle.decode_attn(pool, 0, qb, sub.page_table, sub.seq_lens, sub.scale)

    for _ in range(args.warmup):
        step()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        ts.append(time.perf_counter() - t0)
    units = decode_bytes(sub)
    value = units / statistics.mean(ts) / 1e9
    sample = (f"{len(req)} of {case.B} requests (every {every}th) per step, "
              f"store_kv + decode in fp64")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(ts) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded generator as the pkv arm)",
        "config": {"workload": "llama3-8b-decode", "batch": case.B, "q_heads": case.Hq,
                   "kv_heads": case.Hkv, "head_dim": case.D, "page_size": case.P,
                   "seed": args.seed, "sample": sample, "algorithmic_bytes_per_step": units},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                         "cores": oracle.max_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--main-only", action="store_true",
                    help="skip the other named workloads")
    ap.add_argument("--only", choices=["llama3-8b-decode", "chunked-prefill-extend",
                                       "long-context-decode", "radix-shared-decode",
                                       "tiny-decode", "decode-graph-batches"], default=None,
                    help="run one named workload alone and print its JSON object "
                         "(for profiling); llama3-8b-decode = the main line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--pool-layers", type=int, default=None,
                    help="allocate the pool with this many layers (same attended data)")
    ap.add_argument("--decode-traffic", type=float, default=None,
                    help="ncu dram bytes per decode call, from a capture of this kernel")
    ap.add_argument("--extend-traffic", type=float, default=None,
                    help="ncu dram bytes per extend call, from a capture of this kernel")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def check_gpus(args, world: int):
    """--gpus must match the number of ranks actually running: one rank per
    GPU is launched by torchrun, so `--gpus N` without it (or with another
    count) would measure a different number of GPUs than it reports."""
    if args.gpus != world:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but {world} rank(s) are running "
                         f"(WORLD_SIZE={world}); launch N > 1 with torchrun "
                         f"--nproc-per-node N ... bench.py --gpus N")


def main(argv=None):
    args = parse_args(argv)
    check_gpus(args, dist_env()[1])
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
