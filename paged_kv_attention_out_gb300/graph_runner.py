"""CUDA-graph replay of the fused decode step at padded batch sizes.

The serving engine replays decode steps from CUDA graphs ("Code Notes:
mini-sglang", Engine Layer table, GraphRunner row): graphs are captured once
for a ladder of batch sizes (1, 2, 4, 8, ...) and each step replays the
smallest captured graph whose size is at least the step's batch, the rows
past the real batch being padding.

DecodeGraphRunner does that for one decode step, store_kv fused into split-KV
decode attention (pkv_paged_decode_attn_store) plus the split merge, on one
layer of a caller-owned pool. It owns static device buffers sized for the
largest batch (q, the new K/V rows, page-table rows, seq_lens, o, lse and the
split workspace); a graph captured at size n reads and writes their first n
rows. A padding row has seq_len 0, which the decode call defines as "store
nothing, o = 0, lse = -inf", so padding never touches the pool and never
reads a page-table entry. The replay launches exactly the kernels the eager
call launches; the runner itself only fills its static buffers (plain copies
of the caller's tensors, or the caller writes the views it hands out).
"""
from __future__ import annotations

import torch

from . import binding as B


def default_sizes(max_batch: int) -> list[int]:
    """1, 2, 4, ... up to and including max_batch."""
    sizes, n = [], 1
    while n < max_batch:
        sizes.append(n)
        n *= 2
    sizes.append(max_batch)
    return sizes


class DecodeGraphRunner:
    """Fused store_kv + decode steps replayed from CUDA graphs.

    pool: the (2, layers, pages, page_size, Hkv, D) bf16 pool (caller-owned;
        the graphs hold its address, so it must outlive the runner).
    table_stride: page-table entries per row (the static page table is
        [max_batch, table_stride] int32).
    max_seq_len_hint: a bound on every seq_len of a step; it sets the split
        plan each graph is captured with (a longer row is still correct).
    sizes: the captured batch sizes (default 1, 2, 4, ..., max_batch).
    """

    def __init__(self, pool: torch.Tensor, layer: int, num_q_heads: int, max_batch: int,
                 table_stride: int, max_seq_len_hint: int, scale: float, sizes=None):
        if max_batch < 1 or table_stride < 1:
            raise ValueError("max_batch and table_stride must be positive")
        self.pool = pool
        self.layer = int(layer)
        self.scale = float(scale)
        self.hint = int(max_seq_len_hint)
        _, _, _, _, hkv, d = pool.shape
        self.hq, self.hkv, self.d = int(num_q_heads), int(hkv), int(d)
        self.sizes = sorted(set(int(s) for s in (sizes or default_sizes(max_batch))))
        if self.sizes[0] < 1 or self.sizes[-1] != max_batch:
            raise ValueError("sizes must be positive and end at max_batch")
        dev = pool.device
        self.max_batch = int(max_batch)
        self.q = torch.zeros(max_batch, self.hq, d, dtype=torch.bfloat16, device=dev)
        self.k_new = torch.zeros(max_batch, self.hkv, d, dtype=torch.bfloat16, device=dev)
        self.v_new = torch.zeros_like(self.k_new)
        self.page_table = torch.zeros(max_batch, table_stride, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        self.o = torch.zeros_like(self.q)
        self.lse = torch.zeros(max_batch, self.hq, dtype=torch.float32, device=dev)
        ws = max(B.pkv_decode_workspace_size(n, self.hq, self.hkv, self.d, self.hint)
                 for n in self.sizes)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self._capture_all()

    # ---- one step of n rows (eager form; what each graph holds) ------------
    def _step(self, n: int) -> None:
        B.pkv_paged_decode_attn_store(
            self.pool, self.layer, self.q[:n], self.k_new[:n], self.v_new[:n], self.o[:n],
            self.lse[:n], self.page_table[:n], self.seq_lens[:n], self.scale, self.hint,
            self.workspace)

    def _capture_all(self) -> None:
        # Rows are padding (seq_len 0) while capturing: a warm-up run sets the
        # library's per-device state up outside any capture, and the captured
        # launches read whatever the static buffers hold at replay time.
        self.seq_lens.zero_()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for n in self.sizes:
                self._step(n)
            for n in self.sizes:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    self._step(n)
                self.graphs[n] = g
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()

    # ---- runtime -----------------------------------------------------------
    def padded_size(self, batch: int) -> int:
        """The smallest captured size >= batch."""
        for n in self.sizes:
            if n >= batch:
                return n
        raise ValueError(f"batch {batch} exceeds the largest captured size {self.sizes[-1]}")

    def stage(self, q, k_new, v_new, page_table, seq_lens) -> int:
        """Copies one step's inputs (batch rows each; page_table [batch, <=
        table_stride]) into the static buffers and marks the rows up to the
        padded size as padding. Returns the padded size."""
        b = int(seq_lens.shape[0])
        n = self.padded_size(b)
        if b == 0:
            return n
        self.q[:b].copy_(q)
        self.k_new[:b].copy_(k_new)
        self.v_new[:b].copy_(v_new)
        self.page_table[:b, :page_table.shape[1]].copy_(page_table)
        self.seq_lens[:b].copy_(seq_lens)
        self.seq_lens[b:n].zero_()
        return n

    def replay(self, batch: int):
        """Replays the graph of padded_size(batch) on the staged inputs;
        returns views (o, lse) of the batch's rows."""
        n = self.padded_size(batch)
        self.graphs[n].replay()
        return self.o[:batch], self.lse[:batch]

    def run(self, q, k_new, v_new, page_table, seq_lens):
        """stage() then replay(): one decode step of seq_lens.shape[0] rows."""
        b = int(seq_lens.shape[0])
        self.stage(q, k_new, v_new, page_table, seq_lens)
        return self.replay(b)
