"""Seeded synthetic inputs for the paged KV-cache attention step.

This module is shared by the CUDA path (tests, benchmark) and by the oracle's
tests, and it holds none of the attention arithmetic. It does two things:

* draws numbers: a counter-based generator gives every tensor element a bf16
  value that is a pure function of (seed, stream, row-major position), so the
  same element has the same value whether it is produced on the host or on a
  GPU, and any part of a 50 GB pool can be produced on its own;
* builds the allocator's tables the way a serving scheduler would (page
  rows, out_loc slots, qo_indptr), following the recipes of the five named
  workloads plus a generic builder for sweeps.

Values: the 32-bit counter hash below is a mixer of the "lowbias32" form
published by C. Wellons (hash-prospector); its top 16 bits index a table of
the 65,536 standard-normal quantiles Phi^-1((i + 0.5) / 65536) rounded to
bf16. So values follow N(0, 1) (truncated at about 4.3 sigma) on a bf16 grid.
All integer work is done in int64 without overflow, which makes it exact and
identical on every device.

Layout facts used (page "Code Notes: mini-sglang", Engine Layer table,
BaseKVCachePool row, and Scheduler Layer table): the pool is
(2, layers, pages, page_size, kv_heads, head_dim); a slot is
page * page_size + offset; a page_table row lists the pages of one request.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

M32 = 0xFFFFFFFF

# Stream identifiers: each tensor of a case draws from its own stream.
STREAM_POOL = 0x1F3A
STREAM_Q = 0x2B71
STREAM_K_NEW = 0x3C55
STREAM_V_NEW = 0x4D09
STREAM_AUX = 0x5E83


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for 0 <= x < 2**32, exact in int64 (no overflow)."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _mix32_int(x: int) -> int:
    return int(_mix32(torch.tensor([x & M32], dtype=torch.int64))[0])


def _stream_keys(seed: int, stream: int) -> tuple[int, int]:
    s = _mix32_int((seed & M32) ^ _mix32_int((seed >> 32) & M32))
    k1 = _mix32_int(s ^ stream)
    k2 = _mix32_int(k1 ^ 0x68E31DA4)
    return k1, k2


_TABLES: dict[str, torch.Tensor] = {}


def _normal_table(device: torch.device) -> torch.Tensor:
    key = str(device)
    t = _TABLES.get(key)
    if t is None:
        cpu = _TABLES.get("cpu")
        if cpu is None:
            u = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
            cpu = torch.special.ndtri(u).to(torch.bfloat16)
            _TABLES["cpu"] = cpu
        t = cpu.to(device)
        _TABLES[key] = t
    return t


def normal_bf16(seed: int, stream: int, index: torch.Tensor) -> torch.Tensor:
    """bf16 N(0,1) value of every counter in `index` (int64, >= 0), same device."""
    k1, k2 = _stream_keys(seed, stream)
    idx = index.to(torch.int64)
    lo = idx & M32
    hi = idx >> 32
    h = _mix32(lo ^ k1)
    h = _mix32(h ^ _mix32((hi + k2) & M32))
    return _normal_table(idx.device)[h >> 16]


def fill_normal_(t: torch.Tensor, seed: int, stream: int, base: int = 0,
                 chunk: int = 1 << 24) -> torch.Tensor:
    """t.view(-1)[i] = normal_bf16(seed, stream, base + i); t must be contiguous bf16."""
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError("fill_normal_ wants a contiguous bf16 tensor")
    flat = t.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        idx = torch.arange(base + s, base + e, dtype=torch.int64, device=t.device)
        flat[s:e] = normal_bf16(seed, stream, idx)
    return t


def normal_tensor(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    t = torch.empty(tuple(shape), dtype=torch.bfloat16, device=device)
    return fill_normal_(t, seed, stream)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy uint16 view of the bits of a bf16 tensor."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Cases: shapes, tables and the value recipe of one workload
# --------------------------------------------------------------------------

@dataclass
class Case:
    """One seeded workload. Tables are host numpy int32 arrays.

    kind        "decode" (one new query token per request) or "extend".
    token_slots token_slots[b] = flat slots of request b's keys 0..seq_len-1,
                as the allocator handed them out.
    out_loc     slots written by store_kv for the new tokens, in the order of
                the new-token tensors (one per request for decode; the chunk
                tokens, request by request, for extend).
    """
    name: str
    kind: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    L: int
    NP: int
    layer: int
    scale: float
    seq_lens: np.ndarray
    page_table: np.ndarray
    out_loc: np.ndarray
    token_slots: list
    table_idx: np.ndarray | None = None
    qo_indptr: np.ndarray | None = None
    notes: dict = field(default_factory=dict)

    # ---- sizes -----------------------------------------------------------
    @property
    def n_new(self) -> int:
        return int(self.out_loc.shape[0])

    @property
    def total_q(self) -> int:
        return self.B if self.kind == "decode" else int(self.qo_indptr[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def max_chunk(self) -> int:
        if self.kind != "extend" or self.B == 0:
            return 1
        return int(np.diff(self.qo_indptr).max())

    @property
    def pool_shape(self):
        return (2, self.L, self.NP, self.P, self.Hkv, self.D)

    @property
    def pool_bytes(self) -> int:
        return int(np.prod(self.pool_shape)) * 2

    def referenced_slots(self) -> np.ndarray:
        if not self.token_slots:
            return np.zeros(0, np.int64)
        return np.unique(np.concatenate([np.asarray(s, np.int64) for s in self.token_slots]))

    # ---- values ----------------------------------------------------------
    def pool_rows(self, c: int, slots, device="cpu") -> torch.Tensor:
        """Generator values of pool[c, layer, slot] for the given slots: [n, Hkv, D]."""
        slots = torch.as_tensor(np.asarray(slots, np.int64), device=device)
        row = self.Hkv * self.D
        first = ((c * self.L + self.layer) * self.NP * self.P + slots) * row
        idx = first[:, None] + torch.arange(row, dtype=torch.int64, device=device)[None, :]
        return normal_bf16(self.seed, STREAM_POOL, idx.reshape(-1)).view(
            len(slots), self.Hkv, self.D)

    def q(self, device="cpu") -> torch.Tensor:
        return normal_tensor((self.total_q, self.Hq, self.D), self.seed, STREAM_Q, device)

    def new_kv(self, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
        shape = (self.n_new, self.Hkv, self.D)
        return (normal_tensor(shape, self.seed, STREAM_K_NEW, device),
                normal_tensor(shape, self.seed, STREAM_V_NEW, device))

    def make_pool(self, device="cpu", poison: bool = True,
                  chunk_slots: int = 1 << 16) -> torch.Tensor:
        """Pool tensor with the case's layer filled.

        Slots that hold a key before store_kv get generator values. With
        poison=True every other element of the layer (unreferenced slots, the
        out_loc slots, page tails) is NaN, so a read of anything the method must
        not read shows up in the output. Other layers are left uninitialised:
        nothing may read them.
        """
        pool = torch.empty(self.pool_shape, dtype=torch.bfloat16, device=device)
        before = self.slots_before_store()
        for c in (0, 1):
            plane = pool[c, self.layer].view(self.NP * self.P, self.Hkv, self.D)
            if poison:
                plane.fill_(float("nan"))
            for s in range(0, len(before), chunk_slots):
                part = before[s:s + chunk_slots]
                idx = torch.as_tensor(part, device=device)
                plane[idx] = self.pool_rows(c, part, device)
        return pool

    def slots_before_store(self) -> np.ndarray:
        """Referenced slots whose keys exist before store_kv (all but out_loc)."""
        ref = self.referenced_slots()
        return np.setdiff1d(ref, self.out_loc.astype(np.int64), assume_unique=False)

    def device_tables(self, device) -> dict:
        t = {
            "page_table": torch.as_tensor(self.page_table, dtype=torch.int32).to(device),
            "seq_lens": torch.as_tensor(self.seq_lens, dtype=torch.int32).to(device),
            "out_loc": torch.as_tensor(self.out_loc, dtype=torch.int32).to(device),
        }
        if self.table_idx is not None:
            t["table_idx"] = torch.as_tensor(self.table_idx, dtype=torch.int32).to(device)
        if self.qo_indptr is not None:
            t["qo_indptr"] = torch.as_tensor(self.qo_indptr, dtype=torch.int32).to(device)
        return t

    # ---- compaction for oracle checks of sampled requests ------------------
    def compact(self, requests) -> "Case":
        """The same computation restricted to `requests`, in a fresh small pool.

        Each kept request's pages are renumbered 0, 1, ... in row order (one
        layer, layer 0) and the pool values of every element are the ones the
        full case gives that element. Relocating physical pages changes no
        result of the method (the oracle's tests pin this), so the compact case
        answers for those requests exactly as the full one does.
        """
        requests = [int(r) for r in requests]
        P = self.P
        new_pages, rows, token_slots, out_loc, seq, qo = [], [], [], [], [], [0]
        page_map: dict[int, int] = {}
        for b in requests:
            n = int(self.seq_lens[b])
            row_id = int(self.table_idx[b]) if self.table_idx is not None else b
            pages = [int(p) for p in self.page_table[row_id, :(n + P - 1) // P]]
            row = []
            for p in pages:
                if p not in page_map:
                    page_map[p] = len(new_pages)
                    new_pages.append(p)
                row.append(page_map[p])
            rows.append(row)
            seq.append(n)
            token_slots.append(np.array([row[i // P] * P + i % P for i in range(n)],
                                        np.int64))
        if self.kind == "decode":
            for b in requests:
                out_loc.append(int(self._relocate(int(self.out_loc[b]), page_map)))
        else:
            for b in requests:
                s, e = int(self.qo_indptr[b]), int(self.qo_indptr[b + 1])
                out_loc.extend(int(self._relocate(int(x), page_map))
                               for x in self.out_loc[s:e])
                qo.append(qo[-1] + (e - s))
        stride = max([len(r) for r in rows] + [1])
        pt = np.zeros((len(rows), stride), np.int32)
        for i, r in enumerate(rows):
            pt[i, :len(r)] = r
        sub = CompactCase(
            name=f"{self.name}[compact {len(requests)}]", kind=self.kind, seed=self.seed,
            B=len(requests), Hq=self.Hq, Hkv=self.Hkv, D=self.D, P=P, L=1,
            NP=max(len(new_pages), 1), layer=0, scale=self.scale,
            seq_lens=np.array(seq, np.int32), page_table=pt,
            out_loc=np.array(out_loc, np.int32), token_slots=token_slots,
            qo_indptr=np.array(qo, np.int32) if self.kind == "extend" else None)
        sub.parent = self
        sub.requests = requests
        sub.page_origin = np.array(new_pages, np.int64)
        return sub

    def _relocate(self, slot: int, page_map: dict) -> int:
        return page_map[slot // self.P] * self.P + slot % self.P


class CompactCase(Case):
    """A Case cut out of a bigger one; values come from the parent's positions."""
    parent: Case
    requests: list
    page_origin: np.ndarray

    def pool_rows(self, c, slots, device="cpu"):
        slots = np.asarray(slots, np.int64)
        orig = self.page_origin[slots // self.P] * self.P + slots % self.P
        return self.parent.pool_rows(c, orig, device)

    def q(self, device="cpu"):
        if self.kind == "decode":
            rows = torch.as_tensor(self.requests, dtype=torch.int64)
        else:
            ind = self.parent.qo_indptr
            rows = torch.as_tensor(np.concatenate(
                [np.arange(ind[b], ind[b + 1]) for b in self.requests]), dtype=torch.int64)
        return _rows_of(self.parent, STREAM_Q, self.parent.Hq, rows, device)

    def new_kv(self, device="cpu"):
        if self.kind == "decode":
            rows = torch.as_tensor(self.requests, dtype=torch.int64)
        else:
            ind = self.parent.qo_indptr
            rows = torch.as_tensor(np.concatenate(
                [np.arange(ind[b], ind[b + 1]) for b in self.requests]), dtype=torch.int64)
        return (_rows_of(self.parent, STREAM_K_NEW, self.parent.Hkv, rows, device),
                _rows_of(self.parent, STREAM_V_NEW, self.parent.Hkv, rows, device))


def _rows_of(case: Case, stream: int, heads: int, rows: torch.Tensor, device) -> torch.Tensor:
    """Rows `rows` of a [n, heads, D] generator tensor of `case`."""
    width = heads * case.D
    idx = rows.to(device)[:, None] * width + torch.arange(width, device=device)[None, :]
    return normal_bf16(case.seed, stream, idx.reshape(-1)).view(len(rows), heads, case.D)


# --------------------------------------------------------------------------
# Allocation helpers (what a scheduler's page allocator would hand out)
# --------------------------------------------------------------------------

def _pad_rows(rows: list, stride: int, filler: np.ndarray) -> np.ndarray:
    """Page-table matrix; entries past a row's pages name unreferenced pages."""
    pt = np.empty((len(rows), max(stride, 1)), np.int32)
    k = 0
    for i, r in enumerate(rows):
        pt[i, :len(r)] = r
        for j in range(len(r), pt.shape[1]):
            pt[i, j] = filler[k % len(filler)] if len(filler) else 0
            k += 1
    return pt


def _slots_of_row(row, P: int, n: int) -> np.ndarray:
    row = np.asarray(row, np.int64)
    i = np.arange(n, dtype=np.int64)
    return row[i // P] * P + i % P


def random_case(seed: int, *, kind: str = "decode", seq_lens, chunk_lens=None,
                Hq: int = 4, Hkv: int = 2, D: int = 64, P: int = 1, L: int = 1,
                layer: int = 0, extra_pages: int = 64, shared_prefix: int = 0,
                group_size: int = 1, use_table_idx: bool = False,
                scale: float | None = None, name: str | None = None) -> Case:
    """Generic seeded case for sweeps.

    seq_lens     keys per request after store_kv (prefix + chunk for extend).
    chunk_lens   extend only: new tokens per request (the chunk).
    shared_prefix, group_size: consecutive groups of `group_size` requests
                 share their first `shared_prefix` tokens (a multiple of P),
                 as a radix-cache hit would give.
    use_table_idx rows live at shuffled page_table rows named by table_idx,
                 among extra unused rows.
    """
    rng = np.random.default_rng(seed)
    seq = np.asarray(seq_lens, np.int64)
    B = len(seq)
    if kind == "extend":
        chunks = np.asarray(chunk_lens, np.int64)
        if len(chunks) != B or np.any(chunks > seq - shared_prefix):
            raise ValueError("a chunk must fit after the shared prefix")
    if shared_prefix % P:
        raise ValueError("a shared prefix must cover whole pages")
    need = 0
    groups = (B + group_size - 1) // max(group_size, 1)
    for b in range(B):
        own = int(seq[b]) - (shared_prefix if shared_prefix else 0)
        if own < 0:
            raise ValueError("seq_len shorter than the shared prefix")
        need += (own + P - 1) // P
    need += groups * (shared_prefix // P)
    NP = need + extra_pages
    perm = rng.permutation(NP)
    cursor = 0
    rows = []
    prefix_pages = {}
    for b in range(B):
        g = b // max(group_size, 1)
        row = []
        if shared_prefix:
            if g not in prefix_pages:
                k = shared_prefix // P
                prefix_pages[g] = list(perm[cursor:cursor + k])
                cursor += k
            row += prefix_pages[g]
        own = int(seq[b]) - shared_prefix
        k = (own + P - 1) // P
        row += list(perm[cursor:cursor + k])
        cursor += k
        rows.append(row)
    filler = perm[cursor:]
    stride = max((int(s) + P - 1) // P for s in seq) if B else 1
    token_slots = [_slots_of_row(rows[b], P, int(seq[b])) for b in range(B)]
    pt = _pad_rows(rows, stride + 1, filler)
    table_idx = None
    if use_table_idx:
        n_rows = B + 3
        order = rng.permutation(n_rows)[:B]
        full = _pad_rows([[] for _ in range(n_rows)], pt.shape[1], filler[::-1])
        full[order] = pt
        pt = full
        table_idx = order.astype(np.int32)
    if kind == "decode":
        out_loc = np.array([token_slots[b][-1] for b in range(B)], np.int64)
        qo = None
    else:
        out_loc = np.concatenate([token_slots[b][int(seq[b] - chunks[b]):]
                                  for b in range(B)]) if B else np.zeros(0, np.int64)
        qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return Case(name=name or f"random-{kind}-{seed}", kind=kind, seed=seed, B=B, Hq=Hq,
                Hkv=Hkv, D=D, P=P, L=L, NP=NP, layer=layer,
                scale=scale if scale is not None else 1.0 / math.sqrt(D),
                seq_lens=seq.astype(np.int32), page_table=pt,
                out_loc=out_loc.astype(np.int32), token_slots=token_slots,
                table_idx=table_idx, qo_indptr=qo)


def cascade_case(seed: int, *, group_sizes, prefix_lens, suffix_lo: int = 1,
                 suffix_hi: int = 64, Hq: int = 4, Hkv: int = 2, D: int = 64, P: int = 1,
                 shuffled: bool = True, extra_pages: int = 16,
                 scale: float | None = None, name: str | None = None) -> Case:
    """Decode case whose requests come in groups sharing a prefix, as a radix
    cache hit gives: group k has group_sizes[k] members that share its first
    prefix_lens[k] keys (a multiple of P, possibly 0); each member then has a
    private suffix of U[suffix_lo, suffix_hi] keys on pages of its own. The
    request order is shuffled unless `shuffled` is false; the group of each
    request and each group's prefix length are kept in `notes`."""
    rng = np.random.default_rng(seed)
    sizes = [int(n) for n in group_sizes]
    plens = [int(n) for n in prefix_lens]
    if len(sizes) != len(plens) or any(n < 1 for n in sizes) or any(p % P for p in plens):
        raise ValueError("one prefix length (a multiple of P) per non-empty group")
    group_of = np.repeat(np.arange(len(sizes)), sizes)
    B = len(group_of)
    suffix = rng.integers(suffix_lo, suffix_hi + 1, size=B)
    need = sum(p // P for p in plens) + int(sum((int(n) + P - 1) // P for n in suffix))
    NP = need + extra_pages
    perm = rng.permutation(NP)
    cursor = 0
    prefix_pages = []
    for p in plens:
        prefix_pages.append(list(perm[cursor:cursor + p // P]))
        cursor += p // P
    rows = []
    for b in range(B):
        k = (int(suffix[b]) + P - 1) // P
        rows.append(prefix_pages[group_of[b]] + list(perm[cursor:cursor + k]))
        cursor += k
    order = rng.permutation(B) if shuffled else np.arange(B)
    rows = [rows[i] for i in order]
    group_of = group_of[order]
    seq = np.array([plens[group_of[b]] + int(suffix[order[b]]) for b in range(B)], np.int64)
    filler = perm[cursor:]
    stride = max((int(n) + P - 1) // P for n in seq)
    token_slots = [_slots_of_row(rows[b], P, int(seq[b])) for b in range(B)]
    pt = _pad_rows(rows, stride + 1, filler)
    out_loc = np.array([token_slots[b][-1] for b in range(B)], np.int64)
    return Case(name=name or f"cascade-{seed}", kind="decode", seed=seed, B=B, Hq=Hq, Hkv=Hkv,
                D=D, P=P, L=1, NP=NP, layer=0,
                scale=scale if scale is not None else 1.0 / math.sqrt(D),
                seq_lens=seq.astype(np.int32), page_table=pt, out_loc=out_loc.astype(np.int32),
                token_slots=token_slots,
                notes={"group_of_request": group_of.tolist(), "group_prefix": plens})


def cascade_tables(case: Case) -> dict:
    """The tables of a cascade decode call for a case whose requests share
    per-group prefixes (cascade_case, radix_shared_decode): per group the
    prefix's page row and length, the member lists, and per request the page
    row and length of its private suffix. Host numpy int32 arrays; the
    suffix pages follow from the same slots as the request's full row."""
    group_of = np.asarray(case.notes["group_of_request"], np.int64)
    G = int(group_of.max()) + 1 if case.B else 0
    plens = case.notes.get("group_prefix")
    if plens is None:
        plens = [int(case.notes["prefix"])] * G
    plens = np.asarray(plens, np.int64)
    P = case.P
    members = np.argsort(group_of, kind="stable").astype(np.int32)
    counts = np.bincount(group_of, minlength=G)
    member_indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    prefix_rows, suffix_rows = [], []
    for k in range(G):
        first = int(members[member_indptr[k]])
        slots = np.asarray(case.token_slots[first][:plens[k]], np.int64)
        prefix_rows.append(list(slots[::P] // P))
    suffix_lens = np.zeros(case.B, np.int64)
    for b in range(case.B):
        slots = np.asarray(case.token_slots[b][plens[group_of[b]]:], np.int64)
        suffix_lens[b] = len(slots)
        suffix_rows.append(list(slots[::P] // P))
    pstride = max(max((len(r) for r in prefix_rows), default=0), 1)
    sstride = max(max((len(r) for r in suffix_rows), default=0), 1)
    zero = np.zeros(1, np.int64)
    return {"prefix_page_table": _pad_rows(prefix_rows, pstride, zero),
            "prefix_lens": plens.astype(np.int32),
            "member_indptr": member_indptr, "members": members,
            "page_table": _pad_rows(suffix_rows, sstride, zero),
            "seq_lens": suffix_lens.astype(np.int32)}


# --------------------------------------------------------------------------
# The five named workloads
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 0) -> Case:
    """4 requests, seq_lens {1,7,16,33}, 4 q / 2 kv heads, head_dim 64,
    page_size 1, 256-slot pool, rows drawn from one seeded permutation."""
    rng = np.random.default_rng(seed)
    seq = [1, 7, 16, 33]
    perm = rng.permutation(256)
    rows, cur = [], 0
    for n in seq:
        rows.append(list(perm[cur:cur + n]))
        cur += n
    pt = _pad_rows(rows, max(seq), perm[cur:])
    token_slots = [np.asarray(r, np.int64) for r in rows]
    out_loc = np.array([r[-1] for r in rows], np.int32)
    return Case(name="tiny-decode", kind="decode", seed=seed, B=4, Hq=4, Hkv=2, D=64,
                P=1, L=1, NP=256, layer=0, scale=1.0 / math.sqrt(64),
                seq_lens=np.array(seq, np.int32), page_table=pt, out_loc=out_loc,
                token_slots=token_slots)


def llama8b_decode(seed: int = 0, batch: int = 64) -> Case:
    """Llama-3-8B-shaped decode: batch 64, 32 q / 8 kv heads, head_dim 128,
    page_size 1, seq_lens uniform in [512, 4096], slots drawn without
    replacement from a 400k-slot pool of 32 layers, one layer attended."""
    rng = np.random.default_rng(seed)
    seq = rng.integers(512, 4097, size=batch)
    NP, L = 400_000, 32
    layer = int(rng.integers(L))
    slots = rng.choice(NP, size=int(seq.sum()), replace=False)
    rows, cur = [], 0
    for n in seq:
        rows.append(slots[cur:cur + int(n)])
        cur += int(n)
    used = np.zeros(NP, bool)
    used[slots] = True
    filler = np.flatnonzero(~used)[:4096]
    pt = _pad_rows([list(r) for r in rows], 4096, filler)
    token_slots = [np.asarray(r, np.int64) for r in rows]
    out_loc = np.array([r[-1] for r in rows], np.int32)
    return Case(name="llama3-8b-decode", kind="decode", seed=seed, B=batch, Hq=32, Hkv=8,
                D=128, P=1, L=L, NP=NP, layer=layer, scale=1.0 / math.sqrt(128),
                seq_lens=seq.astype(np.int32), page_table=pt, out_loc=out_loc,
                token_slots=token_slots)


def radix_shared_decode(seed: int = 0, shuffled: bool = False) -> Case:
    """256 requests in 8 groups of 32; a group's rows share 2048 prefix slots,
    each request adds a private suffix of uniform [1, 512] tokens; 32 q / 8 kv
    heads, head_dim 128, page_size 1, 200k-slot pool. Group-major request order
    unless shuffled."""
    rng = np.random.default_rng(seed)
    NP, groups, per, prefix = 200_000, 8, 32, 2048
    perm = rng.permutation(NP)
    cur = 0
    rows = []
    for g in range(groups):
        pre = perm[cur:cur + prefix]
        cur += prefix
        for _ in range(per):
            n = int(rng.integers(1, 513))
            rows.append(np.concatenate([pre, perm[cur:cur + n]]))
            cur += n
    order = np.arange(len(rows))
    if shuffled:
        order = rng.permutation(len(rows))
    rows = [rows[i] for i in order]
    seq = np.array([len(r) for r in rows], np.int32)
    pt = _pad_rows([list(r) for r in rows], prefix + 512, perm[cur:])
    token_slots = [np.asarray(r, np.int64) for r in rows]
    out_loc = np.array([r[-1] for r in rows], np.int32)
    return Case(name="radix-shared-decode" + ("-shuffled" if shuffled else ""),
                kind="decode", seed=seed, B=len(rows), Hq=32, Hkv=8, D=128, P=1, L=1,
                NP=NP, layer=0, scale=1.0 / math.sqrt(128), seq_lens=seq, page_table=pt,
                out_loc=out_loc, token_slots=token_slots,
                notes={"groups": groups, "group_size": per, "prefix": prefix,
                       "group_prefix": [prefix] * groups,
                       "group_of_request": (order // per).tolist()})


def chunked_prefill_extend(seed: int = 0) -> Case:
    """8 requests, cached prefix uniform in [0, 8192], chunk lengths in
    [512, 2048] summing to 8192, 32 q / 8 kv heads, head_dim 128, page_size 1,
    slots from a permutation of an 80k-slot pool."""
    rng = np.random.default_rng(seed)
    B, total = 8, 8192
    prefix = rng.integers(0, 8193, size=B)
    while True:
        c = rng.integers(512, 2049, size=B).astype(np.float64)
        c = np.rint(c * total / c.sum()).astype(np.int64)
        c[-1] += total - int(c.sum())
        if c.min() >= 512 and c.max() <= 2048:
            break
    NP = 80_000
    perm = rng.permutation(NP)
    rows, cur = [], 0
    seq = prefix + c
    for n in seq:
        rows.append(perm[cur:cur + int(n)])
        cur += int(n)
    pt = _pad_rows([list(r) for r in rows], int(seq.max()), perm[cur:])
    token_slots = [np.asarray(r, np.int64) for r in rows]
    out_loc = np.concatenate([rows[b][int(prefix[b]):] for b in range(B)]).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
    return Case(name="chunked-prefill-extend", kind="extend", seed=seed, B=B, Hq=32,
                Hkv=8, D=128, P=1, L=1, NP=NP, layer=0, scale=1.0 / math.sqrt(128),
                seq_lens=seq.astype(np.int32), page_table=pt, out_loc=out_loc,
                token_slots=token_slots, qo_indptr=qo,
                notes={"prefix": prefix.tolist(), "chunks": c.tolist()})


def long_context_decode(seed: int = 0) -> Case:
    """Batch 16, seq_lens uniform in [32768, 131072], 32 q / 4 kv heads,
    head_dim 128, page_size 16, pages scattered by a seeded permutation of
    sum(ceil(seq/16)) + 1024 pages."""
    rng = np.random.default_rng(seed)
    B, P = 16, 16
    seq = rng.integers(32768, 131073, size=B)
    npages = (seq + P - 1) // P
    NP = int(npages.sum()) + 1024
    perm = rng.permutation(NP)
    rows, cur = [], 0
    for k in npages:
        rows.append(perm[cur:cur + int(k)])
        cur += int(k)
    pt = _pad_rows([list(r) for r in rows], int(npages.max()), perm[cur:])
    token_slots = [_slots_of_row(rows[b], P, int(seq[b])) for b in range(B)]
    out_loc = np.array([s[-1] for s in token_slots], np.int32)
    return Case(name="long-context-decode", kind="decode", seed=seed, B=B, Hq=32, Hkv=4,
                D=128, P=P, L=1, NP=NP, layer=0, scale=1.0 / math.sqrt(128),
                seq_lens=seq.astype(np.int32), page_table=pt, out_loc=out_loc,
                token_slots=token_slots)


NAMED = {
    "tiny-decode": tiny_decode,
    "llama3-8b-decode": llama8b_decode,
    "radix-shared-decode": radix_shared_decode,
    "chunked-prefill-extend": chunked_prefill_extend,
    "long-context-decode": long_context_decode,
}
