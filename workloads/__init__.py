"""Seeded synthetic inputs for the paged decode read.

This module is shared by the tests, ``bench.py`` and the package entry's
``smoke()``.  It builds inputs only: it holds none of the read's arithmetic
(no scores, no softmax, no address walk of the kind the kernels do).  The
oracle and the CUDA library both receive the bytes it produces.

The workloads reproduce the shapes, sizes and value distributions of the
decode configurations the paged read is measured on: one query token per
row, K/V ~ N(0, 1), a pool of fixed-size blocks with block tables drawn from a
shuffled free list, ragged context lengths, and each step's new token written
through a slot mapping before the read.

Randomness: ``torch.Generator`` streams seeded per workload (CPU streams for
small metadata; the value tensors are drawn on the device the caller names,
so a full-size pool can be drawn on the GPU).  Nothing here is a golden
value: expected results come from the oracle on the same bytes.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One decode-step configuration.

    ctx: ("fixed", (c0, c1, ...)) | ("uniform", lo, hi) | ("loguniform", lo, hi)
        context length per row, *including* the token appended this step.
    pool: ("fixed", n) | ("exact",) | ("factor", f) | ("capacity",) | ("spare", n)
        how many physical blocks the pool has: a fixed count; exactly the
        blocks the rows need; f x that; rows x table capacity; needed + n.
    """

    name: str
    rows: int
    q_heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    dtype: str  # "f32" | "bf16"
    ctx: tuple
    pool: tuple
    seed: int
    scale: float | None = None  # None -> 1/sqrt(head_dim)
    description: str = ""
    table_capacity: int | None = None  # tokens a block table can hold (default: max context)
    query_len: int = 1  # new (query) tokens per row: its last query_len positions

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_context(self) -> int:
        if self.table_capacity is not None:
            return self.table_capacity
        kind = self.ctx[0]
        return max(self.ctx[1]) if kind == "fixed" else int(self.ctx[2])

    @property
    def max_blocks_per_row(self) -> int:
        return -(-self.max_context // self.block_size)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny-fp32", rows=2, q_heads=4, kv_heads=2, head_dim=16,
                 block_size=8, dtype="f32", ctx=("fixed", (16, 64)),
                 pool=("fixed", 32), seed=0, scale=0.25,
                 description="tiny fp32: 2 rows, contexts 16 and 64, 32-block "
                             "pool with permuted tables"),
        Workload("llama-fp32", rows=8, q_heads=32, kv_heads=8, head_dim=128,
                 block_size=16, dtype="f32", ctx=("uniform", 512, 2048),
                 pool=("exact",), seed=1,
                 description="fp32 Llama-style decode, contexts U[512, 2048]"),
        Workload("bf16-gqa4", rows=64, q_heads=32, kv_heads=8, head_dim=128,
                 block_size=16, dtype="bf16", ctx=("uniform", 1024, 8192),
                 pool=("factor", 1.25), seed=2,
                 description="bf16 KV, fp32 accumulate, contexts U[1024, 8192], "
                             "pool 1.25x the needed blocks"),
        Workload("bf16-long", rows=16, q_heads=64, kv_heads=8, head_dim=128,
                 block_size=32, dtype="bf16", ctx=("uniform", 32768, 131072),
                 pool=("capacity",), seed=3,
                 description="bf16 long context (split-K), contexts "
                             "U[32768, 131072], 8.6 GB K+V pool"),
        Workload("bf16-ragged-bs8", rows=256, q_heads=40, kv_heads=8,
                 head_dim=128, block_size=8, dtype="bf16",
                 ctx=("loguniform", 16, 16384), pool=("spare", 256), seed=4,
                 description="bf16 ragged batch, contexts log-uniform "
                             "[16, 16384], block 8, append then read"),
        Workload("bf16-ragged-bs32", rows=256, q_heads=40, kv_heads=8,
                 head_dim=128, block_size=32, dtype="bf16",
                 ctx=("loguniform", 16, 16384), pool=("spare", 256), seed=4,
                 description="bf16 ragged batch, contexts log-uniform "
                             "[16, 16384], block 32, append then read"),
        Workload("llama-fp32-kv16", rows=8, q_heads=64, kv_heads=16, head_dim=128,
                 block_size=16, dtype="f32", ctx=("uniform", 512, 2048),
                 pool=("exact",), seed=5,
                 description="fp32 decode with 16 kv heads (two 8-head groups per "
                             "row, so one bulk copy per token row), contexts "
                             "U[512, 2048]"),
        Workload("bf16-mqa", rows=64, q_heads=8, kv_heads=1, head_dim=128,
                 block_size=16, dtype="bf16", ctx=("uniform", 1024, 8192),
                 pool=("factor", 1.25), seed=6,
                 description="bf16 decode with one kv head (a GQA-8 model's per-GPU "
                             "slice under 8-way tensor parallelism), contexts "
                             "U[1024, 8192]"),
        Workload("bf16-kv2", rows=64, q_heads=16, kv_heads=2, head_dim=128,
                 block_size=16, dtype="bf16", ctx=("uniform", 1024, 8192),
                 pool=("factor", 1.25), seed=7,
                 description="bf16 decode with two kv heads (a GQA-8 model's per-GPU "
                             "slice under 4-way tensor parallelism), contexts "
                             "U[1024, 8192]"),
        Workload("bf16-kv4", rows=64, q_heads=32, kv_heads=4, head_dim=128,
                 block_size=16, dtype="bf16", ctx=("uniform", 1024, 8192),
                 pool=("factor", 1.25), seed=8,
                 description="bf16 decode with four kv heads (a GQA-8 model's per-GPU "
                             "slice under 2-way tensor parallelism), contexts "
                             "U[1024, 8192]"),
        Workload("bf16-gqa4-q4", rows=64, q_heads=32, kv_heads=8, head_dim=128,
                 block_size=16, dtype="bf16", ctx=("uniform", 1024, 8192),
                 pool=("factor", 1.25), seed=2, query_len=4,
                 description="bf16-gqa4 with 4 query tokens per row (speculative "
                             "decode): 4 new tokens appended, each attending "
                             "causally"),
    ]
}


def context_lengths(w: Workload) -> torch.Tensor:
    """Per-row context length (int32, CPU), including this step's new token."""
    g = torch.Generator().manual_seed(w.seed * 7919 + 1)
    kind = w.ctx[0]
    if kind == "fixed":
        vals = list(w.ctx[1])
        assert len(vals) == w.rows
        return torch.tensor(vals, dtype=torch.int32)
    lo, hi = int(w.ctx[1]), int(w.ctx[2])
    if kind == "uniform":
        return torch.randint(lo, hi + 1, (w.rows,), generator=g, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        u = torch.rand(w.rows, generator=g, dtype=torch.float64)
        c = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        return torch.round(c).clamp(lo, hi).to(torch.int32)
    raise ValueError(kind)


def truncated(w: Workload, rows: int) -> Workload:
    """The same recipe with only its first ``rows`` rows (same contexts)."""
    cl = context_lengths(w)[:rows]
    pool = w.pool if w.pool[0] != "fixed" else ("spare", 0)
    if pool[0] == "capacity":
        pool = ("spare", 0)
    return w.replace(name=f"{w.name}[:{rows}]", rows=rows,
                     ctx=("fixed", tuple(int(c) for c in cl)), pool=pool,
                     table_capacity=w.max_context,
                     description=f"{w.description}; first {rows} rows")


def pool_blocks(w: Workload, needed_total: int) -> int:
    kind = w.pool[0]
    if kind == "fixed":
        return int(w.pool[1])
    if kind == "exact":
        return needed_total
    if kind == "factor":
        return int(math.ceil(needed_total * float(w.pool[1])))
    if kind == "capacity":
        return w.rows * w.max_blocks_per_row
    if kind == "spare":
        return needed_total + int(w.pool[1])
    raise ValueError(kind)


@dataclass
class Metadata:
    context_lens: torch.Tensor  # [rows] int32
    block_tables: torch.Tensor  # [rows, max_blocks_per_row] int32, unused = -1
    slot_mapping: torch.Tensor  # [rows] (or [rows, query_len]) int64: new tokens' slots
    num_blocks: int


def metadata(w: Workload, context_lens: torch.Tensor | None = None,
             unused_entry: int = -1) -> Metadata:
    """Block tables from a shuffled free list, plus the new tokens' slots.

    Rows take their blocks, in row order, from a random permutation of the
    pool's physical block ids (the allocator's free list).  Table entries past
    a row's last needed block hold ``unused_entry``.  Each row's new token is
    the last of its history (position context_lens[r] - 1); its slot is where
    that position lives under the row's table.
    """
    cl = context_lengths(w) if context_lens is None else context_lens.to(torch.int32).cpu()
    bs, mb = w.block_size, w.max_blocks_per_row
    needed = [(-(-int(c) // bs)) for c in cl.tolist()]
    nb = pool_blocks(w, sum(needed))
    if sum(needed) > nb:
        raise ValueError("pool too small for the rows' contexts")
    g = torch.Generator().manual_seed(w.seed * 104729 + 3)
    free_list = torch.randperm(nb, generator=g).to(torch.int32)
    bt = torch.full((w.rows, mb), unused_entry, dtype=torch.int32)
    qn = w.query_len
    slots = torch.full((w.rows, qn), -1, dtype=torch.int64)
    pos = 0
    for r, n in enumerate(needed):
        bt[r, :n] = free_list[pos:pos + n]
        pos += n
        c = int(cl[r])
        for j in range(qn):  # new token j is position c - qn + j
            t = c - qn + j
            if t >= 0:
                slots[r, j] = int(bt[r, t // bs]) * bs + t % bs
    return Metadata(cl, bt, slots[:, 0].clone() if qn == 1 else slots, nb)


def history_slot_mask(w: Workload, md: Metadata, include_new: bool = False) -> torch.Tensor:
    """Bool [num_blocks * block_size]: True for slots holding a row's history.

    Excludes each row's new-token slots unless ``include_new``.  Used only to
    poison every other slot with NaN, so a read that touches a slot it should
    not shows up as a NaN in the output.
    """
    bs = w.block_size
    mask = torch.zeros(md.num_blocks * bs, dtype=torch.bool)
    for r in range(w.rows):
        c = int(md.context_lens[r])
        n = c if include_new else c - w.query_len
        if n <= 0:
            continue
        nblk = -(-n // bs)
        blocks = md.block_tables[r, :nblk].to(torch.int64)
        s = (blocks[:, None] * bs + torch.arange(bs)[None, :]).reshape(-1)[:n]
        mask[s] = True
    return mask


def _normal(shape, gen: torch.Generator, device, dtype: torch.dtype,
            chunk: int = 1 << 27) -> torch.Tensor:
    """N(0,1) in fp32, rounded to ``dtype`` (round-to-nearest-even), drawn in chunks."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(dtype)
    return out


@dataclass
class Inputs:
    w: Workload
    md: Metadata
    q: torch.Tensor  # [rows, q_heads, head_dim]
    k_pool: torch.Tensor  # [num_blocks, block_size, kv_heads, head_dim]
    v_pool: torch.Tensor
    k_new: torch.Tensor  # [rows, kv_heads, head_dim]
    v_new: torch.Tensor

    @property
    def block_tables(self):
        return self.md.block_tables

    @property
    def context_lens(self):
        return self.md.context_lens

    @property
    def slot_mapping(self):
        return self.md.slot_mapping


def make_inputs(w: Workload, device="cpu", *, poison: bool = True,
                md: Metadata | None = None) -> Inputs:
    """All tensors of one decode step of workload ``w``.

    q, k_new, v_new and every history slot of the pools are N(0,1) drawn from
    a generator on ``device`` seeded by the workload.  With ``poison``, every
    slot that is not part of some row's history before this step (free
    blocks, tails of last blocks, and the slots the new tokens are about to be
    written to) holds NaN.  Metadata tensors stay on the CPU (callers move
    them).
    """
    md = metadata(w) if md is None else md
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(w.seed * 1000003 + 17)
    dt = w.torch_dtype
    lead = (w.rows,) if w.query_len == 1 else (w.rows, w.query_len)
    q = _normal(lead + (w.q_heads, w.head_dim), gen, dev, dt)
    k_new = _normal(lead + (w.kv_heads, w.head_dim), gen, dev, dt)
    v_new = _normal(lead + (w.kv_heads, w.head_dim), gen, dev, dt)
    shape = (md.num_blocks, w.block_size, w.kv_heads, w.head_dim)
    k_pool = _normal(shape, gen, dev, dt)
    v_pool = _normal(shape, gen, dev, dt)
    if poison:
        keep = history_slot_mask(w, md).to(dev)
        bad = (~keep).view(md.num_blocks, w.block_size)
        k_pool[bad] = float("nan")
        v_pool[bad] = float("nan")
    return Inputs(w, md, q, k_pool, v_pool, k_new, v_new)


def host_array(t: torch.Tensor) -> np.ndarray:
    """A CPU numpy copy; bf16 comes back as its raw uint16 bit pattern."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def row_subproblem(inp: Inputs, rows: list[int], max_tokens: int | None = None) -> dict:
    """Host copies of the blocks a few rows need, with tables renumbered.

    For a full-size pool the oracle cannot take the whole pool; it takes the
    listed rows' blocks (gathered by torch indexing, block order kept) and a
    table that points at them in order.  Paging only moves where K/V live, so
    this is the same read.  Call it BEFORE any kernel touches the pool.
    ``max_tokens`` keeps each row's first max_tokens history tokens only (a
    prefix of the read, for timing samples); a new token past the prefix is
    then not appended (its slot is -1).
    """
    w, md = inp.w, inp.md
    bs = w.block_size
    ids, tables, offs = [], [], 0
    cl = md.context_lens[rows]
    if max_tokens is not None:
        cl = torch.clamp(cl, max=max_tokens)
    mb = max(1, max((-(-int(c) // bs)) for c in cl.tolist()))
    bt = torch.full((len(rows), mb), -1, dtype=torch.int32)
    qn = w.query_len
    slots = torch.full((len(rows), qn), -1, dtype=torch.int64)
    for i, r in enumerate(rows):
        c = int(cl[i])
        n = -(-c // bs)
        ids.append(md.block_tables[r, :n].to(torch.int64))
        bt[i, :n] = torch.arange(offs, offs + n, dtype=torch.int32)
        full = int(md.context_lens[r])
        for j in range(qn):
            t = full - qn + j
            if 0 <= t < c:
                slots[i, j] = (offs + t // bs) * bs + t % bs
        offs += n
    if qn == 1:
        slots = slots[:, 0].clone()
    idx = torch.cat(ids) if ids else torch.zeros(0, dtype=torch.int64)
    if idx.numel() == 0:
        idx = torch.zeros(1, dtype=torch.int64)
    dev_idx = idx.to(inp.k_pool.device)
    sel = torch.tensor(rows, dtype=torch.int64, device=inp.q.device)
    return dict(
        q=host_array(inp.q[sel]),
        k_new=host_array(inp.k_new[sel]),
        v_new=host_array(inp.v_new[sel]),
        k_pool=host_array(inp.k_pool[dev_idx]),
        v_pool=host_array(inp.v_pool[dev_idx]),
        block_tables=bt.numpy(),
        context_lens=cl.numpy().astype(np.int32),
        slot_mapping=slots.numpy(),
    )


def kv_bytes(w: Workload, context_lens: torch.Tensor) -> int:
    """K and V bytes of history one read must stream: sum_r c_r * 2 * Hk * D * es."""
    return int(context_lens.to(torch.int64).sum()) * 2 * w.kv_heads * w.head_dim * w.elem_size


def full_host(inp: Inputs) -> dict:
    """Host copies of every input of the step (small workloads only)."""
    return dict(
        q=host_array(inp.q), k_new=host_array(inp.k_new), v_new=host_array(inp.v_new),
        k_pool=host_array(inp.k_pool), v_pool=host_array(inp.v_pool),
        block_tables=inp.block_tables.numpy().copy(),
        context_lens=inp.context_lens.numpy().astype(np.int32),
        slot_mapping=inp.slot_mapping.numpy().copy(),
    )


# Tolerances of the parity gate: fp32 output within atol 1e-5 + rtol 1e-4
# (the kernel tolerance the streamed read is held to against the exact
# reference); bf16 output within atol 2e-2 of the exact result on the same
# bf16 inputs (the bf16 rounding of the output alone is up to 2^-9 relative).
TOLERANCE = {"f32": (1e-5, 1e-4), "bf16": (2e-2, 0.0)}
