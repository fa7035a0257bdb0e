"""Caller-side device buffers for one attention layer (torch allocations; no compute).

The library allocates nothing: these helpers size and allocate, with torch, the buffers the C
ABI describes -- the paged entry cache (blocks of 128 raw tokens), the indexer-key cache, the
state cache (window ring, pending raw rows, rows of the current call's new tokens) -- and build
the matching descriptors.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

from . import (BLOCK_TOKENS, LCS_ROW_BF16, LCS_ROW_FP8_SPLIT, ROPE_DIMS, WINDOW, Batch, Compressor, IndexKeys,
               Paging, RowSet, State)


def row_format_code(name: str) -> int:
    return {"bf16": LCS_ROW_BF16, "fp8_split": LCS_ROW_FP8_SPLIT}[name]


def alloc_rows(fmt: int, dim: int, n: int, device, zero: bool = True) -> RowSet:
    mk = torch.zeros if zero else torch.empty
    n_alloc = max(n, 1)
    if fmt == LCS_ROW_BF16:
        return RowSet(fmt, dim, n, mk((n_alloc, dim), dtype=torch.bfloat16, device=device))
    return RowSet(fmt, dim, n, mk((n_alloc, dim - ROPE_DIMS), dtype=torch.uint8, device=device),
                  mk((n_alloc, ROPE_DIMS), dtype=torch.bfloat16, device=device),
                  mk((n_alloc,), dtype=torch.float32, device=device))


def make_batch(seq_len_after: Sequence[int], new_tokens: Sequence[int], device,
               max_seq_len: Optional[int] = None) -> Batch:
    cu = [0]
    for q in new_tokens:
        cu.append(cu[-1] + int(q))
    return Batch(torch.tensor(cu, dtype=torch.int32, device=device),
                 torch.tensor(list(seq_len_after), dtype=torch.int32, device=device),
                 len(new_tokens), cu[-1], max(new_tokens) if len(new_tokens) else 0,
                 max_seq_len if max_seq_len is not None else max(seq_len_after))


@dataclasses.dataclass
class LayerCache:
    """Entry cache, indexer keys (CSA) and state cache of one layer for num_seqs sequences."""
    m: int
    overlap: bool
    dim: int
    fmt: int
    num_seqs: int
    capacity: int                  # raw tokens per sequence the block table covers
    paging: Paging
    entries: RowSet
    state: State
    keys: Optional[IndexKeys]

    @property
    def entries_per_block(self) -> int:
        return BLOCK_TOKENS // self.m


def alloc_layer(num_seqs: int, capacity: int, dim: int, fmt: int, m: int, overlap: bool, new_rows_cap: int,
                device, index_rank: int = 0, block_order: Optional[Sequence[int]] = None,
                per_channel: bool = False) -> LayerCache:
    """``block_order`` optionally permutes the physical blocks (to exercise the block table);
    ``per_channel`` adds the pending score rows of a per-channel compressor."""
    bps = math.ceil(capacity / BLOCK_TOKENS)
    epb = BLOCK_TOKENS // m
    nblocks = num_seqs * bps
    phys = list(range(nblocks)) if block_order is None else list(block_order)
    assert len(phys) == nblocks
    table = torch.tensor(phys, dtype=torch.int32, device=device).reshape(num_seqs, bps)
    paging = Paging(table, epb, bps)
    entries = alloc_rows(fmt, dim, nblocks * epb, device)
    slots = 2 * m if overlap else m
    pending = torch.zeros((num_seqs, slots, dim), dtype=torch.bfloat16, device=device)
    window = alloc_rows(fmt, dim, num_seqs * WINDOW, device)
    new_rows = alloc_rows(fmt, dim, new_rows_cap, device) if new_rows_cap > 0 else None
    pending_scores = (torch.zeros((num_seqs, slots, dim), dtype=torch.bfloat16, device=device)
                      if per_channel else None)
    state = State(window, pending, slots, new_rows, pending_scores)
    keys = None
    if index_rank:
        keys = IndexKeys(torch.zeros((nblocks * epb, index_rank // 2), dtype=torch.uint8, device=device),
                         torch.full((nblocks * epb, index_rank // 32), 127, dtype=torch.uint8, device=device),
                         index_rank, nblocks * epb)
    return LayerCache(m, overlap, dim, fmt, num_seqs, capacity, paging, entries, state, keys)


def compressor(w: torch.Tensor, bias: torch.Tensor, m: int, overlap: bool) -> Compressor:
    return Compressor(w, bias, m, overlap)
