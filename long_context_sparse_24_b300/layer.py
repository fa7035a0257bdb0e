"""One CSA or HCA attention layer driven through the C ABI.

Owns the caller-side buffers (entry cache, indexer keys, state cache, workspaces) and issues the
library calls of one step in order:
  CSA: (csa_compress -> csa_attend_window) || csa_index_topk, then csa_attend_topk
       [-> lcs_window_commit]
  HCA: hca_compress -> hca_attend [-> lcs_window_commit]
(lcs_window_commit only for multi-token steps; single-token steps keep the window in the ring.)
No arithmetic of the method happens here.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

from . import (LCS_INDEX_RELU, LCS_INDEX_SPARE_SMS, WINDOW, Batch, Compressor, csa_attend, csa_attend_topk,
               csa_attend_window, csa_compress, csa_index_topk, hca_attend, hca_compress, lcs_attend_workspace,
               lcs_index_topk_workspace, lcs_window_commit)
from . import buffers


class Layer:
    def __init__(self, kind: str, num_seqs: int, capacity: int, heads: int, dim: int = 512, fmt: int = 1,
                 m: Optional[int] = None, top_k: int = 512, index_heads: int = 4, index_rank: int = 128,
                 max_new: int = 1, softmax_scale: Optional[float] = None, relu: bool = False, device="cuda",
                 block_order: Optional[Sequence[int]] = None):
        assert kind in ("csa", "hca")
        self.kind = kind
        self.m = m if m is not None else (4 if kind == "csa" else 128)
        self.overlap = kind == "csa"
        self.heads, self.dim, self.fmt = heads, dim, fmt
        self.top_k, self.index_heads, self.index_rank = top_k, index_heads, index_rank
        self.relu = relu
        self.num_seqs, self.capacity, self.max_new = num_seqs, capacity, max_new
        self.scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(dim)
        self.device = device
        # one new token per sequence: the window ring takes every token directly (token p replaces
        # p-128, outside p's window), so there are no separate new-token rows and no commit step
        self.ring_only = max_new <= 1
        self.cache = buffers.alloc_layer(num_seqs, capacity, dim, fmt, self.m, self.overlap,
                                         0 if self.ring_only else num_seqs * max_new,
                                         device, index_rank=index_rank if kind == "csa" else 0,
                                         block_order=block_order)
        # compression and the window part of attention do not feed the indexer: they run on a side
        # stream next to it
        self.side = torch.cuda.Stream(device=device) if kind == "csa" else None
        self.comp: Optional[Compressor] = None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.sms = torch.cuda.get_device_properties(device).multi_processor_count
        # workspaces sized for the largest step this layer will run
        T = num_seqs * max_new
        probe = Batch(0, 0, num_seqs, T, max_new, capacity)
        self.topk_ws_bytes = (lcs_index_topk_workspace(probe, index_heads, self.cache.keys, self.cache.paging, self.m,
                                                       top_k) if kind == "csa" else 0)
        rows = (top_k + WINDOW) if kind == "csa" else (capacity // self.m + WINDOW)
        self.attend_rows = rows
        # the split plan (and so the workspace) depends on the step's token count: take the largest
        self.attend_ws_bytes = max(lcs_attend_workspace(Batch(0, 0, num_seqs, n, max_new, capacity), heads, dim, rows)
                                   for n in sorted({*range(1, min(T, 160) + 1), T}))
        # the index workspace starts with counters that must be zero before the first call (every
        # call leaves them zero)
        self.topk_ws = torch.zeros(max(self.topk_ws_bytes, 256), dtype=torch.uint8, device=device)
        self.attend_ws = torch.empty(max(self.attend_ws_bytes, 256), dtype=torch.uint8, device=device)
        self.topk_idx = torch.empty((T, max(top_k, 1)), dtype=torch.int32, device=device)
        self.topk_cnt = torch.empty((T,), dtype=torch.int32, device=device)

    def set_compressor(self, w: torch.Tensor, bias: torch.Tensor) -> None:
        self.comp = Compressor(w.contiguous(), bias.contiguous(), self.m, self.overlap)

    def batch(self, seq_len_after, new_tokens, cu_new=None, seq_len=None) -> Batch:
        b = buffers.make_batch(seq_len_after, new_tokens, self.device, max_seq_len=self.capacity)
        if cu_new is not None:
            b.cu_new, b.seq_len = cu_new, seq_len
        return b

    def compress(self, batch: Batch, raw: torch.Tensor, stream=None) -> None:
        fn = csa_compress if self.kind == "csa" else hca_compress
        fn(batch, raw, self.comp, self.cache.state, self.cache.entries, self.cache.paging, self.status, stream)

    def fill(self, batch: Batch, raw: torch.Tensor, stream=None) -> None:
        """Compress a chunk whose tokens are not attended in this call (cache building)."""
        st = buffers.State(self.cache.state.window, self.cache.state.pending, self.cache.state.pending_slots, None,
                           self.cache.state.pending_scores)
        fn = csa_compress if self.kind == "csa" else hca_compress
        fn(batch, raw, self.comp, st, self.cache.entries, self.cache.paging, self.status, stream)

    def select(self, batch: Batch, q_fp4, q_scale, head_w, stream=None, phase: int = 0, spare_sms: int = 0) -> None:
        """Indexer top-k; phase: 0 both phases, LCS_INDEX_SCORE_ONLY or LCS_INDEX_SELECT_ONLY;
        spare_sms: SMs the scorer leaves free for work running next to it."""
        csa_index_topk(batch, q_fp4, q_scale, head_w, self.index_heads, self.cache.keys, self.cache.paging, self.m,
                       self.top_k, (LCS_INDEX_RELU if self.relu else 0) | phase | LCS_INDEX_SPARE_SMS(spare_sms),
                       self.topk_idx, self.topk_cnt, self.topk_ws, self.topk_ws_bytes, self.status, stream)

    def window_ctas(self, batch: Batch) -> int:
        """SMs the indexer leaves to the window part of attention: one per query and 64-head group
        when they are few, and the indexer's scan is short enough (up to 65,536 entries a
        sequence) that the window part would otherwise lengthen the step; at longer contexts the
        scan dominates the step and keeps every SM (measured: 32 x 128K step 117.6 -> 109.7 us
        with the SMs left free, 32 x 1M 252 -> 284 us)."""
        n = batch.total_new * ((self.heads + 63) // 64)
        return n if n * 4 <= self.sms and batch.max_seq_len // self.m <= 65536 else 0

    def attend(self, batch: Batch, q: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
               stream=None) -> None:
        if self.kind == "csa":
            csa_attend(batch, q, self.heads, self.topk_idx, self.topk_cnt, self.top_k, self.m, self.cache.entries,
                       self.cache.paging, self.cache.state, self.scale, out, lse, self.attend_ws,
                       self.attend_ws_bytes, self.status, stream)
        else:
            hca_attend(batch, q, self.heads, self.m, self.cache.entries, self.cache.paging, self.cache.state,
                       self.scale, out, lse, self.attend_ws, self.attend_ws_bytes, self.status, stream)

    def commit(self, batch: Batch, stream=None) -> None:
        if not self.ring_only:
            lcs_window_commit(batch, self.cache.state, self.status, stream)

    def step(self, batch: Batch, raw_new: torch.Tensor, q: torch.Tensor, out: torch.Tensor,
             lse: Optional[torch.Tensor] = None, idx_q_fp4=None, idx_q_scale=None, head_w=None, stream=None,
             q_ready: Optional[torch.cuda.Event] = None) -> None:
        """One pass of the hot path for the batch's new tokens.  CSA: compression, then the window
        part of attention (side stream), run next to the indexer (scoring with the top-k fused
        in), which leaves SMs free for the window part's CTAs (about 208 KB of shared memory
        each: they could not start beside the indexer's CTAs otherwise); the top-k part of
        attention, with the merge of the two parts, waits for both.  q_ready: an event the
        attention waits for before reading q (q still arriving, e.g. copied from the host on
        another stream), so that compression and the indexer need not wait for it."""
        main = stream if stream is not None else torch.cuda.current_stream()
        if self.kind == "csa":
            self.side.wait_stream(main)
            self.compress(batch, raw_new, self.side)
            if q_ready is not None:
                self.side.wait_event(q_ready)
            csa_attend_window(batch, q, self.heads, self.top_k, self.m, self.cache.entries, self.cache.paging,
                              self.cache.state, self.scale, self.attend_ws, self.attend_ws_bytes, self.status,
                              self.side)
            self.select(batch, idx_q_fp4, idx_q_scale, head_w, main, spare_sms=self.window_ctas(batch))
            main.wait_stream(self.side)
            csa_attend_topk(batch, q, self.heads, self.topk_idx, self.topk_cnt, self.top_k, self.m, self.cache.entries,
                            self.cache.paging, self.cache.state, self.scale, out, lse, self.attend_ws,
                            self.attend_ws_bytes, self.status, main)
        else:
            self.compress(batch, raw_new, main)
            if q_ready is not None:
                main.wait_event(q_ready)
            self.attend(batch, q, out, lse, main)
        self.commit(batch, main)
