"""A stack of hybrid attention layers driven through the C ABI, CSA and HCA layers alternating.

Defined by: m.x-techcon.com/article/133366, section 2 (the two compressed attention types are
combined in alternation across layers; which layer uses which is fixed in advance, as the
latetalk.qiaomu.ai notes on V4's attention also say) and section 4 "专门为混合注意力设计的KV缓存管理"
(the compressed caches are allocated in blocks covering LCM(4, 128) = 128 raw tokens, so one
block table serves every layer: block i of a sequence holds 32 CSA entries in a CSA layer's pool
and one HCA entry in an HCA layer's pool).

Owns one Layer per attention layer; a step runs every layer's hot path for the batch's new
tokens, in layer order.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import torch

from . import LCS_ROW_FP8_SPLIT
from .layer import Layer


class HybridStack:
    def __init__(self, num_layers: int, num_seqs: int, capacity: int, heads: int, dim: int = 512,
                 fmt: int = LCS_ROW_FP8_SPLIT, csa_m: int = 4, hca_m: int = 128, top_k: int = 1024,
                 index_heads: int = 4, index_rank: int = 128, max_new: int = 1, first: str = "csa",
                 block_order: Optional[Sequence[int]] = None, device="cuda"):
        assert first in ("csa", "hca")
        kinds = ["csa", "hca"] if first == "csa" else ["hca", "csa"]
        self.kinds = [kinds[i % 2] for i in range(num_layers)]
        self.num_seqs, self.capacity, self.heads, self.dim = num_seqs, capacity, heads, dim
        # one physical block order for every layer (the shared block table)
        nblocks = num_seqs * math.ceil(capacity / 128)
        order = list(block_order) if block_order is not None else list(range(nblocks))
        self.layers: List[Layer] = [
            Layer(kd, num_seqs, capacity, heads, dim, fmt, csa_m if kd == "csa" else hca_m, top_k=top_k,
                  index_heads=index_heads, index_rank=index_rank, max_new=max_new, device=device,
                  block_order=order)
            for kd in self.kinds]

    def batch(self, seq_len_after, new_tokens):
        return self.layers[0].batch(seq_len_after, new_tokens)

    def step(self, batch, raw_new: Sequence[torch.Tensor], q: Sequence[torch.Tensor], out: Sequence[torch.Tensor],
             idx_q_fp4: Sequence[Optional[torch.Tensor]], idx_q_scale: Sequence[Optional[torch.Tensor]],
             head_w: Sequence[Optional[torch.Tensor]], stream=None) -> None:
        """Every layer's step for the batch's new tokens: per layer l, raw_new[l] (its new KV rows),
        q[l] (queries), out[l] (outputs) and, for CSA layers, the indexer query codes."""
        for li, layer in enumerate(self.layers):
            layer.step(batch, raw_new[li], q[li], out[li], idx_q_fp4=idx_q_fp4[li], idx_q_scale=idx_q_scale[li],
                       head_w=head_w[li], stream=stream)

    @property
    def status(self) -> List[int]:
        return [int(layer.status.item()) for layer in self.layers]
