"""Algorithmic byte ledger of the decode path (host-side accounting).

These are the bytes each call must move at minimum -- the numerator of every
GB/s and roofline fraction the benchmark reports. Split-KV partials, the
score workspace and padding reads are overhead, not algorithmic bytes.

Basis ("18 e2e inference serving" tutorial, sections 2.4-2.6): one token of
one layer stores K and V for every KV head, ``2 * Hkv * D * b`` bytes
(2048 B for Qwen2.5-7B's 4 KV heads x 128 dims in bf16); decode attention
reads each of those bytes once for the G = Hq / Hkv query heads sharing it,
so its arithmetic intensity is ``2 * Hq / (Hkv * b)`` FLOP per byte
(7 for 28/4 heads in bf16): far below the GPU's balance point, HBM-bound.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np

BF16 = 2


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elem_bytes: int = BF16) -> int:
    """K and V of one token in one layer: 2 * Hkv * D * b."""
    return 2 * num_kv_heads * head_dim * elem_bytes


def kv_bytes_per_block(num_kv_heads: int, head_dim: int, block_size: int, num_layers: int = 1,
                       elem_bytes: int = BF16) -> int:
    return kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes) * block_size * num_layers


def decode_arithmetic_intensity(num_q_heads: int, num_kv_heads: int, elem_bytes: int = BF16) -> float:
    """FLOP per KV byte of decode attention: 2 * Hq / (Hkv * b)."""
    return 2.0 * num_q_heads / (num_kv_heads * elem_bytes)


@dataclass
class StepBytes:
    reshape: int
    meta: int
    dense: int
    select: int
    sparse: int

    @property
    def total(self) -> int:
        return self.reshape + self.meta + self.dense + self.select + self.sparse

    def as_dict(self) -> Dict[str, int]:
        return dict(reshape=self.reshape, meta=self.meta, dense=self.dense, select=self.select,
                    sparse=self.sparse, total=self.total)


def step_bytes(context_lens: np.ndarray, slot_mapping: np.ndarray, Hq: int, Hkv: int, D: int,
               BS: int, topk: int, selected: Optional[np.ndarray] = None,
               elem_bytes: int = BF16, io_elem_bytes: int = BF16, q_rows: int = 1,
               block_scales: bool = False) -> StepBytes:
    """Algorithmic bytes of one step's five calls.

    reshape: new K and V rows read and written, plus the slots;
    meta:    new K rows read, min and max rows of each touched block read and
             written, plus the slots;
    dense:   K and V of every valid token, q, out, block-table entries, ctx;
    select:  min and max rows of every valid block, q, block-table entries,
             ctx, the selection written;
    sparse:  K and V of the valid tokens of the selected blocks, q, out, the
             selection and the block-table entries it dereferences, ctx.

    elem_bytes is the size of one cache / metadata element (2 for bf16, 1
    for an 8-bit cache); io_elem_bytes that of q, out and the new K/V rows
    (bf16 in both cases). q_rows is the number of query rows per sequence of
    the dense call (multi-token rows: each sequence's KV is still read once,
    the query and output bytes scale with the rows). block_scales: an 8-bit
    cache with per-block scales, whose fp32 K and V scale per (block, KV
    head) are read with each block (K only for the selection) and read and
    written by the write path for each touched block.
    """
    ctx = np.clip(np.asarray(context_lens, dtype=np.int64), 0, None)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    B = ctx.shape[0]
    row = Hkv * D * elem_bytes          # one token's K (or V) row in the cache
    row_io = Hkv * D * io_elem_bytes    # one new token's K (or V) row as passed in
    nb = (ctx + BS - 1) // BS
    valid = slots[slots >= 0]
    t_valid = int(valid.shape[0])
    touched = int(np.unique(valid // BS).shape[0])
    q_bytes = B * Hq * D * io_elem_bytes
    reshape = 2 * t_valid * (row_io + row) + 8 * slots.shape[0]
    meta = t_valid * row_io + touched * row * 2 * 2 + 8 * slots.shape[0]
    dense = int(ctx.sum()) * 2 * row + 2 * q_bytes * q_rows + int(nb.sum()) * 4 + 4 * B
    select = int(nb.sum()) * 2 * row + q_bytes + int(nb.sum()) * 4 + 4 * B + B * Hkv * topk * 4
    if selected is None:
        sparse = 0
    else:
        sel = np.asarray(selected, dtype=np.int64)
        tokens = 0
        nsel = 0
        for b in range(B):
            for g in range(Hkv):
                js = sel[b, g]
                js = js[(js >= 0) & (js < nb[b])]
                nsel += js.shape[0]
                tokens += int(np.minimum(BS, ctx[b] - js * BS).sum())
        sparse = tokens * 2 * D * elem_bytes + 2 * q_bytes + B * Hkv * topk * 4 + nsel * 4 + 4 * B
    if block_scales:
        reshape += touched * Hkv * 2 * 4 * 2
        dense += int(nb.sum()) * Hkv * 2 * 4
        select += int(nb.sum()) * Hkv * 4
        if selected is not None:
            sparse += nsel * 2 * 4
    return StepBytes(reshape=int(reshape), meta=int(meta), dense=int(dense), select=int(select),
                     sparse=int(sparse))
