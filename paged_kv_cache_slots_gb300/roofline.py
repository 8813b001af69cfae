"""Byte and time accounting of a decode step (the measurement model).

decode_step_roofline restates the model of "Batching and Scheduling",
Example 1: a decode step moves the weights once plus every sequence's KV
cache, does 2 * params flops per token, and takes the larger of bytes /
bandwidth and flops / peak.  The tests pin it to that example's printed
table.  attention_bytes is the same bytes model restricted to the part this
library runs: the algorithmic bytes of one paged decode-attention launch and
of one append.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """K and V of one token over all layers (128 KiB for 32 x 8 x 128 x f16)."""
    return num_layers * num_kv_heads * head_dim * 2 * elem_bytes


def decode_step_roofline(batch: int, params: float, bits_per_weight: float, context: int,
                         kv_bytes_token: float, peak_flops: float, bandwidth: float) -> dict:
    weight_bytes = params * bits_per_weight / 8
    kv = batch * context * kv_bytes_token
    total = weight_bytes + kv
    flops = 2 * params * batch
    step = max(total / bandwidth, flops / peak_flops)
    return {"bytes": total, "kv_bytes": kv, "step_s": step, "tok_s": batch / step,
            "tok_s_per_seq": 1 / step, "util": flops / step / peak_flops}


def sequences_that_fit(vram: float, params: float, bits_per_weight: float, context: int,
                       kv_bytes_token: float) -> int:
    return int((vram - params * bits_per_weight / 8) // (context * kv_bytes_token))


@dataclass
class AttentionBytes:
    kv: int        # K and V rows read (every cached token, once per KV-head group)
    q: int
    out: int
    tables: int    # the block-table entries the kernel reads
    lens: int
    append: int    # new K/V rows read and written by the append

    @property
    def attention(self) -> int:
        return self.kv + self.q + self.out + self.tables + self.lens

    @property
    def step(self) -> int:
        return self.attention + self.append


def attention_bytes(context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    elem_bytes: int, block_size: int, out_elem_bytes: int,
                    appended_tokens: int, kv_elem_bytes: int | None = None) -> AttentionBytes:
    """Algorithmic bytes of one layer: split partials and the reduce are overhead, not counted.

    elem_bytes: q and the new K/V rows; kv_elem_bytes: the cache (default
    elem_bytes; 1 for an E4M3 cache, whose append reads elem_bytes per value
    and writes one byte)."""
    kvb = elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    ctx = np.asarray(context_lens, dtype=np.int64)
    B = len(ctx)
    kv = int(ctx.sum()) * num_kv_heads * head_dim * 2 * kvb
    q = B * num_q_heads * head_dim * elem_bytes
    out = B * num_q_heads * head_dim * out_elem_bytes
    tables = int(((ctx + block_size - 1) // block_size).sum()) * 4
    lens = B * 4
    append = 2 * appended_tokens * num_kv_heads * head_dim * (elem_bytes + kvb) + appended_tokens * 4
    return AttentionBytes(kv, q, out, tables, lens, append)
