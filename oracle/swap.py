"""Oracle for swapping KV blocks to host memory and back (test
infrastructure; only the tests import it).

Follows "Batching and Scheduling", Example 8 (preemption by swap: a request's
KV entries go to CPU memory and come back later).  A swapped block carries
every layer's K and V rows of one physical block.  Record i of a host buffer
holds, for layer l = 0, 1, ..., first the K rows and then the V rows of block
block_ids[i], each as the [num_kv_heads, block_size, head_dim] slice of that
layer's pool; records follow one another with no gaps.

Plain loops over records and layers, on CPU tensors (any element type; the
copy moves element bit patterns and does no arithmetic).
"""
from __future__ import annotations

import torch


def record_units(num_layers: int) -> list[tuple[int, str]]:
    """(layer, "K" | "V") of each unit of a record, in record order."""
    out = []
    for layer in range(num_layers):
        out.append((layer, "K"))
        out.append((layer, "V"))
    return out


def swap_out(k_layers, v_layers, block_ids) -> torch.Tensor:
    """Records of the listed blocks: [n, 2 * num_layers, Hkv, bs, D]."""
    units = record_units(len(k_layers))
    shape = tuple(k_layers[0].shape[1:])
    out = torch.empty((len(block_ids), len(units)) + shape, dtype=k_layers[0].dtype)
    for i, b in enumerate(block_ids):
        for u, (layer, kind) in enumerate(units):
            src = k_layers[layer] if kind == "K" else v_layers[layer]
            out[i, u] = src[int(b)]
    return out


def swap_in(k_layers, v_layers, records, block_ids):
    """New per-layer K and V lists with records[i] written to block block_ids[i]."""
    units = record_units(len(k_layers))
    k_new = [k.clone() for k in k_layers]
    v_new = [v.clone() for v in v_layers]
    for i, b in enumerate(block_ids):
        for u, (layer, kind) in enumerate(units):
            dst = k_new[layer] if kind == "K" else v_new[layer]
            dst[int(b)] = records[i, u]
    return k_new, v_new
