"""Swapping KV blocks to host memory and back ("Batching and Scheduling",
Example 8): the oracle pinned on the CPU, the library's sizes against the
page's numbers, and (on a GPU) the library's copy kernels against the oracle.
"""
from __future__ import annotations

import ctypes
import importlib.util
import json
import os
import types

import pytest
import torch

from oracle import swap as oracle_swap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "swap_example8.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _coded_pool(num_layers, num_blocks, hkv, bs, d):
    """Pool whose every element is its own (layer, K/V, block, head, token, dim) code."""
    ks, vs = [], []
    idx = torch.arange(num_blocks * hkv * bs * d, dtype=torch.int64).view(num_blocks, hkv, bs, d)
    for layer in range(num_layers):
        ks.append(idx + (2 * layer) * 10**9)
        vs.append(idx + (2 * layer + 1) * 10**9)
    return ks, vs


def _expected_code(layer, kind, block, hkv, bs, d):
    base = (2 * layer + (0 if kind == "K" else 1)) * 10**9 + block * hkv * bs * d
    return base + torch.arange(hkv * bs * d, dtype=torch.int64).view(hkv, bs, d)


def _check_closed_form(module):
    L, NB, H, BS, D = 3, 7, 2, 4, 8
    ks, vs = _coded_pool(L, NB, H, BS, D)
    ids = [5, 0, 6, 5]
    rec = module.swap_out(ks, vs, ids)
    assert tuple(rec.shape) == (len(ids), 2 * L, H, BS, D)
    for i, b in enumerate(ids):
        for layer in range(L):
            for j, kind in enumerate("KV"):
                assert torch.equal(rec[i, 2 * layer + j], _expected_code(layer, kind, b, H, BS, D))
    # Swap-in to other blocks of a zero pool: exactly those blocks change.
    zk = [torch.zeros_like(k) for k in ks]
    zv = [torch.zeros_like(v) for v in vs]
    dst = [1, 2, 3, 4]
    nk, nv = module.swap_in(zk, zv, rec, dst)
    for layer in range(L):
        for b in range(NB):
            if b in dst:
                src = ids[dst.index(b)]
                assert torch.equal(nk[layer][b], ks[layer][src])
                assert torch.equal(nv[layer][b], vs[layer][src])
            else:
                assert not nk[layer][b].any() and not nv[layer][b].any()
    # The inputs are left as they were.
    assert not any(k.any() for k in zk) and not any(v.any() for v in zv)


def test_oracle_records_follow_the_closed_form():
    _check_closed_form(oracle_swap)


MUTATIONS = [
    ("V before K", 'out.append((layer, "K"))\n        out.append((layer, "V"))',
     'out.append((layer, "V"))\n        out.append((layer, "K"))'),
    ("swap_out reads the list position", "out[i, u] = src[int(b)]", "out[i, u] = src[i]"),
    ("swap_in writes the list position", "dst[int(b)] = records[i, u]", "dst[i] = records[i, u]"),
    ("swap_in writes in place", "k_new = [k.clone() for k in k_layers]", "k_new = list(k_layers)"),
]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_closed_form_catches_planted_mistakes(what, old, new):
    with open(importlib.util.find_spec("oracle.swap").origin) as f:
        src = f.read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_swap_mutant")
    exec(compile(src.replace(old, new), "<mutant>", "exec"), mod.__dict__)
    with pytest.raises(AssertionError):
        _check_closed_form(mod)


def _pool_cfg(**kw):
    from paged_kv_cache_slots_gb300 import _PoolConfig
    c = dict(num_layers=32, num_blocks=200, block_size=16, num_kv_heads=8, head_dim=128, dtype=2,
             device=0)
    c.update(kw)
    return _PoolConfig(c["num_layers"], c["num_blocks"], c["block_size"], c["num_kv_heads"],
                       c["head_dim"], c["dtype"], c["device"])


def test_swap_bytes_match_the_page():
    # 2000 tokens of the 8B shape: 250 MiB each way, 16.6 ms out and back at
    # the 31.5 GB/s of a PCIe 4.0 x16 link.
    from paged_kv_cache_slots_gb300 import load_library
    g = _golden()
    lib = load_library()
    cfg = _pool_cfg()
    n = lib.kv_pool_bytes(ctypes.byref(cfg))
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(ctypes.byref(cfg), ctypes.c_void_p(0x10000000), n, ctypes.byref(h)) == 0
    try:
        blocks = g["tokens"] // g["block_size"]
        each_way = lib.kv_swap_bytes(h, blocks)
        assert each_way == g["each_way_bytes"] == g["tokens"] * g["bytes_per_token"]
        assert each_way == g["each_way_mib"] * 2**20
        assert round(2 * each_way / g["link_bytes_per_s"] * 1e3, 1) == g["out_and_back_ms"]
        assert lib.kv_swap_bytes(h, 0) == 0 and lib.kv_swap_bytes(h, -1) == 0
        # The oracle's record of one block has the same size.
        k = [torch.zeros((1, 8, 16, 128), dtype=torch.bfloat16)] * 32
        rec = oracle_swap.swap_out(k, k, [0])
        assert rec.numel() * rec.element_size() == lib.kv_swap_bytes(h, 1)
        # Nothing to copy: no CUDA call is made.
        assert lib.kv_swap_out(h, None, 0, None, 0, None) == 0
        assert lib.kv_swap_in(h, None, 0, None, 0, None) == 0
        # Host-side checks that need no GPU.
        fake = ctypes.c_void_p(0x20000000)
        assert lib.kv_swap_out(h, fake, 1, fake, each_way // blocks - 1, None) == 1
        assert lib.kv_swap_out(h, fake, -1, fake, 0, None) == 1
        assert lib.kv_swap_out(None, fake, 1, fake, 1 << 30, None) == 1
        assert lib.kv_swap_out(h, fake, 1, ctypes.c_void_p(0x20000008), 1 << 30, None) == 1
    finally:
        lib.kv_pool_destroy(h)


# ------------------------------------------------------------------ GPU


def _fill(pool, seed):
    g = torch.Generator(device=pool.device).manual_seed(seed)
    for layer in range(pool.num_layers):
        k, v = pool.layer(layer)
        for t in (k, v):
            t.copy_(torch.randn(t.shape, generator=g, device=pool.device).to(t.dtype))


def _layers(pool):
    ks, vs = [], []
    for layer in range(pool.num_layers):
        k, v = pool.layer(layer)
        ks.append(k.cpu())
        vs.append(v.cpu())
    return ks, vs


def _bits(t):
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.float16) else t.view(torch.int32)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,hkv,bs,d", [("bf16", 2, 16, 64), ("f32", 3, 8, 32), ("f16", 8, 16, 128)])
def test_swap_out_and_in_match_the_oracle(dtype, hkv, bs, d):
    from paged_kv_cache_slots_gb300 import KVPool
    pool = KVPool(3, 40, bs, hkv, d, dtype)
    _fill(pool, 7)
    ids = [39, 0, 17, 5, 6, 21, 38]
    host = pool.swap_out(ids)
    torch.cuda.synchronize()
    ks, vs = _layers(pool)
    want = oracle_swap.swap_out(ks, vs, ids)
    assert host.numel() == pool.swap_bytes(len(ids))
    got = host[:pool.swap_bytes(len(ids))].view(want.dtype).view(want.shape)
    assert torch.equal(_bits(got), _bits(want))
    # Swap back into other blocks; every other block keeps its contents.
    dst = [1, 2, 3, 30, 31, 32, 33]
    pool.swap_in(dst, host)
    torch.cuda.synchronize()
    wk, wv = oracle_swap.swap_in(ks, vs, want, dst)
    nk, nv = _layers(pool)
    for layer in range(pool.num_layers):
        assert torch.equal(_bits(nk[layer]), _bits(wk[layer]))
        assert torch.equal(_bits(nv[layer]), _bits(wv[layer]))


@pytest.mark.gpu
def test_swap_round_trip_of_the_page_context():
    # The page's preempted request: 2000 tokens of the 8B shape (125 blocks of
    # 16 tokens, 32 layers), swapped out, its blocks overwritten, swapped back.
    from paged_kv_cache_slots_gb300 import KVPool, device_status
    g = _golden()
    nblk = g["tokens"] // g["block_size"]
    pool = KVPool(32, 2 * nblk + 6, 16, 8, 128, "bf16")
    _fill(pool, 11)
    perm = torch.randperm(2 * nblk + 6, generator=torch.Generator().manual_seed(3))
    ids = perm[:nblk].to(torch.int32)
    before = pool.buffer.clone()
    host = pool.swap_out(ids)
    torch.cuda.synchronize()
    assert host.numel() == g["each_way_bytes"]
    for layer in (0, 31):
        k, v = pool.layer(layer)
        k[ids.long().cuda()] = 0
        v[ids.long().cuda()] = 0
    pool.swap_in(ids, host)
    torch.cuda.synchronize()
    assert torch.equal(pool.buffer, before)
    assert device_status() == (0, 0)
    # Sampled records against the oracle.
    ks, vs = _layers(pool)
    rec = host.view(torch.bfloat16).view(nblk, 64, 8, 16, 128)
    for i in (0, 61, nblk - 1):
        want = oracle_swap.swap_out(ks, vs, [int(ids[i])])
        assert torch.equal(_bits(rec[i]), _bits(want[0]))


@pytest.mark.gpu
def test_swap_refuses_pageable_memory_and_flags_bad_ids():
    from paged_kv_cache_slots_gb300 import FLAG_BAD_BLOCK_ID, KVError, KVPool, device_status
    pool = KVPool(2, 8, 16, 2, 64, "bf16")
    _fill(pool, 1)
    pageable = torch.empty(pool.swap_bytes(2), dtype=torch.uint8)
    with pytest.raises(KVError, match="pageable"):
        pool.swap_out([0, 1], host=pageable)
    host = pool.swap_out([1, 2])
    torch.cuda.synchronize()
    before = pool.buffer.clone()
    pool.swap_in([3, 8], host)  # 8 is out of range: skipped and flagged
    torch.cuda.synchronize()
    st, flags = device_status()
    assert flags & FLAG_BAD_BLOCK_ID and st != 0
    assert device_status() == (0, 0)  # reading the word clears it
    nk, nv = _layers(pool)
    ks = host[:pool.swap_bytes(1)].view(torch.bfloat16).view(4, 2, 16, 64)
    assert torch.equal(_bits(nk[0][3]), _bits(ks[0])) and torch.equal(_bits(nv[1][3]), _bits(ks[3]))
    # Blocks other than 3 are untouched.
    after = pool.buffer.view(torch.bfloat16).view(2, 2, 8, 2, 16, 64)
    prior = before.view(torch.bfloat16).view(2, 2, 8, 2, 16, 64)
    mask = torch.ones(8, dtype=torch.bool)
    mask[3] = False
    assert torch.equal(_bits(after[:, :, mask]), _bits(prior[:, :, mask]))
