"""Block pool with prefix caching: the oracle and the library's pool against
the printed output of "Reading Inference Engine Codebases", Example 13, and
against each other on seeded request streams (CPU only)."""
from __future__ import annotations

import importlib.util
import json
import os
import types

import pytest

from oracle import prefix_pool as oracle_pool
from workloads import prefix_request_trace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "prefix_cache_block_pool_example13.json")


def _example():
    with open(GOLDEN) as f:
        return json.load(f)


class _OracleAdapter:
    """The oracle behind the binding's interface (None when out of blocks)."""

    def __init__(self, module, num_blocks, block_size):
        self.p = module.PrefixPool(num_blocks, block_size)
        self.module = module

    def allocate(self, tokens):
        try:
            return self.p.allocate(tokens)
        except self.module.OutOfBlocks:
            return None

    def free(self, blocks):
        self.p.free(blocks)

    def free_queue(self):
        return self.p.free_queue()

    def cache_size(self):
        return self.p.cache_size()


def _lines(pool, g):
    """Replays the example and formats what its program prints."""
    out, held = [], {}
    for op in g["ops"]:
        if op["op"] == "free":
            pool.free(held.pop(op["name"]))
            continue
        tokens = op["tokens"]
        blocks, cached, evicted = pool.allocate(tokens)
        held[op["name"]] = blocks
        out += [f"  evict block {b}" for b in evicted]
        out.append(f"{op['name']}: {len(tokens)} tokens, cached {cached}, computed "
                   f"{len(tokens) - cached}, blocks {blocks}, free {len(pool.free_queue())}")
    return out


def test_golden_tokens_follow_the_printed_recipe():
    g = _example()
    allocs = [op for op in g["ops"] if op["op"] == "allocate"]
    recipe = [(8, 5, 500), (8, 3, 900), (8, 0, 0), (0, 15, 300)]
    for op, (shared, own, seed) in zip(allocs, recipe):
        assert op["tokens"] == [100 + i if i < shared else seed + i for i in range(shared + own)]


def test_oracle_reproduces_example13():
    g = _example()
    assert _lines(_OracleAdapter(oracle_pool, g["num_blocks"], g["block_size"]), g) == g["printed"]


def test_library_pool_reproduces_example13():
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    g = _example()
    assert _lines(PrefixCachePool(g["num_blocks"], g["block_size"]), g) == g["printed"]


def _queue_after_a(pool, g):
    blocks, _, _ = pool.allocate(g["ops"][0]["tokens"])
    pool.free(blocks)
    return pool.free_queue()


def test_example13_free_queue_after_request_a():
    # Freeing A walks its blocks tail first: the unhashed partial block 3 goes
    # to the front, the hashed blocks 2, 1, 0 to the back in that order.
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    g = _example()
    for pool in (PrefixCachePool(8, 4), _OracleAdapter(oracle_pool, 8, 4)):
        assert _queue_after_a(pool, g) == g["free_queue_after_freeing_a"]
        assert pool.cache_size() == (3, 3)


# Plausible mistakes, planted in a copy of the oracle's source; each must make
# the oracle disagree with the printed output or the stated free queue.
MUTATIONS = [
    ("no cap on hits", "max_hit = (n - 1) // bs if n > 0 else 0", "max_hit = full"),
    ("free walks head first", "for b in reversed(blocks):", "for b in blocks:"),
    ("unhashed block to the back", "self.queue.insert(0, b)", "self.queue.append(b)"),
    ("hashed block to the front", "                    self.queue.append(b)",
     "                    self.queue.insert(0, b)"),
    ("pop from the back", "b = self.queue.pop(0)", "b = self.queue.pop()"),
    ("hits stay in the queue", "                self.queue.remove(b)\n", "                pass\n"),
    ("prefix is the block alone", "key = tuple(tokens[:(i + 1) * bs])\n            if key",
     "key = tuple(tokens[i * bs:(i + 1) * bs])\n            if key"),
    ("partial block cached", "            if i < full:", "            if True:"),
    ("no eviction", "                evicted.append(b)\n", ""),
]


def _mutant(src, old, new):
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_prefix_pool_mutant")
    exec(compile(src.replace(old, new), "<mutant>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_example13_catches_planted_mistakes(what, old, new):
    g = _example()
    spec = importlib.util.find_spec("oracle.prefix_pool")
    with open(spec.origin) as f:
        src = f.read()
    mod = _mutant(src, old, new)
    try:
        lines = _lines(_OracleAdapter(mod, g["num_blocks"], g["block_size"]), g)
        queue = _queue_after_a(_OracleAdapter(mod, g["num_blocks"], g["block_size"]), g)
    except Exception:
        return  # the mistake breaks the replay outright
    assert lines != g["printed"] or queue != g["free_queue_after_freeing_a"], what


def _invariants(pool, live, num_blocks):
    q = pool.free_queue()
    assert len(q) == len(set(q))
    held = {b for blocks in live for b in blocks}
    assert held.isdisjoint(q)
    assert held | set(q) == set(range(num_blocks))


@pytest.mark.parametrize("seed,num_blocks,block_size", [(1, 24, 4), (2, 40, 4), (3, 64, 16),
                                                        (4, 12, 1), (5, 30, 7)])
def test_library_pool_matches_oracle_on_request_streams(seed, num_blocks, block_size):
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    lib = PrefixCachePool(num_blocks, block_size)
    ref = _OracleAdapter(oracle_pool, num_blocks, block_size)
    live = []
    hits = evictions = refusals = 0
    for op, arg in prefix_request_trace(seed, 400):
        if op == "free":
            if not live:
                continue
            blocks = live.pop(arg % len(live))
            lib.free(blocks)
            ref.free(blocks)
        else:
            got, want = lib.allocate(arg), ref.allocate(arg)
            assert got == want
            if got is None:
                refusals += 1
            else:
                live.append(got[0])
                hits += got[1] > 0
                evictions += len(got[2])
        assert lib.free_queue() == ref.free_queue()
        assert lib.cache_size() == ref.cache_size()
        _invariants(lib, live, num_blocks)
    # The stream exercised hits, evictions and refusals.
    assert hits > 0 and evictions > 0 and refusals > 0


def test_full_match_recomputes_the_last_block():
    # A request equal to a cached 3-block prefix hits 2 blocks: the last token
    # is always computed again, and only whole blocks count.
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    for pool in (PrefixCachePool(10, 4), _OracleAdapter(oracle_pool, 10, 4)):
        toks = list(range(12))
        a, _, _ = pool.allocate(toks)
        b, cached, _ = pool.allocate(toks)
        assert cached == 8 and b[:2] == a[:2] and b[2] != a[2]
        # 13 tokens: 3 full blocks may hit, 1 new block.
        c, cached, _ = pool.allocate(toks + [99])
        assert cached == 12 and c[:3] == a[:3]
        # Equal blocks are not merged: the third block's prefix now has two blocks.
        assert pool.cache_size() == (3, 4)


def test_same_block_tokens_after_different_prefixes_do_not_match():
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    for pool in (PrefixCachePool(10, 2), _OracleAdapter(oracle_pool, 10, 2)):
        pool.allocate([1, 2, 5, 6, 0])
        _, cached, _ = pool.allocate([3, 4, 5, 6, 0])
        assert cached == 0


def test_refused_allocation_changes_nothing():
    from paged_kv_cache_slots_gb300 import PrefixCachePool
    pool = PrefixCachePool(4, 4)
    a, _, _ = pool.allocate(list(range(10)))
    q = pool.free_queue()
    assert pool.allocate(list(range(100, 110))) is None
    assert pool.free_queue() == q and pool.cache_size() == (2, 2)
    # A request that hits a freed cached block may still fit.
    pool.free(a)
    b, cached, _ = pool.allocate(list(range(9)) + [77, 78, 79, 80, 81, 82, 83])
    assert cached == 8 and len(b) == 4


def test_library_pool_errors():
    from paged_kv_cache_slots_gb300 import KVError, PrefixCachePool
    pool = PrefixCachePool(4, 4)
    a, _, _ = pool.allocate([1, 2, 3])
    with pytest.raises(KVError):
        pool.free([7])
    with pytest.raises(KVError):
        pool.free(a + a)  # one reference, freed twice
    assert pool.free_queue() == [1, 2, 3]
    pool.free(a)
    with pytest.raises(KVError):
        pool.free(a)
    with pytest.raises(KVError):
        PrefixCachePool(0, 4)
    assert pool.allocate([]) == ([], 0, [])
