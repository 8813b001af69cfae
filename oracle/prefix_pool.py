"""Oracle for the block pool with prefix caching (test infrastructure).

Only the tests import this module; the library never calls it and it never
calls the library.

Follows "Reading Inference Engine Codebases", Examples 12 and 13 (vLLM's
KV cache manager and block pool), in plain Python:

  * a full block is identified by the whole token prefix that ends with it.
    The pages identify it by a hash chained over parent hash and block
    tokens; that hash stands for exactly this prefix, so the oracle keys its
    cache on the prefix itself (a tuple of token ids), with no hash function;
  * allocate: the hits are the longest run of cached full blocks matching the
    request, at most (num_tokens - 1) // block_size of them; a hit gains a
    reference and leaves the free queue if it was in it; the remaining blocks
    are taken from the front of the free queue, and a taken block that still
    holds a prefix loses it (it is evicted); each new full block is cached
    under its prefix, after any earlier blocks cached under the same prefix
    (equal blocks are not merged, a lookup takes the first);
  * free: the request's blocks are walked last to first; a block whose count
    reaches zero goes to the front of the queue if it holds no prefix and to
    the back if it does;
  * the free queue starts as every block in increasing id order.
"""
from __future__ import annotations


class OutOfBlocks(Exception):
    pass


class PrefixPool:
    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.ref = [0] * num_blocks
        self.prefix = [None] * num_blocks   # prefix tuple held by each block, or None
        self.queue = list(range(num_blocks))  # front first
        self.cache = {}                      # prefix tuple -> list of blocks, oldest first

    def allocate(self, tokens):
        """Returns (blocks, cached_tokens, evicted)."""
        bs = self.block_size
        n = len(tokens)
        full = n // bs
        total = -(-n // bs)
        max_hit = (n - 1) // bs if n > 0 else 0
        hits = []
        for i in range(min(full, max_hit)):
            key = tuple(tokens[:(i + 1) * bs])
            if key not in self.cache:
                break
            hits.append(self.cache[key][0])
        leaving = sum(1 for b in hits if self.ref[b] == 0)
        if total - len(hits) > len(self.queue) - leaving:
            raise OutOfBlocks(f"{total - len(hits)} blocks needed")
        for b in hits:
            if self.ref[b] == 0:
                self.queue.remove(b)
            self.ref[b] += 1
        blocks = list(hits)
        evicted = []
        for i in range(len(hits), total):
            b = self.queue.pop(0)
            if self.prefix[b] is not None:
                owners = self.cache[self.prefix[b]]
                owners.remove(b)
                if not owners:
                    del self.cache[self.prefix[b]]
                self.prefix[b] = None
                evicted.append(b)
            self.ref[b] = 1
            if i < full:
                key = tuple(tokens[:(i + 1) * bs])
                self.prefix[b] = key
                self.cache.setdefault(key, []).append(b)
            blocks.append(b)
        return blocks, len(hits) * bs, evicted

    def free(self, blocks):
        blocks = list(blocks)
        for b in set(blocks):
            if not 0 <= b < len(self.ref) or blocks.count(b) > self.ref[b]:
                raise ValueError(f"block {b} is not in use")
        for b in reversed(blocks):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if self.prefix[b] is None:
                    self.queue.insert(0, b)
                else:
                    self.queue.append(b)

    def free_queue(self):
        return list(self.queue)

    def cache_size(self):
        return len(self.cache), sum(len(v) for v in self.cache.values())

