// Host block pool with prefix caching ("Reading Inference Engine Codebases",
// Examples 12 and 13: vLLM's KV cache manager and block pool).
//
// Behaviour restated from those examples:
//   - a full block's hash covers its parent's hash and its own tokens, so a
//     hash identifies the whole prefix up to the end of that block;
//   - a new request reuses the longest run of cached full blocks matching its
//     prefix, capped so that the last token is always computed again
//     ((num_tokens - 1) / block_size blocks at most); a hit block gains a
//     reference and leaves the free queue;
//   - the other blocks are popped from the front of the free queue; a popped
//     block that still carries a hash is evicted from the cache;
//   - equal blocks are not de-duplicated: one hash may map to several blocks,
//     a lookup takes the first;
//   - freeing walks a request's blocks tail first; a block whose count drops
//     to zero goes to the front of the queue when it has no hash and to the
//     back when it has one (least recently used first).
// The hash function is this file's own (64-bit FNV-1a over the parent hash
// and the token ids); a lookup also compares the stored parent hash and
// tokens, so only exact prefix equality counts.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

using pkv::report_error;

namespace {

struct PBlock {
    int32_t id = 0;
    int32_t ref = 0;
    bool hashed = false;
    uint64_t hash = 0;
    uint64_t parent = 0;
    std::vector<int32_t> tokens;  // the block's tokens (when hashed)
    std::list<int32_t>::iterator qpos;
    bool queued = false;
};

uint64_t chain_hash(uint64_t parent, const int32_t* tok, int n) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint64_t v) {
        for (int i = 0; i < 8; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= 1099511628211ull;
        }
    };
    mix(parent);
    for (int i = 0; i < n; ++i) mix(static_cast<uint32_t>(tok[i]));
    return h;
}

constexpr uint64_t kNoParent = 0x9e3779b97f4a7c15ull;

}  // namespace

struct kv_prefix_pool {
    int block_size = 0;
    std::vector<PBlock> blocks;
    std::list<int32_t> free_q;  // front = next to reuse / evict
    std::unordered_map<uint64_t, std::vector<int32_t>> cached;

    void dequeue(PBlock& b) {
        if (b.queued) {
            free_q.erase(b.qpos);
            b.queued = false;
        }
    }
    void push_front(PBlock& b) {
        free_q.push_front(b.id);
        b.qpos = free_q.begin();
        b.queued = true;
    }
    void push_back(PBlock& b) {
        free_q.push_back(b.id);
        b.qpos = std::prev(free_q.end());
        b.queued = true;
    }
    // First cached block for (hash, parent, tokens), or -1.
    int32_t lookup(uint64_t h, uint64_t parent, const int32_t* tok) const {
        auto it = cached.find(h);
        if (it == cached.end()) return -1;
        for (int32_t id : it->second) {
            const PBlock& b = blocks[id];
            if (b.parent == parent &&
                std::memcmp(b.tokens.data(), tok, sizeof(int32_t) * block_size) == 0)
                return id;
        }
        return -1;
    }
    void evict(PBlock& b) {
        auto it = cached.find(b.hash);
        if (it != cached.end()) {
            auto& v = it->second;
            for (size_t i = 0; i < v.size(); ++i)
                if (v[i] == b.id) {
                    v.erase(v.begin() + static_cast<long>(i));
                    break;
                }
            if (v.empty()) cached.erase(it);
        }
        b.hashed = false;
        b.tokens.clear();
    }
};

extern "C" {

kv_status_t kv_prefix_pool_create(int num_blocks, int block_size, kv_prefix_pool_t** out) {
    if (!out || num_blocks <= 0 || block_size <= 0)
        return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_create: %d blocks of %d tokens",
                            num_blocks, block_size);
    *out = nullptr;
    kv_prefix_pool* p = new (std::nothrow) kv_prefix_pool;
    if (!p) return report_error(KV_ERR_OUT_OF_MEMORY, "kv_prefix_pool_create: out of host memory");
    p->block_size = block_size;
    p->blocks.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) {  // the queue starts in block-id order
        p->blocks[i].id = i;
        p->push_back(p->blocks[i]);
    }
    *out = p;
    return KV_OK;
}

void kv_prefix_pool_destroy(kv_prefix_pool_t* p) { delete p; }

kv_status_t kv_prefix_pool_allocate(kv_prefix_pool_t* p, const int32_t* tokens, int num_tokens,
                                    int32_t* blocks_out, int capacity, int* num_blocks_out,
                                    int* cached_tokens_out, int32_t* evicted_out,
                                    int evicted_capacity, int* num_evicted_out) {
    if (!p || num_tokens < 0 || (num_tokens > 0 && !tokens) || !blocks_out || !num_blocks_out)
        return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_allocate: null argument or %d tokens",
                            num_tokens);
    const int bs = p->block_size;
    const int total = (num_tokens + bs - 1) / bs;
    const int full = num_tokens / bs;
    if (total > capacity)
        return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_allocate: %d blocks > capacity %d",
                            total, capacity);
    // Hashes of the full blocks, chained.
    std::vector<uint64_t> hs(full), parents(full);
    uint64_t parent = kNoParent;
    for (int i = 0; i < full; ++i) {
        parents[i] = parent;
        hs[i] = parent = chain_hash(parent, tokens + i * bs, bs);
    }
    // Longest run of hits, capped so that the last token is computed again.
    const int max_hit = num_tokens > 0 ? (num_tokens - 1) / bs : 0;
    std::vector<int32_t> hits;
    for (int i = 0; i < full && i < max_hit; ++i) {
        const int32_t id = p->lookup(hs[i], parents[i], tokens + i * bs);
        if (id < 0) break;
        hits.push_back(id);
    }
    // Enough free blocks?  A hit that sits in the free queue leaves it.
    int hits_in_queue = 0;
    for (int32_t id : hits) hits_in_queue += p->blocks[id].ref == 0;
    const int need = total - static_cast<int>(hits.size());
    const int avail = static_cast<int>(p->free_q.size()) - hits_in_queue;
    if (need > avail)
        return report_error(KV_ERR_OUT_OF_BLOCKS, "kv_prefix_pool_allocate: %d new blocks, %d free",
                            need, avail);
    int n = 0, ne = 0;
    for (int32_t id : hits) {  // touch
        PBlock& b = p->blocks[id];
        if (b.ref == 0) p->dequeue(b);
        ++b.ref;
        blocks_out[n++] = id;
    }
    for (int i = static_cast<int>(hits.size()); i < total; ++i) {
        PBlock& b = p->blocks[p->free_q.front()];
        p->dequeue(b);
        if (b.hashed) {
            p->evict(b);
            if (evicted_out && ne < evicted_capacity) evicted_out[ne] = b.id;
            ++ne;
        }
        b.ref = 1;
        if (i < full) {  // a full block is cached under its prefix hash
            b.hashed = true;
            b.hash = hs[i];
            b.parent = parents[i];
            b.tokens.assign(tokens + i * bs, tokens + (i + 1) * bs);
            p->cached[b.hash].push_back(b.id);
        }
        blocks_out[n++] = b.id;
    }
    *num_blocks_out = n;
    if (cached_tokens_out) *cached_tokens_out = static_cast<int>(hits.size()) * bs;
    if (num_evicted_out) *num_evicted_out = ne;
    return KV_OK;
}

kv_status_t kv_prefix_pool_free(kv_prefix_pool_t* p, const int32_t* blocks, int n) {
    if (!p || n < 0 || (n > 0 && !blocks))
        return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_free: null argument");
    // Every count must stay >= 0, also when a block is listed twice.
    std::unordered_map<int32_t, int> drops;
    for (int i = 0; i < n; ++i) {
        if (blocks[i] < 0 || blocks[i] >= static_cast<int>(p->blocks.size()))
            return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_free: block %d out of range",
                                blocks[i]);
        if (++drops[blocks[i]] > p->blocks[blocks[i]].ref)
            return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_free: block %d is not in use",
                                blocks[i]);
    }
    for (int i = n - 1; i >= 0; --i) {  // tail first
        PBlock& b = p->blocks[blocks[i]];
        if (--b.ref == 0) {
            if (b.hashed)
                p->push_back(b);
            else
                p->push_front(b);
        }
    }
    return KV_OK;
}

kv_status_t kv_prefix_pool_free_queue(const kv_prefix_pool_t* p, int32_t* out, int capacity,
                                      int* count_out) {
    if (!p || capacity < 0 || (capacity > 0 && !out))
        return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_free_queue: null argument");
    const int n = static_cast<int>(p->free_q.size());
    if (count_out) *count_out = n;
    if (out) {
        if (n > capacity)
            return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_free_queue: %d > capacity %d", n,
                                capacity);
        int i = 0;
        for (int32_t id : p->free_q) out[i++] = id;
    }
    return KV_OK;
}

kv_status_t kv_prefix_pool_cache_size(const kv_prefix_pool_t* p, int* hashes_out,
                                      int* blocks_out) {
    if (!p) return report_error(KV_ERR_INVALID_ARG, "kv_prefix_pool_cache_size: null pool");
    int nb = 0;
    for (const auto& kv : p->cached) nb += static_cast<int>(kv.second.size());
    if (hashes_out) *hashes_out = static_cast<int>(p->cached.size());
    if (blocks_out) *blocks_out = nb;
    return KV_OK;
}

}  // extern "C"
