// prefix_cache.cpp -- block-hash prefix cache with LRU eviction of leaves, on
// top of the block pool (host only).
//
// A finished request's full blocks stay cached so that a later request with
// the same leading tokens reuses their K/V ("PagedAttention, chunked prefill,
// and the launch that cascades", opening section; "Waste, and three ways to
// reclaim it", "SGLang -- RadixAttention" and "Block sharing versus prefix
// caching?").  Matching is exact and block-aligned from the first token, keyed
// per tenant ("Waste, and three ways to reclaim it", fast answers and "The
// isolation question").
//
// Structure: every cached block is a node whose parent is the cached block
// before it in the same prefix, so the nodes form a tree of shared beginnings
// with 16-token edges.  A node is found through a hash index on its chain hash
// (the parent's chain hash folded with the block's 16 token ids; the root seed
// is derived from the tenant key); a candidate counts only if its parent node,
// tenant key and 16 tokens are equal to the query's, so collisions cost a
// compare, never a wrong block.  Leaves live in an ordered set keyed by
// (last use, creation serial): eviction walks it from the oldest end, skipping
// leaves a running request still holds (pool refcount > 1).
#include <cstring>
#include <mutex>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>
#include <algorithm>

#include "../../include/pagedkv.h"

namespace {

constexpr int BS = 16;

// FNV-1a over the 16 token ids, seeded with the parent's chain hash, then the
// SplitMix64 finaliser for avalanche.  Not cryptographic: exactness comes from
// the token compare.
inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

inline uint64_t chain_hash(uint64_t parent, const int32_t *tok)
{
    uint64_t h = parent ^ 0xcbf29ce484222325ull;
    for (int i = 0; i < BS; ++i) {
        h ^= static_cast<uint32_t>(tok[i]);
        h *= 0x100000001b3ull;
    }
    return mix64(h);
}

inline uint64_t root_seed(uint64_t salt) { return mix64(salt + 0x9e3779b97f4a7c15ull); }

struct Node {
    uint64_t hash = 0;
    uint64_t salt = 0;
    uint64_t tick = 0;
    uint64_t serial = 0;
    int32_t parent = -1;
    int32_t block = -1;
    int32_t children = 0;
    int32_t depth = 0;
    int32_t tok[BS];
    bool live = false;
};

using LeafKey = std::tuple<uint64_t, uint64_t, int32_t>;   // (tick, serial, node)

}  // namespace

struct kv_prefix_cache {
    kv_pool *pool = nullptr;
    std::vector<Node> nodes;
    std::vector<int32_t> free_nodes;
    std::unordered_multimap<uint64_t, int32_t> index;
    std::set<LeafKey> leaves;
    uint64_t clock = 0, serial = 0;
    int64_t lookups = 0, query_blocks = 0, hit_blocks = 0, inserted_blocks = 0, evicted_blocks = 0;
    int32_t cached = 0;
    mutable std::mutex mu;
};

namespace {

LeafKey leaf_key(const kv_prefix_cache *c, int32_t i)
{
    const Node &n = c->nodes[i];
    return LeafKey(n.tick, n.serial, i);
}

int32_t find(const kv_prefix_cache *c, uint64_t h, int32_t parent, uint64_t salt, const int32_t *tok)
{
    auto r = c->index.equal_range(h);
    for (auto it = r.first; it != r.second; ++it) {
        const Node &n = c->nodes[it->second];
        if (n.parent == parent && n.salt == salt && std::memcmp(n.tok, tok, sizeof n.tok) == 0) return it->second;
    }
    return -1;
}

void touch(kv_prefix_cache *c, int32_t i)
{
    Node &n = c->nodes[i];
    if (n.tick == c->clock) return;
    if (n.children == 0) c->leaves.erase(leaf_key(c, i));
    n.tick = c->clock;
    if (n.children == 0) c->leaves.insert(leaf_key(c, i));
}

int32_t refcount(const kv_prefix_cache *c, int32_t block)
{
    int32_t r = 0;
    if (kv_block_refcount(c->pool, block, &r) != KV_OK) return -1;
    return r;
}

// frees up to n blocks; ids to out (nullable).  Caller holds the mutex.
int32_t evict_locked(kv_prefix_cache *c, int32_t n, int32_t *out)
{
    int32_t freed = 0;
    auto it = c->leaves.begin();
    while (freed < n && it != c->leaves.end()) {
        const int32_t i = std::get<2>(*it);
        Node &nd = c->nodes[i];
        if (refcount(c, nd.block) != 1) {   // a running request still holds it
            ++it;
            continue;
        }
        it = c->leaves.erase(it);
        auto r = c->index.equal_range(nd.hash);
        for (auto jt = r.first; jt != r.second; ++jt)
            if (jt->second == i) {
                c->index.erase(jt);
                break;
            }
        const int32_t b = nd.block;
        kv_block_free(c->pool, &b, 1);
        if (out) out[freed] = b;
        ++freed;
        --c->cached;
        nd.live = false;
        c->free_nodes.push_back(i);
        if (nd.parent >= 0) {
            Node &p = c->nodes[nd.parent];
            if (--p.children == 0) {
                // the parent becomes a leaf; every leaf before the cursor was
                // skipped as in use, so resume at the parent if it sorts earlier
                auto pit = c->leaves.insert(leaf_key(c, nd.parent)).first;
                if (it == c->leaves.end() || *pit < *it) it = pit;
            }
        }
    }
    c->evicted_blocks += freed;
    return freed;
}

}  // namespace

extern "C" {

kv_status kv_prefix_cache_create(kv_pool *pool, kv_prefix_cache **out)
{
    if (!pool || !out) return KV_ERR_INVALID;
    auto *c = new (std::nothrow) kv_prefix_cache();
    if (!c) return KV_ERR_OUT_OF_BLOCKS;
    c->pool = pool;
    *out = c;
    return KV_OK;
}

void kv_prefix_cache_destroy(kv_prefix_cache *c)
{
    if (!c) return;
    {
        std::lock_guard<std::mutex> g(c->mu);
        for (const Node &n : c->nodes)
            if (n.live) kv_block_free(c->pool, &n.block, 1);
    }
    delete c;
}

kv_status kv_prefix_match(kv_prefix_cache *c, const int32_t *tokens, int32_t n_tokens, uint64_t salt,
                          int32_t max_blocks, int32_t *out_block_ids, int32_t *out_n_blocks)
{
    if (!c || n_tokens < 0 || max_blocks < 0 || !out_n_blocks || (n_tokens > 0 && !tokens) ||
        (max_blocks > 0 && !out_block_ids))
        return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(c->mu);
    const int32_t nfull = std::min(n_tokens / BS, max_blocks);
    ++c->clock;
    std::vector<int32_t> path;
    int32_t parent = -1;
    uint64_t h = root_seed(salt);
    for (int32_t j = 0; j < nfull; ++j) {
        const int32_t *tok = tokens + (size_t)j * BS;
        const uint64_t hj = chain_hash(h, tok);
        const int32_t i = find(c, hj, parent, salt, tok);
        if (i < 0) break;
        path.push_back(i);
        parent = i;
        h = hj;
    }
    for (size_t k = 0; k < path.size(); ++k) out_block_ids[k] = c->nodes[path[k]].block;
    if (!path.empty()) {
        const kv_status st = kv_block_share(c->pool, out_block_ids, (int32_t)path.size());
        if (st != KV_OK) return st;   // cannot happen: the cache holds each block
    }
    for (int32_t i : path) touch(c, i);
    c->lookups++;
    c->query_blocks += nfull;
    c->hit_blocks += (int64_t)path.size();
    *out_n_blocks = (int32_t)path.size();
    return KV_OK;
}

kv_status kv_prefix_insert(kv_prefix_cache *c, const int32_t *tokens, int32_t n_tokens, uint64_t salt,
                           const int32_t *block_ids, int32_t n_blocks, int32_t *out_n_new)
{
    if (!c || n_tokens < 0 || n_blocks < 0 || (n_tokens > 0 && !tokens) || (n_blocks > 0 && !block_ids))
        return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(c->mu);
    const int32_t n = std::min(n_tokens / BS, n_blocks);
    for (int32_t j = 0; j < n; ++j)
        if (refcount(c, block_ids[j]) < 1) return KV_ERR_INVALID;
    ++c->clock;
    int32_t parent = -1, fresh = 0;
    uint64_t h = root_seed(salt);
    for (int32_t j = 0; j < n; ++j) {
        const int32_t *tok = tokens + (size_t)j * BS;
        const uint64_t hj = chain_hash(h, tok);
        int32_t i = find(c, hj, parent, salt, tok);
        if (i >= 0) {
            touch(c, i);
        } else {
            if (kv_block_share(c->pool, block_ids + j, 1) != KV_OK) return KV_ERR_INVALID;
            if (c->free_nodes.empty()) {
                c->nodes.emplace_back();
                i = (int32_t)c->nodes.size() - 1;
            } else {
                i = c->free_nodes.back();
                c->free_nodes.pop_back();
            }
            Node &nd = c->nodes[i];
            nd.hash = hj;
            nd.salt = salt;
            nd.tick = c->clock;
            nd.serial = c->serial++;
            nd.parent = parent;
            nd.block = block_ids[j];
            nd.children = 0;
            nd.depth = parent >= 0 ? c->nodes[parent].depth + 1 : 0;
            std::memcpy(nd.tok, tok, sizeof nd.tok);
            nd.live = true;
            if (parent >= 0 && c->nodes[parent].children++ == 0) c->leaves.erase(leaf_key(c, parent));
            c->leaves.insert(leaf_key(c, i));
            c->index.emplace(hj, i);
            ++c->cached;
            ++fresh;
        }
        parent = i;
        h = hj;
    }
    c->inserted_blocks += fresh;
    if (out_n_new) *out_n_new = fresh;
    return KV_OK;
}

kv_status kv_prefix_evict(kv_prefix_cache *c, int32_t n, int32_t *out_ids, int32_t *out_n)
{
    if (!c || n < 0) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(c->mu);
    const int32_t f = evict_locked(c, n, out_ids);
    if (out_n) *out_n = f;
    return KV_OK;
}

kv_status kv_prefix_alloc(kv_prefix_cache *c, int32_t n, int32_t *out_ids)
{
    if (!c || n < 0 || (n > 0 && !out_ids)) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(c->mu);
    kv_pool_stats_t ps;
    if (kv_pool_stats(c->pool, &ps) != KV_OK) return KV_ERR_INVALID;
    if (n > ps.free_blocks) evict_locked(c, n - ps.free_blocks, nullptr);
    return kv_block_alloc(c->pool, n, out_ids);
}

kv_status kv_prefix_stats(const kv_prefix_cache *c, kv_prefix_stats_t *out)
{
    if (!c || !out) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(c->mu);
    out->lookups = c->lookups;
    out->query_blocks = c->query_blocks;
    out->hit_blocks = c->hit_blocks;
    out->inserted_blocks = c->inserted_blocks;
    out->evicted_blocks = c->evicted_blocks;
    out->cached_blocks = c->cached;
    // evictable now or after the blocks below it: refcount 1 and every child
    // evictable; visit the deepest nodes first
    std::vector<int32_t> order;
    order.reserve(c->cached);
    for (int32_t i = 0; i < (int32_t)c->nodes.size(); ++i)
        if (c->nodes[i].live) order.push_back(i);
    std::sort(order.begin(), order.end(),
              [&](int32_t a, int32_t b) { return c->nodes[a].depth > c->nodes[b].depth; });
    std::vector<int32_t> blocked(c->nodes.size(), 0);
    int32_t ev = 0;
    for (int32_t i : order) {
        const bool ok = blocked[i] == 0 && refcount(c, c->nodes[i].block) == 1;
        if (ok) ++ev;
        else if (c->nodes[i].parent >= 0) blocked[c->nodes[i].parent]++;
    }
    out->evictable_blocks = ev;
    return KV_OK;
}

}  // extern "C"
