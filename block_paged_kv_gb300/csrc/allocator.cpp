// Host block allocator for the paged K/V pools ("paged-cache.md": the
// BlockAllocator row of the component table, the PagedKVCacheAdapter
// per-request lifecycle, the grow-on-demand rule of the pool-sizing passage).
//
// State per block: refcount, published hash (if any), and membership of the
// free set (ordered: the lowest id is handed out first) or of the LRU list of
// cache-only blocks (published, refcount 0, in release order).  The prefix
// table maps a block hash to the block holding it.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <list>
#include <set>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

// FNV-1a, 64-bit: offset basis 14695981039346656037, prime 1099511628211
struct Fnv1a {
    uint64_t h = 14695981039346656037ull;
    void bytes(const void *p, size_t n)
    {
        const unsigned char *b = static_cast<const unsigned char *>(p);
        for (size_t i = 0; i < n; ++i) {
            h ^= b[i];
            h *= 1099511628211ull;
        }
    }
    void u64(uint64_t v)
    {
        unsigned char b[8];
        for (int i = 0; i < 8; ++i) b[i] = static_cast<unsigned char>(v >> (8 * i));
        bytes(b, 8);
    }
    void i32(int32_t v)
    {
        const uint32_t u = static_cast<uint32_t>(v);
        unsigned char b[4];
        for (int i = 0; i < 4; ++i) b[i] = static_cast<unsigned char>(u >> (8 * i));
        bytes(b, 4);
    }
};

uint64_t block_hash(uint64_t parent, const int32_t *tokens, int32_t bs, uint64_t extra)
{
    Fnv1a f;
    f.u64(parent);
    for (int32_t i = 0; i < bs; ++i) f.i32(tokens[i]);
    f.u64(extra);
    return f.h;
}

struct Block {
    int32_t refcount = 0;
    bool published = false;
    uint64_t hash = 0;
    bool cached = false;  // on the LRU list
    std::list<int32_t>::iterator lru_it;
};

struct Request {
    std::vector<int32_t> table;
    std::vector<uint64_t> hashes;  // hash chain of the table's full blocks seen so far
    int32_t published = 0;         // leading table blocks already handled by publish
    bool fresh = true;             // nothing looked up or reserved yet
};

}  // namespace

struct pkv_allocator {
    int32_t bs = 16, max_blocks = 0, grows = 0, next_req = 0;
    std::vector<Block> blocks;
    std::set<int32_t> free_set;
    std::list<int32_t> lru;  // front = least recently released
    std::unordered_map<uint64_t, int32_t> table;
    std::unordered_map<int32_t, Request> reqs;

    int32_t num_blocks() const { return static_cast<int32_t>(blocks.size()); }

    void grow_to(int32_t n)
    {
        for (int32_t b = num_blocks(); b < n; ++b) free_set.insert(b);
        blocks.resize(static_cast<size_t>(n));
        ++grows;
    }

    // one reference less; at zero a published block becomes cache-only (LRU
    // tail), any other block free
    void drop_ref(int32_t b)
    {
        Block &blk = blocks[b];
        if (--blk.refcount > 0) return;
        if (blk.published) {
            blk.cached = true;
            blk.lru_it = lru.insert(lru.end(), b);
        } else {
            free_set.insert(b);
        }
    }

    void evict_one()
    {
        const int32_t b = lru.front();
        lru.pop_front();
        Block &blk = blocks[b];
        blk.cached = false;
        table.erase(blk.hash);
        blk.published = false;
        free_set.insert(b);
    }

    // k more blocks for a request, or false with nothing changed
    bool take(int32_t k, std::vector<int32_t> &out)
    {
        const int32_t nfree = static_cast<int32_t>(free_set.size());
        if (k > nfree) {
            const int32_t ncached = static_cast<int32_t>(lru.size());
            const int32_t cur = num_blocks();
            if (k > nfree + ncached && cur < max_blocks) {
                // grow before evicting: double, or straight to what is needed
                const int64_t want = std::max<int64_t>(2ll * cur, static_cast<int64_t>(cur) + (k - nfree));
                grow_to(static_cast<int32_t>(std::min<int64_t>(want, max_blocks)));
            }
            const int32_t avail = static_cast<int32_t>(free_set.size() + lru.size());
            if (k > avail) return false;
            while (static_cast<int32_t>(free_set.size()) < k) evict_one();
        }
        for (int32_t i = 0; i < k; ++i) {
            const int32_t b = *free_set.begin();
            free_set.erase(free_set.begin());
            blocks[b].refcount = 1;
            out.push_back(b);
        }
        return true;
    }
};

extern "C" {

pkv_allocator *pkv_allocator_create(int32_t block_size, int32_t initial_blocks, int32_t max_blocks)
{
    if (block_size <= 0 || initial_blocks < 0 || max_blocks < initial_blocks) return nullptr;
    pkv_allocator *a = new pkv_allocator();
    a->bs = block_size;
    a->max_blocks = max_blocks;
    a->blocks.resize(static_cast<size_t>(initial_blocks));
    for (int32_t b = 0; b < initial_blocks; ++b) a->free_set.insert(b);
    return a;
}

void pkv_allocator_destroy(pkv_allocator *a) { delete a; }

int32_t pkv_allocator_begin(pkv_allocator *a)
{
    if (a == nullptr) return -1;
    const int32_t id = a->next_req++;
    a->reqs.emplace(id, Request{});
    return id;
}

pkv_status pkv_allocator_find_cached_prefix(pkv_allocator *a, int32_t req, const int32_t *tokens,
                                            int32_t n_tokens, const uint64_t *extra_keys,
                                            int32_t *cached_tokens)
{
    if (a == nullptr || cached_tokens == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
        return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end() || !it->second.fresh) return PKV_ERR_INVALID_ARG;
    Request &r = it->second;
    r.fresh = false;
    const int32_t nfull = n_tokens / a->bs;
    uint64_t parent = 0;
    for (int32_t i = 0; i < nfull; ++i) {
        const uint64_t h = block_hash(parent, tokens + static_cast<int64_t>(i) * a->bs, a->bs,
                                      extra_keys ? extra_keys[i] : 0);
        auto f = a->table.find(h);
        if (f == a->table.end()) break;
        Block &blk = a->blocks[f->second];
        if (blk.cached) {
            a->lru.erase(blk.lru_it);
            blk.cached = false;
        }
        ++blk.refcount;
        r.table.push_back(f->second);
        r.hashes.push_back(h);
        parent = h;
    }
    r.published = static_cast<int32_t>(r.table.size());  // hits are published already
    *cached_tokens = static_cast<int32_t>(r.table.size()) * a->bs;
    return PKV_OK;
}

pkv_status pkv_allocator_reserve(pkv_allocator *a, int32_t req, int32_t n_tokens)
{
    if (a == nullptr || n_tokens < 0) return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end()) return PKV_ERR_INVALID_ARG;
    Request &r = it->second;
    r.fresh = false;
    const int64_t need_blocks = (static_cast<int64_t>(n_tokens) + a->bs - 1) / a->bs;
    const int64_t k = need_blocks - static_cast<int64_t>(r.table.size());
    if (k <= 0) return PKV_OK;
    if (k > INT32_MAX) return PKV_ERR_OUT_OF_BLOCKS;
    std::vector<int32_t> got;
    if (!a->take(static_cast<int32_t>(k), got)) return PKV_ERR_OUT_OF_BLOCKS;
    r.table.insert(r.table.end(), got.begin(), got.end());
    return PKV_OK;
}

pkv_status pkv_allocator_publish(pkv_allocator *a, int32_t req, const int32_t *tokens,
                                 int32_t n_tokens, const uint64_t *extra_keys)
{
    if (a == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
        return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end()) return PKV_ERR_INVALID_ARG;
    Request &r = it->second;
    const int64_t nfull = n_tokens / a->bs;
    if (nfull > static_cast<int64_t>(r.table.size())) return PKV_ERR_INVALID_ARG;
    for (int32_t i = r.published; i < nfull; ++i) {
        const uint64_t parent = i > 0 ? r.hashes[i - 1] : 0;
        const uint64_t h = block_hash(parent, tokens + static_cast<int64_t>(i) * a->bs, a->bs,
                                      extra_keys ? extra_keys[i] : 0);
        r.hashes.push_back(h);
        const int32_t b = r.table[i];
        if (b >= 0 && a->table.find(h) == a->table.end()) {  // an expired entry: chain only
            a->table.emplace(h, b);
            a->blocks[b].published = true;
            a->blocks[b].hash = h;
        }
    }
    if (nfull > r.published) r.published = static_cast<int32_t>(nfull);
    return PKV_OK;
}

pkv_status pkv_allocator_expire(pkv_allocator *a, int32_t req, int32_t first_live_token)
{
    if (a == nullptr || first_live_token < 0) return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end()) return PKV_ERR_INVALID_ARG;
    std::vector<int32_t> &t = it->second.table;
    const int64_t n = std::min<int64_t>(first_live_token / a->bs, static_cast<int64_t>(t.size()));
    for (int64_t i = 0; i < n; ++i) {
        if (t[i] < 0) continue;
        a->drop_ref(t[i]);
        t[i] = -1;
    }
    return PKV_OK;
}

pkv_status pkv_allocator_release(pkv_allocator *a, int32_t req)
{
    if (a == nullptr) return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end()) return PKV_ERR_INVALID_ARG;
    for (const int32_t b : it->second.table)
        if (b >= 0) a->drop_ref(b);
    a->reqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_allocator_table(const pkv_allocator *a, int32_t req, int32_t *out, int32_t cap,
                               int32_t *n_blocks)
{
    if (a == nullptr || n_blocks == nullptr || cap < 0 || (cap > 0 && out == nullptr))
        return PKV_ERR_INVALID_ARG;
    auto it = a->reqs.find(req);
    if (it == a->reqs.end()) return PKV_ERR_INVALID_ARG;
    const std::vector<int32_t> &t = it->second.table;
    const size_t n = std::min<size_t>(t.size(), static_cast<size_t>(cap));
    if (n > 0) std::memcpy(out, t.data(), n * sizeof(int32_t));
    *n_blocks = static_cast<int32_t>(t.size());
    return PKV_OK;
}

int32_t pkv_allocator_refcount(const pkv_allocator *a, int32_t block)
{
    if (a == nullptr || block < 0 || block >= a->num_blocks()) return -1;
    return a->blocks[block].refcount;
}

pkv_status pkv_allocator_stats(const pkv_allocator *a, int32_t *num_blocks, int32_t *free_blocks,
                               int32_t *cached_blocks, int32_t *grows)
{
    if (a == nullptr) return PKV_ERR_INVALID_ARG;
    if (num_blocks) *num_blocks = a->num_blocks();
    if (free_blocks) *free_blocks = static_cast<int32_t>(a->free_set.size());
    if (cached_blocks) *cached_blocks = static_cast<int32_t>(a->lru.size());
    if (grows) *grows = a->grows;
    return PKV_OK;
}

}  // extern "C"
