// Host block manager: free pool, reference counts, copy-on-write and the
// parent-chained prefix hash (kgptalkie "Day 28: PagedAttention / vLLM":
// "Growth Needs Only Another Free Block", "Shared Blocks Must Not Be Changed
// in Place", "Prefix Sharing Is a Natural Extension"; zenaique "How does
// PagedAttention enable prefix sharing across requests ...": answer text,
// "Most common mistake", follow-ups on the parent hash and the cache key).
//
// Plain C++ bookkeeping that runs on the host between decode steps and hands
// the GPU three small arrays: the slot of each new token, the block tables,
// and the (src, dst) pairs to copy.  Semantics are spelled out in pa.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a(const uint8_t* p, size_t n, uint64_t h = kFnvOffset) {
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= kFnvPrime;
    }
    return h;
}

void put_le(std::vector<uint8_t>& buf, uint64_t v, int bytes) {
    for (int i = 0; i < bytes; ++i) buf.push_back(static_cast<uint8_t>(v >> (8 * i)));
}

// Hash of one full block chained to its parent's hash.
uint64_t chain_hash(uint64_t parent, uint64_t salt, const int32_t* tokens, int n) {
    std::vector<uint8_t> buf;
    buf.reserve(16 + 4 * static_cast<size_t>(n));
    put_le(buf, parent, 8);
    put_le(buf, salt, 8);
    for (int i = 0; i < n; ++i) put_le(buf, static_cast<uint32_t>(tokens[i]), 4);
    return fnv1a(buf.data(), buf.size());
}

struct Request {
    std::vector<int32_t> table;   // logical block -> physical block
    std::vector<int32_t> tokens;  // token ids held so far
    std::vector<uint64_t> hashes; // chained hash of each full block
    uint64_t salt = 0;
};

struct CacheEntry {
    int32_t block;
    int32_t parent;               // physical block of the previous logical block, -1 first
    std::vector<int32_t> tokens;
};

}  // namespace

struct pa_bm {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_fifo;
    std::vector<int32_t> refcount;
    std::unordered_map<uint64_t, CacheEntry> cache;      // hash -> cached block
    std::unordered_map<int32_t, uint64_t> block_key;     // cached block -> hash
    std::unordered_map<int, Request> requests;
    int next_id = 0;
    // Retention (off unless pa_bm_set_retention turns it on): a cached block
    // whose last user leaves stays in the hash table, evictable, in the order
    // the blocks were released (least recent first).
    bool retain = false;
    std::list<int32_t> evictable;
    std::unordered_map<int32_t, std::list<int32_t>::iterator> evict_pos;

    Request* find(int id) {
        auto it = requests.find(id);
        return it == requests.end() ? nullptr : &it->second;
    }

    void release(int32_t blk) {
        if (--refcount[blk] == 0) {
            auto it = block_key.find(blk);
            if (it != block_key.end()) {
                if (retain) {                   // keep it findable; reuse it last
                    evictable.push_back(blk);
                    evict_pos[blk] = std::prev(evictable.end());
                    return;
                }
                cache.erase(it->second);
                block_key.erase(it);
            }
            free_fifo.push_back(blk);
        }
    }

    // A block for new tokens: the free pool first, then the least recently
    // released cached block (which leaves the hash table).  False: none left,
    // nothing changed.
    bool take(int32_t* out) {
        if (!free_fifo.empty()) {
            *out = free_fifo.front();
            free_fifo.pop_front();
            return true;
        }
        if (evictable.empty()) return false;
        const int32_t b = evictable.front();
        evictable.pop_front();
        evict_pos.erase(b);
        auto it = block_key.find(b);
        cache.erase(it->second);
        block_key.erase(it);
        *out = b;
        return true;
    }

    // A cache hit on a block nobody holds: it is in use again.
    void revive(int32_t blk) {
        auto it = evict_pos.find(blk);
        if (it == evict_pos.end()) return;
        evictable.erase(it->second);
        evict_pos.erase(it);
    }

    int append(int id, int32_t token, int64_t* slot, int64_t* src, int64_t* dst) {
        Request* r = find(id);
        if (!r) return PA_ERR_UNKNOWN_REQUEST;
        const int B = block_size;
        const int64_t pos = static_cast<int64_t>(r->tokens.size());
        const int64_t logical = pos / B;
        const int64_t offset = pos % B;
        int32_t blk;
        *src = -1;
        *dst = -1;
        if (offset == 0) {
            if (!take(&blk)) return PA_ERR_NO_FREE_BLOCK;
            refcount[blk] = 1;
            r->table.push_back(blk);
        } else {
            blk = r->table[logical];
            if (refcount[blk] > 1) {           // another request still reads it: copy first
                int32_t fresh;
                if (!take(&fresh)) return PA_ERR_NO_FREE_BLOCK;
                refcount[blk] -= 1;
                refcount[fresh] = 1;
                r->table[logical] = fresh;
                *src = blk;
                *dst = fresh;
                blk = fresh;
            }
        }
        r->tokens.push_back(token);
        if (offset == B - 1) {                  // the block is now full: hash and register it
            const int32_t* toks = r->tokens.data() + logical * B;
            uint64_t parent = r->hashes.empty() ? 0 : r->hashes.back();
            uint64_t h = chain_hash(parent, r->salt, toks, B);
            r->hashes.push_back(h);
            if (cache.find(h) == cache.end()) {
                CacheEntry e;
                e.block = blk;
                e.parent = logical > 0 ? r->table[logical - 1] : -1;
                e.tokens.assign(toks, toks + B);
                cache.emplace(h, std::move(e));
                block_key[blk] = h;
            }
        }
        *slot = static_cast<int64_t>(blk) * B + offset;
        return PA_OK;
    }
};

extern "C" {

uint64_t pa_bm_fnv1a64(const uint8_t* data, size_t n) { return fnv1a(data, n); }

int pa_bm_create(int num_blocks, int block_size, const int32_t* free_order, pa_bm** out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
    pa_bm* bm = new (std::nothrow) pa_bm();
    if (!bm) return PA_ERR_OUT_OF_MEMORY;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refcount.assign(num_blocks, 0);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete bm;
                return PA_ERR_INVALID_ARG;
            }
            seen[b] = 1;
            bm->free_fifo.push_back(b);
        }
    } else {
        for (int i = 0; i < num_blocks; ++i) bm->free_fifo.push_back(i);
    }
    *out = bm;
    return PA_OK;
}

int pa_bm_destroy(pa_bm* bm) {
    delete bm;
    return PA_OK;
}

int pa_bm_add_request(pa_bm* bm, const int32_t* tokens, int n, uint64_t salt, int* req,
                      int* cached_tokens) {
    if (!bm || !req || n < 0 || (n > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    Request r;
    r.salt = salt;
    const int B = bm->block_size;
    uint64_t parent_hash = 0;
    int32_t parent_blk = -1;
    for (int i = 0; i < n / B; ++i) {
        const int32_t* toks = tokens + static_cast<int64_t>(i) * B;
        uint64_t h = chain_hash(parent_hash, salt, toks, B);
        auto it = bm->cache.find(h);
        if (it == bm->cache.end() || it->second.parent != parent_blk ||
            std::memcmp(it->second.tokens.data(), toks, sizeof(int32_t) * B) != 0)
            break;                                 // first miss ends the reuse
        int32_t blk = it->second.block;
        if (bm->refcount[blk] == 0) bm->revive(blk);
        bm->refcount[blk] += 1;
        r.table.push_back(blk);
        r.tokens.insert(r.tokens.end(), toks, toks + B);
        r.hashes.push_back(h);
        parent_hash = h;
        parent_blk = blk;
    }
    int id = bm->next_id++;
    if (cached_tokens) *cached_tokens = static_cast<int>(r.tokens.size());
    bm->requests.emplace(id, std::move(r));
    *req = id;
    return PA_OK;
}

int pa_bm_fork(pa_bm* bm, int parent, int* child) {
    if (!bm || !child) return PA_ERR_INVALID_ARG;
    Request* p = bm->find(parent);
    if (!p) return PA_ERR_UNKNOWN_REQUEST;
    for (int32_t b : p->table) bm->refcount[b] += 1;
    Request c = *p;
    int id = bm->next_id++;
    bm->requests.emplace(id, std::move(c));
    *child = id;
    return PA_OK;
}

int pa_bm_append_slot(pa_bm* bm, int req, int32_t token, int64_t* slot, int64_t* cow_src,
                      int64_t* cow_dst) {
    if (!bm || !slot || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
    return bm->append(req, token, slot, cow_src, cow_dst);
}

int pa_bm_append_slots(pa_bm* bm, int n, const int32_t* reqs, const int32_t* tokens,
                       int64_t* slots, int64_t* cow_pairs, int* num_pairs, int* num_done) {
    if (!bm || n < 0 || (n > 0 && (!reqs || !tokens || !slots || !cow_pairs)) || !num_pairs)
        return PA_ERR_INVALID_ARG;
    int pairs = 0, done = 0, rc = PA_OK;
    for (int i = 0; i < n; ++i) {
        int64_t src, dst;
        rc = bm->append(reqs[i], tokens[i], &slots[i], &src, &dst);
        if (rc != PA_OK) break;
        if (src >= 0) {
            cow_pairs[2 * pairs] = src;
            cow_pairs[2 * pairs + 1] = dst;
            ++pairs;
        }
        ++done;
    }
    *num_pairs = pairs;
    if (num_done) *num_done = done;
    return rc;
}

int pa_bm_free_request(pa_bm* bm, int req) {
    if (!bm) return PA_ERR_INVALID_ARG;
    Request* r = bm->find(req);
    if (!r) return PA_ERR_UNKNOWN_REQUEST;
    for (int32_t b : r->table)
        if (bm->refcount[b] <= 0) return PA_ERR_REFCOUNT;
    if (bm->retain) {
        // deepest block first, so a chain's leaves are evicted before its root
        for (auto it = r->table.rbegin(); it != r->table.rend(); ++it) bm->release(*it);
    } else {
        for (int32_t b : r->table) bm->release(b);
    }
    bm->requests.erase(req);
    return PA_OK;
}

int pa_bm_block_table(pa_bm* bm, int req, int32_t* out, int cap, int* n) {
    if (!bm || !n || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    Request* r = bm->find(req);
    if (!r) return PA_ERR_UNKNOWN_REQUEST;
    *n = static_cast<int>(r->table.size());
    for (int i = 0; i < *n && i < cap; ++i) out[i] = r->table[i];
    return PA_OK;
}

int pa_bm_batch_tables(pa_bm* bm, int n, const int32_t* reqs, int width, int32_t* tables,
                       int32_t* lens) {
    if (!bm || n < 0 || width < 0 || (n > 0 && (!reqs || !lens || (width > 0 && !tables))))
        return PA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        Request* r = bm->find(reqs[i]);
        if (!r) return PA_ERR_UNKNOWN_REQUEST;
        if (static_cast<int>(r->table.size()) > width) return PA_ERR_INVALID_ARG;
        int32_t* row = tables + static_cast<int64_t>(i) * width;
        std::copy(r->table.begin(), r->table.end(), row);
        std::fill(row + r->table.size(), row + width, -1);
        lens[i] = static_cast<int32_t>(r->tokens.size());
    }
    return PA_OK;
}

int pa_bm_batch_width(pa_bm* bm, int n, const int32_t* reqs, int* width) {
    if (!bm || n < 0 || !width || (n > 0 && !reqs)) return PA_ERR_INVALID_ARG;
    int w = 0;
    for (int i = 0; i < n; ++i) {
        const Request* r = bm->find(reqs[i]);
        if (!r) return PA_ERR_UNKNOWN_REQUEST;
        w = std::max(w, static_cast<int>(r->table.size()));
    }
    *width = w;
    return PA_OK;
}

int pa_bm_seq_len(pa_bm* bm, int req) {
    if (!bm) return -1;
    Request* r = bm->find(req);
    return r ? static_cast<int>(r->tokens.size()) : -1;
}

int pa_bm_refcount(pa_bm* bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[block];
}

int pa_bm_num_free(pa_bm* bm) { return bm ? static_cast<int>(bm->free_fifo.size()) : -1; }

int pa_bm_free_list(pa_bm* bm, int32_t* out, int cap, int* n) {
    if (!bm || !n || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    *n = static_cast<int>(bm->free_fifo.size());
    int i = 0;
    for (int32_t b : bm->free_fifo) {
        if (i >= cap) break;
        out[i++] = b;
    }
    return PA_OK;
}

int pa_bm_prefix_groups(pa_bm* bm, int n, const int32_t* reqs, int32_t* group_offsets,
                        int32_t* group_seqs, int32_t* group_shared_blocks, int* num_groups) {
    if (!bm || n < 0 || !num_groups || (n > 0 && (!reqs || !group_offsets || !group_seqs ||
                                                   !group_shared_blocks)))
        return PA_ERR_INVALID_ARG;
    std::vector<Request*> r(n);
    for (int i = 0; i < n; ++i) {
        r[i] = bm->find(reqs[i]);
        if (!r[i]) return PA_ERR_UNKNOWN_REQUEST;
    }
    // batch entries keyed by their first physical block, in batch order
    std::unordered_map<int32_t, std::vector<int>> by_first;
    std::vector<int32_t> order;
    for (int i = 0; i < n; ++i) {
        if (r[i]->table.empty() || static_cast<int>(r[i]->tokens.size()) < bm->block_size) continue;
        const int32_t b0 = r[i]->table[0];
        auto it = by_first.find(b0);
        if (it == by_first.end()) {
            order.push_back(b0);
            by_first[b0] = {i};
        } else {
            it->second.push_back(i);
        }
    }
    int ng = 0, pos = 0;
    group_offsets[0] = 0;
    for (int32_t b0 : order) {
        const std::vector<int>& m = by_first[b0];
        if (m.size() < 2) continue;
        // leading blocks that are the same physical block for every member and
        // full in every member's context
        size_t full = SIZE_MAX;
        for (int i : m) full = std::min(full, r[i]->tokens.size() / bm->block_size);
        size_t lcp = 0;
        while (lcp < full) {
            const int32_t b = r[m[0]]->table[lcp];
            bool same = true;
            for (int i : m) same = same && r[i]->table[lcp] == b;
            if (!same) break;
            ++lcp;
        }
        if (lcp == 0) continue;
        for (int i : m) group_seqs[pos++] = i;
        group_shared_blocks[ng] = static_cast<int32_t>(lcp);
        group_offsets[++ng] = pos;
    }
    *num_groups = ng;
    return PA_OK;
}

int pa_bm_set_retention(pa_bm* bm, int on) {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (!on) {                                  // retained blocks leave the table, join the pool
        for (int32_t b : bm->evictable) {
            auto it = bm->block_key.find(b);
            bm->cache.erase(it->second);
            bm->block_key.erase(it);
            bm->free_fifo.push_back(b);
        }
        bm->evictable.clear();
        bm->evict_pos.clear();
    }
    bm->retain = on != 0;
    return PA_OK;
}

int pa_bm_num_evictable(pa_bm* bm) { return bm ? static_cast<int>(bm->evictable.size()) : -1; }

int pa_bm_evictable_list(pa_bm* bm, int32_t* out, int cap, int* n) {
    if (!bm || !n || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    *n = static_cast<int>(bm->evictable.size());
    int i = 0;
    for (int32_t b : bm->evictable) {
        if (i >= cap) break;
        out[i++] = b;
    }
    return PA_OK;
}

int pa_bm_is_cached(pa_bm* bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->block_key.count(block) ? 1 : 0;
}

}  // extern "C"
