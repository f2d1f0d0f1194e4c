// Host-side block manager behind the pkv_pool_* / pkv_block_* / pkv_seq_*
// entry points of pkv.h.
//
// A flat pool of physical blocks handed out from a LIFO free stack, one
// reference count per block ("A Ideia de 60 Anos Que Domou a Memória da GPU",
// section "o código: a diferença entre reservar e mapear"), per-sequence block
// tables grown one block at a time when the tail fills (same page, section "a
// ideia roubada"), fork by sharing and copy-on-write of a partially filled
// shared tail ("The 8GB VRAM Breakthrough", §3 "Copy-on-Write (CoW) Prefix
// Sharing").  Appends count every block they need before touching anything,
// so a failure leaves the state unchanged.
//
// Prefix cache ("Capítulo 8 — Gerenciamento de KV Cache de Próxima Geração",
// §8.3: hash the prompt in block-sized chunks; a chunk already in the global
// cache of computed blocks is mapped into the new request's table and its
// prefill skipped; otherwise the prefill runs and the block is registered).
// An entry is one full block, keyed by its parent entry (the entry of the
// previous block, so equal chunks at different prefixes differ) and its
// block_size token ids; the 64-bit hash only buckets candidates, which are
// then compared exactly.  The cache holds one reference on each entry's
// block, so cached blocks outlive the sequences that computed them until
// evicted (least recently used first, leaves only, blocks no one else holds).

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace {

struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
};

struct PrefixEntry {
    int32_t block = -1;           // physical block (one reference held by the cache)
    int64_t parent = -1;          // entry of the previous block, -1 for the first
    std::vector<int32_t> tokens;  // the block's token ids
    uint64_t last_use = 0;        // LRU clock
    int32_t children = 0;         // entries whose parent is this one
};

// 64-bit hash of the parent id and the chunk's token ids: FNV-1a over
// 32-bit words (buckets only: candidates are compared exactly).
uint64_t chunk_hash(int64_t parent, const int32_t* tokens, int32_t n) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint32_t x) {
        h ^= x;
        h *= 1099511628211ull;
    };
    mix(static_cast<uint32_t>(static_cast<uint64_t>(parent)));
    mix(static_cast<uint32_t>(static_cast<uint64_t>(parent) >> 32));
    for (int32_t i = 0; i < n; ++i) mix(static_cast<uint32_t>(tokens[i]));
    return h ^ (h >> 29);
}

}  // namespace

struct pkv_pool {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_stack;  // back() is the next block handed out
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Seq> seqs;
    int64_t next_seq = 0;
    int64_t fail_after = -1;  // allocations left before injected failures

    // prefix cache
    std::unordered_map<int64_t, PrefixEntry> entries;
    std::unordered_multimap<uint64_t, int64_t> index;  // chunk hash -> entry
    int64_t next_entry = 0;
    uint64_t clock = 0;
    int64_t lookups = 0, hit_blocks = 0;

    // The entry for (parent, chunk), or -1.
    int64_t find_entry(int64_t parent, const int32_t* tokens) const {
        auto range = index.equal_range(chunk_hash(parent, tokens, block_size));
        for (auto it = range.first; it != range.second; ++it) {
            const PrefixEntry& e = entries.at(it->second);
            if (e.parent == parent &&
                std::memcmp(e.tokens.data(), tokens, sizeof(int32_t) * block_size) == 0)
                return it->second;
        }
        return -1;
    }

    void drop_entry(int64_t id) {
        PrefixEntry& e = entries.at(id);
        auto range = index.equal_range(chunk_hash(e.parent, e.tokens.data(), block_size));
        for (auto it = range.first; it != range.second; ++it) {
            if (it->second == id) {
                index.erase(it);
                break;
            }
        }
        if (e.parent >= 0) --entries.at(e.parent).children;
        decref(e.block);
        entries.erase(id);
    }

    // Blocks that can actually be allocated right now (injection included).
    int64_t allocatable() const {
        int64_t n = static_cast<int64_t>(free_stack.size());
        if (fail_after >= 0 && fail_after < n) n = fail_after;
        return n;
    }

    int32_t alloc_unchecked() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        if (fail_after > 0) --fail_after;
        return b;
    }

    int decref(int32_t b) {
        if (b < 0 || b >= num_blocks) return PKV_ERR_INVALID_ARG;
        if (ref[b] <= 0) return PKV_ERR_DOUBLE_FREE;
        if (--ref[b] == 0) free_stack.push_back(b);
        return PKV_OK;
    }

    // Blocks one append of n tokens to s needs (clone + growth).
    int64_t blocks_needed(const Seq& s, int64_t n) const {
        if (n <= 0) return 0;
        int64_t need = 0;
        if (s.len % block_size != 0 && ref[s.table.back()] > 1) need += 1;
        int64_t after = (s.len + n + block_size - 1) / block_size;
        need += after - static_cast<int64_t>(s.table.size());
        return need;
    }

    // Performs an append already known to fit.  Returns the number of copy
    // pairs written to pairs (0 or 1).
    int append_fitting(Seq& s, int32_t n, int64_t* slots, int32_t* pairs) {
        int copies = 0;
        if (n <= 0) return 0;
        if (s.len % block_size != 0 && ref[s.table.back()] > 1) {
            int32_t src = s.table.back();
            int32_t dst = alloc_unchecked();
            --ref[src];  // > 0 afterwards: it was shared
            s.table.back() = dst;
            if (pairs) {
                pairs[0] = src;
                pairs[1] = dst;
            }
            copies = 1;
        }
        for (int32_t i = 0; i < n; ++i) {
            if (s.len % block_size == 0) s.table.push_back(alloc_unchecked());
            slots[i] = static_cast<int64_t>(s.table[s.len / block_size]) * block_size +
                       s.len % block_size;
            ++s.len;
        }
        return copies;
    }
};

extern "C" {

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_OUT_OF_BLOCKS: return "out of blocks";
        case PKV_ERR_BAD_HANDLE: return "bad pool handle";
        case PKV_ERR_BAD_SEQ: return "unknown sequence";
        case PKV_ERR_DOUBLE_FREE: return "block already free";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_DEVICE_BOUNDS: return "device index out of bounds";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        default: return "unknown status";
    }
}

int pkv_version(void) { return 1; }

int pkv_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                    pkv_pool** out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_pool* p = new (std::nothrow) pkv_pool();
    if (!p) return PKV_ERR_INVALID_ARG;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->ref.assign(num_blocks, 0);
    p->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return PKV_ERR_INVALID_ARG;
            }
            seen[b] = 1;
            p->free_stack[num_blocks - 1 - i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) p->free_stack[num_blocks - 1 - i] = i;
    }
    *out = p;
    return PKV_OK;
}

int pkv_pool_destroy(pkv_pool* pool) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    delete pool;
    return PKV_OK;
}

int pkv_pool_num_free(const pkv_pool* pool, int32_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out) return PKV_ERR_INVALID_ARG;
    *out = static_cast<int32_t>(pool->free_stack.size());
    return PKV_OK;
}

int pkv_pool_num_blocks(const pkv_pool* pool, int32_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out) return PKV_ERR_INVALID_ARG;
    *out = pool->num_blocks;
    return PKV_OK;
}

int pkv_pool_block_size(const pkv_pool* pool, int32_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out) return PKV_ERR_INVALID_ARG;
    *out = pool->block_size;
    return PKV_OK;
}

int pkv_block_alloc(pkv_pool* pool, int32_t* block) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!block) return PKV_ERR_INVALID_ARG;
    if (pool->allocatable() < 1) return PKV_ERR_OUT_OF_BLOCKS;
    *block = pool->alloc_unchecked();
    return PKV_OK;
}

int pkv_block_incref(pkv_pool* pool, int32_t block) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (block < 0 || block >= pool->num_blocks) return PKV_ERR_INVALID_ARG;
    if (pool->ref[block] <= 0) return PKV_ERR_DOUBLE_FREE;
    ++pool->ref[block];
    return PKV_OK;
}

int pkv_block_decref(pkv_pool* pool, int32_t block) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    return pool->decref(block);
}

int pkv_block_refcount(const pkv_pool* pool, int32_t block, int32_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out || block < 0 || block >= pool->num_blocks) return PKV_ERR_INVALID_ARG;
    *out = pool->ref[block];
    return PKV_OK;
}

int pkv_seq_create(pkv_pool* pool, int64_t* seq) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!seq) return PKV_ERR_INVALID_ARG;
    int64_t id = pool->next_seq++;
    pool->seqs.emplace(id, Seq());
    *seq = id;
    return PKV_OK;
}

int pkv_seq_free(pkv_pool* pool, int64_t seq) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    for (int32_t b : it->second.table) {
        int st = pool->decref(b);
        if (st != PKV_OK) return st;  // only reachable if the state was corrupted
    }
    pool->seqs.erase(it);
    return PKV_OK;
}

int pkv_seq_fork(pkv_pool* pool, int64_t parent, int64_t* child) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!child) return PKV_ERR_INVALID_ARG;
    auto it = pool->seqs.find(parent);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    Seq s = it->second;  // copy the table first: emplace may rehash
    for (int32_t b : s.table) ++pool->ref[b];
    int64_t id = pool->next_seq++;
    pool->seqs.emplace(id, std::move(s));
    *child = id;
    return PKV_OK;
}

int pkv_seq_append(pkv_pool* pool, int64_t seq, int32_t n_tokens, int64_t* slots_out,
                   int32_t* copy_pairs_out, int32_t* n_copies) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PKV_ERR_INVALID_ARG;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    Seq& s = it->second;
    int64_t need = pool->blocks_needed(s, n_tokens);
    if (need > pool->allocatable()) return PKV_ERR_OUT_OF_BLOCKS;
    bool cow = n_tokens > 0 && s.len % pool->block_size != 0 && pool->ref[s.table.back()] > 1;
    if (cow && !copy_pairs_out) return PKV_ERR_INVALID_ARG;
    int c = pool->append_fitting(s, n_tokens, slots_out, copy_pairs_out);
    if (n_copies) *n_copies = c;
    return PKV_OK;
}

int pkv_seq_append_batch(pkv_pool* pool, const int64_t* seqs, int32_t n, int32_t n_tokens_each,
                         int64_t* slots_out, int32_t* copy_pairs_out, int32_t* n_copies) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (n < 0 || n_tokens_each < 0 || (n > 0 && (!seqs || !copy_pairs_out)) ||
        (n > 0 && n_tokens_each > 0 && !slots_out))
        return PKV_ERR_INVALID_ARG;
    std::vector<Seq*> ss(n);
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->seqs.find(seqs[i]);
        if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
        for (int32_t j = 0; j < i; ++j)
            if (ss[j] == &it->second) return PKV_ERR_INVALID_ARG;  // duplicates
        ss[i] = &it->second;
        need += pool->blocks_needed(it->second, n_tokens_each);
    }
    if (need > pool->allocatable()) return PKV_ERR_OUT_OF_BLOCKS;
    int total = 0;
    for (int32_t i = 0; i < n; ++i)
        total += pool->append_fitting(*ss[i], n_tokens_each,
                                      slots_out + static_cast<int64_t>(i) * n_tokens_each,
                                      copy_pairs_out + 2 * total);
    if (n_copies) *n_copies = total;
    return PKV_OK;
}

int pkv_seq_len(const pkv_pool* pool, int64_t seq, int64_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out) return PKV_ERR_INVALID_ARG;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    *out = it->second.len;
    return PKV_OK;
}

int pkv_seq_num_blocks(const pkv_pool* pool, int64_t seq, int32_t* out) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!out) return PKV_ERR_INVALID_ARG;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    *out = static_cast<int32_t>(it->second.table.size());
    return PKV_OK;
}

int pkv_seq_block_table(const pkv_pool* pool, int64_t seq, int32_t* out, int32_t capacity) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    const auto& t = it->second.table;
    if (capacity < 0 || static_cast<size_t>(capacity) < t.size() || (!out && !t.empty()))
        return PKV_ERR_INVALID_ARG;
    if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
    return PKV_OK;
}

int pkv_build_block_tables(const pkv_pool* pool, const int64_t* seqs, int32_t n, int32_t* tables,
                           int32_t max_blocks, int32_t* context_lens) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (n < 0 || max_blocks < 0 || (n > 0 && (!seqs || !context_lens)) ||
        (n > 0 && max_blocks > 0 && !tables))
        return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->seqs.find(seqs[i]);
        if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
        if (it->second.table.size() > static_cast<size_t>(max_blocks)) return PKV_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) {
        const Seq& s = pool->seqs.find(seqs[i])->second;
        int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
        size_t nb = s.table.size();
        for (size_t j = 0; j < nb; ++j) row[j] = s.table[j];
        for (int32_t j = static_cast<int32_t>(nb); j < max_blocks; ++j) row[j] = -1;
        context_lens[i] = static_cast<int32_t>(s.len);
    }
    return PKV_OK;
}

int pkv_prefix_register(pkv_pool* pool, int64_t seq, const int32_t* tokens, int32_t n_tokens,
                        int32_t* n_new) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (n_tokens < 0 || (n_tokens > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_BAD_SEQ;
    const Seq& s = it->second;
    if (n_tokens > s.len) return PKV_ERR_INVALID_ARG;
    const int32_t bs = pool->block_size;
    const int32_t full = n_tokens / bs;
    int32_t added = 0;
    int64_t parent = -1;
    for (int32_t i = 0; i < full; ++i) {
        const int32_t* chunk = tokens + static_cast<int64_t>(i) * bs;
        int64_t id = pool->find_entry(parent, chunk);
        if (id < 0) {
            // a new full block: the cache takes a reference on the sequence's block
            id = pool->next_entry++;
            PrefixEntry e;
            e.block = s.table[i];
            e.parent = parent;
            e.tokens.assign(chunk, chunk + bs);
            e.last_use = ++pool->clock;
            ++pool->ref[e.block];
            if (parent >= 0) ++pool->entries.at(parent).children;
            pool->index.emplace(chunk_hash(parent, chunk, bs), id);
            pool->entries.emplace(id, std::move(e));
            ++added;
        }
        parent = id;
    }
    if (n_new) *n_new = added;
    return PKV_OK;
}

int pkv_prefix_match(pkv_pool* pool, const int32_t* tokens, int32_t n_tokens, int64_t* seq_out,
                     int32_t* matched_tokens) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!seq_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
    const int32_t bs = pool->block_size;
    Seq s;
    int64_t parent = -1;
    const uint64_t now = ++pool->clock;
    for (int32_t i = 0; i < n_tokens / bs; ++i) {
        const int64_t id = pool->find_entry(parent, tokens + static_cast<int64_t>(i) * bs);
        if (id < 0) break;
        PrefixEntry& e = pool->entries.at(id);
        e.last_use = now;
        s.table.push_back(e.block);
        parent = id;
    }
    for (int32_t b : s.table) ++pool->ref[b];
    s.len = static_cast<int64_t>(s.table.size()) * bs;
    ++pool->lookups;
    pool->hit_blocks += static_cast<int64_t>(s.table.size());
    const int64_t id = pool->next_seq++;
    if (matched_tokens) *matched_tokens = static_cast<int32_t>(s.len);
    pool->seqs.emplace(id, std::move(s));
    *seq_out = id;
    return PKV_OK;
}

int pkv_prefix_evict(pkv_pool* pool, int32_t n_blocks, int32_t* n_freed) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (n_blocks < 0) return PKV_ERR_INVALID_ARG;
    int32_t freed = 0;
    while (freed < n_blocks) {
        // least recently used leaf whose block only the cache holds
        int64_t victim = -1;
        uint64_t oldest = 0;
        for (const auto& kv : pool->entries) {
            const PrefixEntry& e = kv.second;
            if (e.children != 0 || pool->ref[e.block] != 1) continue;
            if (victim < 0 || e.last_use < oldest || (e.last_use == oldest && kv.first < victim)) {
                victim = kv.first;
                oldest = e.last_use;
            }
        }
        if (victim < 0) break;
        pool->drop_entry(victim);
        ++freed;
    }
    if (n_freed) *n_freed = freed;
    return PKV_OK;
}

int pkv_prefix_clear(pkv_pool* pool) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    // release in registration order (the blocks return to the free stack in
    // a defined order)
    std::vector<int64_t> ids;
    ids.reserve(pool->entries.size());
    for (const auto& kv : pool->entries) ids.push_back(kv.first);
    std::sort(ids.begin(), ids.end());
    for (int64_t id : ids) pool->decref(pool->entries.at(id).block);
    pool->entries.clear();
    pool->index.clear();
    return PKV_OK;
}

int pkv_prefix_stats(const pkv_pool* pool, int64_t* entries, int64_t* lookups, int64_t* hit_blocks) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    if (!entries || !lookups || !hit_blocks) return PKV_ERR_INVALID_ARG;
    *entries = static_cast<int64_t>(pool->entries.size());
    *lookups = pool->lookups;
    *hit_blocks = pool->hit_blocks;
    return PKV_OK;
}

int pkv_debug_fail_after(pkv_pool* pool, int64_t n_allocs) {
    if (!pool) return PKV_ERR_BAD_HANDLE;
    pool->fail_after = n_allocs < 0 ? -1 : n_allocs;
    return PKV_OK;
}

}  // extern "C"
