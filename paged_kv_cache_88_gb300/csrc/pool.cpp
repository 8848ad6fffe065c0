// Host block allocator of libpkv: a fixed pool of N blocks with a FIFO free
// queue, a refcount per block and the append-slot / copy-on-write step.
//
// hnwysp.cn/news/103996 §3.2 and §4.1 carve the pool once and thread every
// block onto the free list; §3.4 takes blocks from the head of the free queue
// and returns them to its tail; §3.3 and §4.4 keep a refcount per block and
// recycle a block only when the count reaches zero; §3.3 copies a shared block
// before writing into it. m.lqnn.cn/news/240480 §3.2 step 3 gives the new
// token's place: the current page while it has room, else a fresh page.
//
// One pool is driven by one host thread at a time (the caller serialises); the
// lock-free multi-process queue of hnwysp.cn/news/103996 §3.4 is not needed for
// one process per GPU.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "pkv_internal.h"

namespace {
thread_local std::string g_last_error;
}

namespace pkv {

pkv_status fail(pkv_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

void clear_error() { g_last_error.clear(); }

}  // namespace pkv

using pkv::fail;

namespace {

// ---- free queue (doubly linked list over block ids) --------------------------

inline void q_push_back(pkv_pool *p, int32_t b) {
    p->next[b] = -1;
    p->prev[b] = p->tail;
    if (p->tail >= 0) p->next[p->tail] = b; else p->head = b;
    p->tail = b;
    p->count += 1;
}

inline void q_push_front(pkv_pool *p, int32_t b) {
    p->prev[b] = -1;
    p->next[b] = p->head;
    if (p->head >= 0) p->prev[p->head] = b; else p->tail = b;
    p->head = b;
    p->count += 1;
}

inline void q_remove(pkv_pool *p, int32_t b) {
    if (p->prev[b] >= 0) p->next[p->prev[b]] = p->next[b]; else p->head = p->next[b];
    if (p->next[b] >= 0) p->prev[p->next[b]] = p->prev[b]; else p->tail = p->prev[b];
    p->next[b] = p->prev[b] = -1;
    p->count -= 1;
}

// A block leaving the free queue for reuse loses its cached prefix hash (LRU
// eviction: the queue holds freed blocks in the order they were freed).
struct Evicted {
    int32_t block;
    uint64_t hash;
};

inline void drop_hash(pkv_pool *p, int32_t b, std::vector<Evicted> *log) {
    if (!p->has_hash[b]) return;
    auto it = p->by_hash.find(p->hash_of[b]);
    if (it != p->by_hash.end() && it->second == b) p->by_hash.erase(it);
    if (log) log->push_back({b, p->hash_of[b]});
    p->has_hash[b] = 0;
    p->evictions += 1;
}

inline int32_t q_pop_front(pkv_pool *p, std::vector<Evicted> *log = nullptr) {
    const int32_t b = p->head;
    q_remove(p, b);
    drop_hash(p, b, log);
    return b;
}

pkv_status check_desc(const pkv_pool_desc *d) {
    if (!d) return fail(PKV_ERR_INVALID_ARG, "desc is NULL");
    if (d->num_layers < 1 || d->num_blocks < 1 || d->num_heads < 1)
        return fail(PKV_ERR_INVALID_ARG, "num_layers, num_blocks and num_heads must be >= 1");
    if (!pkv::supported_block_size(d->block_size))
        return fail(PKV_ERR_UNSUPPORTED, "block_size %d not supported (8..512, power of two)", d->block_size);
    if (!pkv::supported_head_dim(d->head_dim))
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", d->head_dim);
    if (d->layout != PKV_LAYOUT_NHD && d->layout != PKV_LAYOUT_HND)
        return fail(PKV_ERR_INVALID_ARG, "layout %d unknown", d->layout);
    if ((int64_t)d->num_blocks * d->block_size * d->num_heads >= (int64_t)1 << 31)
        return fail(PKV_ERR_INVALID_ARG, "num_blocks * block_size * num_heads must be < 2^31");
    if (d->kv_dtype != PKV_KV_F16 && d->kv_dtype != PKV_KV_E4M3)
        return fail(PKV_ERR_INVALID_ARG, "kv_dtype %d unknown", d->kv_dtype);
    if (d->kv_dtype == PKV_KV_E4M3 && d->head_dim > 128)
        return fail(PKV_ERR_UNSUPPORTED, "an E4M3 cache is built for head_dim 64 or 128");
    return PKV_OK;
}

}  // namespace

extern "C" {

const char *pkv_last_error(void) { return g_last_error.c_str(); }

int32_t pkv_version(void) { return 10000; }

pkv_status pkv_pool_create(const pkv_pool_desc *desc, void *k_pool, void *v_pool,
                           const int32_t *initial_free_order, pkv_pool **out) {
    pkv::clear_error();
    if (!out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if ((k_pool == nullptr) != (v_pool == nullptr))
        return fail(PKV_ERR_INVALID_ARG, "k_pool and v_pool must both be set or both be NULL");
    if (k_pool && ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15u))
        return fail(PKV_ERR_INVALID_ARG, "pool pointers must be 16-byte aligned");
    const int32_t N = desc->num_blocks;
    std::vector<int32_t> order(N);
    if (initial_free_order) {
        std::vector<char> seen(N, 0);
        for (int32_t i = 0; i < N; ++i) {
            int32_t b = initial_free_order[i];
            if (b < 0 || b >= N || seen[b])
                return fail(PKV_ERR_INVALID_ARG, "initial_free_order is not a permutation of 0..N-1");
            seen[b] = 1;
            order[i] = b;
        }
    } else {
        for (int32_t i = 0; i < N; ++i) order[i] = i;
    }
    pkv_pool *p = new (std::nothrow) pkv_pool;
    if (!p) return fail(PKV_ERR_INVALID_ARG, "host allocation failed");
    p->desc = *desc;
    p->k_pool = k_pool;
    p->v_pool = v_pool;
    p->k_scale = nullptr;
    p->v_scale = nullptr;
    p->next.assign(N, -1);
    p->prev.assign(N, -1);
    p->head = p->tail = -1;
    p->count = 0;
    for (int32_t i = 0; i < N; ++i) q_push_back(p, order[i]);
    p->refcount.assign(N, 0);
    p->cow_copies = 0;
    p->hash_of.assign(N, 0);
    p->has_hash.assign(N, 0);
    p->prefix_hits = p->prefix_misses = p->evictions = 0;
    *out = p;
    return PKV_OK;
}

pkv_status pkv_pool_set_scales(pkv_pool *pool, void *k_scale, void *v_scale) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (pool->desc.kv_dtype != PKV_KV_E4M3) return fail(PKV_ERR_INVALID_ARG, "not an E4M3 pool");
    if (!k_scale || !v_scale || ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 15u))
        return fail(PKV_ERR_INVALID_ARG, "scale pools must be non-NULL and 16-byte aligned");
    pool->k_scale = static_cast<float *>(k_scale);
    pool->v_scale = static_cast<float *>(v_scale);
    return PKV_OK;
}

pkv_status pkv_pool_destroy(pkv_pool *pool) {
    delete pool;
    return PKV_OK;
}

pkv_status pkv_pool_info(const pkv_pool *pool, pkv_pool_desc *desc, void **k_pool, void **v_pool) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (desc) *desc = pool->desc;
    if (k_pool) *k_pool = pool->k_pool;
    if (v_pool) *v_pool = pool->v_pool;
    return PKV_OK;
}

pkv_status pkv_alloc(pkv_pool *pool, int32_t n, int32_t *out_ids) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (n < 0 || (n > 0 && !out_ids)) return fail(PKV_ERR_INVALID_ARG, "bad count or output");
    if (n > pool->count)
        return fail(PKV_ERR_OUT_OF_BLOCKS, "want %d blocks, %d free", n, pool->count);
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = q_pop_front(pool);
        pool->refcount[id] = 1;
        out_ids[i] = id;
    }
    return PKV_OK;
}

pkv_status pkv_incref(pkv_pool *pool, const int32_t *ids, int32_t n) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (n < 0 || (n > 0 && !ids)) return fail(PKV_ERR_INVALID_ARG, "bad count or ids");
    const int32_t N = pool->desc.num_blocks;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= N) return fail(PKV_ERR_BAD_BLOCK, "block %d out of range", ids[i]);
    for (int32_t i = 0; i < n; ++i)
        if (pool->refcount[ids[i]] == 0) return fail(PKV_ERR_REFCOUNT, "block %d is free", ids[i]);
    for (int32_t i = 0; i < n; ++i) pool->refcount[ids[i]] += 1;
    return PKV_OK;
}

pkv_status pkv_free(pkv_pool *pool, const int32_t *ids, int32_t n) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (n < 0 || (n > 0 && !ids)) return fail(PKV_ERR_INVALID_ARG, "bad count or ids");
    const int32_t N = pool->desc.num_blocks;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= N) return fail(PKV_ERR_BAD_BLOCK, "block %d out of range", ids[i]);
    // check first (repeats count), then apply: all-or-nothing
    std::vector<int32_t> &rc = pool->refcount;
    int32_t i = 0;
    for (; i < n; ++i) {
        if (rc[ids[i]] <= 0) break;
        rc[ids[i]] -= 1;
    }
    if (i < n) {
        for (int32_t j = 0; j < i; ++j) rc[ids[j]] += 1;
        return fail(PKV_ERR_REFCOUNT, "block %d: refcount would go below zero", ids[i]);
    }
    // The decrements above already left the final counts; push the blocks whose
    // count reached 0, each at the point of the list where it reached 0.
    for (int32_t j = 0; j < n; ++j) rc[ids[j]] += 1;
    for (int32_t j = 0; j < n; ++j) {
        rc[ids[j]] -= 1;
        if (rc[ids[j]] == 0) q_push_back(pool, ids[j]);
    }
    return PKV_OK;
}

pkv_status pkv_refcount(const pkv_pool *pool, int32_t id, int32_t *out) {
    if (!pool || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (id < 0 || id >= pool->desc.num_blocks) return fail(PKV_ERR_BAD_BLOCK, "block %d out of range", id);
    *out = pool->refcount[id];
    return PKV_OK;
}

pkv_status pkv_get_stats(const pkv_pool *pool, pkv_stats *out) {
    if (!pool || !out) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    pkv_stats s{};
    s.free_blocks = pool->count;
    for (size_t b = 0; b < pool->refcount.size(); ++b) {
        const int32_t r = pool->refcount[b];
        if (r > 0) s.used_blocks += 1;
        if (r > 1) s.shared_blocks += 1;
        if (r > s.max_refcount) s.max_refcount = r;
        if (pool->has_hash[b]) {
            s.cached_blocks += 1;
            if (r == 0) s.cached_free_blocks += 1;
        }
    }
    s.cow_copies = pool->cow_copies;
    s.prefix_hits = pool->prefix_hits;
    s.prefix_misses = pool->prefix_misses;
    s.evictions = pool->evictions;
    *out = s;
    return PKV_OK;
}

// ---- prefix cache (icman.com.cn/news/78786 §3.2-§3.4; hnwysp.cn/news/103996 §4.3)

uint64_t pkv_block_hash(uint64_t parent, const int32_t *token_ids, int32_t n) {
    // 64-bit FNV-1a over the parent hash (8 bytes, little-endian) and then each
    // token id (4 bytes, little-endian, two's complement).
    uint64_t h = 0xcbf29ce484222325ull;
    auto mix = [&h](uint8_t byte) {
        h ^= byte;
        h *= 0x100000001b3ull;
    };
    for (int i = 0; i < 8; ++i) mix(static_cast<uint8_t>(parent >> (8 * i)));
    for (int32_t t = 0; t < n; ++t) {
        const uint32_t v = static_cast<uint32_t>(token_ids[t]);
        for (int i = 0; i < 4; ++i) mix(static_cast<uint8_t>(v >> (8 * i)));
    }
    return h;
}

pkv_status pkv_prompt_block_hashes(const int32_t *token_ids, int32_t num_tokens, int32_t block_size,
                                   uint64_t *out, int32_t capacity, int32_t *num_hashes) {
    if (!num_hashes) return fail(PKV_ERR_INVALID_ARG, "num_hashes is NULL");
    if (num_tokens < 0 || block_size < 1) return fail(PKV_ERR_INVALID_ARG, "bad token count or block size");
    const int32_t full = num_tokens / block_size;  // a partial last block has no hash
    if (full > 0 && (!token_ids || !out)) return fail(PKV_ERR_INVALID_ARG, "NULL token_ids or out");
    if (capacity < full) return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d full blocks", capacity, full);
    uint64_t parent = 0;  // the first block chains on 0
    for (int32_t i = 0; i < full; ++i) {
        parent = pkv_block_hash(parent, token_ids + (size_t)i * block_size, block_size);
        out[i] = parent;
    }
    *num_hashes = full;
    return PKV_OK;
}

pkv_status pkv_prefix_lookup(pkv_pool *pool, const uint64_t *hashes, int32_t n, int32_t *out_ids,
                             int32_t *num_hits) {
    if (!pool || !num_hits) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    if (n < 0 || (n > 0 && (!hashes || !out_ids))) return fail(PKV_ERR_INVALID_ARG, "bad count or arrays");
    int32_t i = 0;
    for (; i < n; ++i) {
        auto it = pool->by_hash.find(hashes[i]);
        if (it == pool->by_hash.end()) break;
        const int32_t b = it->second;
        if (pool->refcount[b] == 0) q_remove(pool, b);  // a cached free block comes back into use
        pool->refcount[b] += 1;
        out_ids[i] = b;
    }
    *num_hits = i;
    pool->prefix_hits += i;
    pool->prefix_misses += n - i;
    return PKV_OK;
}

pkv_status pkv_prefix_register(pkv_pool *pool, const uint64_t *hashes, const int32_t *ids, int32_t n) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (n < 0 || (n > 0 && (!hashes || !ids))) return fail(PKV_ERR_INVALID_ARG, "bad count or arrays");
    const int32_t N = pool->desc.num_blocks;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= N) return fail(PKV_ERR_BAD_BLOCK, "block %d out of range", ids[i]);
    for (int32_t i = 0; i < n; ++i)
        if (pool->refcount[ids[i]] == 0) return fail(PKV_ERR_REFCOUNT, "block %d is free", ids[i]);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t b = ids[i];
        const uint64_t h = hashes[i];
        if (pool->has_hash[b]) {
            if (pool->hash_of[b] == h) continue;
            auto old = pool->by_hash.find(pool->hash_of[b]);
            if (old != pool->by_hash.end() && old->second == b) pool->by_hash.erase(old);
            pool->has_hash[b] = 0;
        }
        if (pool->by_hash.count(h)) continue;  // another block already holds these tokens
        pool->by_hash[h] = b;
        pool->hash_of[b] = h;
        pool->has_hash[b] = 1;
    }
    return PKV_OK;
}

pkv_status pkv_free_queue(const pkv_pool *pool, int32_t *out, int32_t capacity, int32_t *count) {
    if (!pool || !count) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    *count = pool->count;
    if (capacity < pool->count || (pool->count > 0 && !out))
        return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d", capacity, pool->count);
    int32_t i = 0;
    for (int32_t b = pool->head; b >= 0; b = pool->next[b]) out[i++] = b;
    return PKV_OK;
}

pkv_status pkv_validate(const pkv_pool *pool) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const int32_t N = pool->desc.num_blocks;
    std::vector<char> inq(N, 0);
    int32_t seen = 0, last = -1;
    for (int32_t b = pool->head; b >= 0; b = pool->next[b]) {
        if (b >= N || inq[b] || seen >= N || pool->prev[b] != last)
            return fail(PKV_ERR_REFCOUNT, "free queue corrupt at position %d", seen);
        inq[b] = 1;
        last = b;
        seen += 1;
    }
    if (seen != pool->count || last != pool->tail) return fail(PKV_ERR_REFCOUNT, "free queue count/tail wrong");
    for (int32_t b = 0; b < N; ++b) {
        if (pool->refcount[b] < 0) return fail(PKV_ERR_REFCOUNT, "block %d refcount < 0", b);
        if ((pool->refcount[b] == 0) != (inq[b] != 0))
            return fail(PKV_ERR_REFCOUNT, "block %d: refcount %d but %s the free queue", b,
                        pool->refcount[b], inq[b] ? "in" : "not in");
        if (pool->has_hash[b]) {
            auto it = pool->by_hash.find(pool->hash_of[b]);
            if (it == pool->by_hash.end() || it->second != b)
                return fail(PKV_ERR_REFCOUNT, "block %d: cached hash not in the map", b);
        }
    }
    for (const auto &kv : pool->by_hash)
        if (kv.second < 0 || kv.second >= N || !pool->has_hash[kv.second] || pool->hash_of[kv.second] != kv.first)
            return fail(PKV_ERR_REFCOUNT, "prefix map entry without its block");
    return PKV_OK;
}

pkv_status pkv_prepare_append(pkv_pool *pool, int32_t num_seqs, int32_t *block_tables,
                              int32_t max_blocks, int32_t *context_lens, const int32_t *num_new,
                              int64_t *slot_mapping, int32_t slot_capacity, int32_t *num_slots,
                              int32_t *copy_pairs, int32_t pair_capacity, int32_t *num_pairs) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (num_seqs < 0 || max_blocks < 1 || !num_slots || !num_pairs)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes or NULL counts");
    if (num_seqs > 0 && (!block_tables || !context_lens))
        return fail(PKV_ERR_INVALID_ARG, "NULL tables or lengths");
    const int32_t B = pool->desc.block_size;
    const int32_t N = pool->desc.num_blocks;
    int64_t total = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t k = num_new ? num_new[s] : 1;
        if (k < 0) return fail(PKV_ERR_INVALID_ARG, "num_new[%d] < 0", s);
        if (context_lens[s] < 0) return fail(PKV_ERR_INVALID_ARG, "context_lens[%d] < 0", s);
        total += k;
    }
    if (total > slot_capacity || (total > 0 && !slot_mapping))
        return fail(PKV_ERR_INVALID_ARG, "slot capacity %d < %lld tokens", slot_capacity, (long long)total);

    // Undo log: every change is recorded so that a failure restores the state.
    struct TableEdit { int64_t at; int32_t old; };
    std::vector<int32_t> allocated;  // in pop order
    std::vector<Evicted> evicted;    // cached hashes dropped by those pops
    const int64_t evictions0 = pool->evictions;
    std::vector<int32_t> decrefs;
    std::vector<TableEdit> edits;
    std::vector<int32_t> lens0(context_lens, context_lens + num_seqs);
    const int64_t cow0 = pool->cow_copies;
    int32_t nslot = 0, npair = 0;
    pkv_status st = PKV_OK;

    auto take = [&](int32_t *id) -> bool {
        if (pool->count == 0) {
            st = fail(PKV_ERR_OUT_OF_BLOCKS, "free queue empty");
            return false;
        }
        *id = q_pop_front(pool, &evicted);
        pool->refcount[*id] = 1;
        allocated.push_back(*id);
        return true;
    };

    for (int32_t s = 0; s < num_seqs && st == PKV_OK; ++s) {
        const int32_t k = num_new ? num_new[s] : 1;
        int32_t *row = block_tables + (int64_t)s * max_blocks;
        for (int32_t i = 0; i < k; ++i) {
            const int32_t pos = context_lens[s];
            const int32_t logical = pos / B, offset = pos % B;
            if (logical >= max_blocks) {
                st = fail(PKV_ERR_INVALID_ARG, "sequence %d needs more than %d blocks", s, max_blocks);
                break;
            }
            if (offset == 0) {
                int32_t id;
                if (!take(&id)) break;
                edits.push_back({(int64_t)s * max_blocks + logical, row[logical]});
                row[logical] = id;
            } else {
                const int32_t cur = row[logical];
                if (cur < 0 || cur >= N || pool->refcount[cur] == 0) {
                    st = fail(PKV_ERR_BAD_BLOCK, "sequence %d logical block %d holds %d", s, logical, cur);
                    break;
                }
                if (pool->refcount[cur] > 1) {
                    if (npair >= pair_capacity || !copy_pairs) {
                        st = fail(PKV_ERR_INVALID_ARG, "copy pair capacity %d too small", pair_capacity);
                        break;
                    }
                    int32_t dst;
                    if (!take(&dst)) break;
                    copy_pairs[2 * npair] = cur;
                    copy_pairs[2 * npair + 1] = dst;
                    npair += 1;
                    pool->refcount[cur] -= 1;
                    decrefs.push_back(cur);
                    pool->cow_copies += 1;
                    edits.push_back({(int64_t)s * max_blocks + logical, cur});
                    row[logical] = dst;
                }
            }
            slot_mapping[nslot++] = (int64_t)row[logical] * B + offset;
            context_lens[s] = pos + 1;
        }
    }

    if (st != PKV_OK) {
        for (size_t j = edits.size(); j-- > 0;) block_tables[edits[j].at] = edits[j].old;
        for (int32_t r : decrefs) pool->refcount[r] += 1;
        for (size_t j = allocated.size(); j-- > 0;) {
            pool->refcount[allocated[j]] = 0;
            q_push_front(pool, allocated[j]);
        }
        for (const Evicted &e : evicted) {
            pool->hash_of[e.block] = e.hash;
            pool->has_hash[e.block] = 1;
            pool->by_hash[e.hash] = e.block;
        }
        pool->evictions = evictions0;
        for (int32_t s = 0; s < num_seqs; ++s) context_lens[s] = lens0[s];
        pool->cow_copies = cow0;
        *num_slots = 0;
        *num_pairs = 0;
        return st;
    }
    *num_slots = nslot;
    *num_pairs = npair;
    return PKV_OK;
}

}  // extern "C"
