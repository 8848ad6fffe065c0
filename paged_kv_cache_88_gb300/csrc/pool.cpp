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

inline int32_t ring_pop_front(pkv_pool *p) {
    int32_t id = p->ring[p->head];
    p->head = (p->head + 1) % p->desc.num_blocks;
    p->count -= 1;
    return id;
}

inline void ring_push_back(pkv_pool *p, int32_t id) {
    p->ring[(p->head + p->count) % p->desc.num_blocks] = id;
    p->count += 1;
}

inline void ring_push_front(pkv_pool *p, int32_t id) {
    p->head = (p->head + p->desc.num_blocks - 1) % p->desc.num_blocks;
    p->ring[p->head] = id;
    p->count += 1;
}

pkv_status check_desc(const pkv_pool_desc *d) {
    if (!d) return fail(PKV_ERR_INVALID_ARG, "desc is NULL");
    if (d->num_layers < 1 || d->num_blocks < 1 || d->num_heads < 1)
        return fail(PKV_ERR_INVALID_ARG, "num_layers, num_blocks and num_heads must be >= 1");
    if (!pkv::supported_block_size(d->block_size))
        return fail(PKV_ERR_UNSUPPORTED, "block_size %d not supported (8..256, power of two)", d->block_size);
    if (!pkv::supported_head_dim(d->head_dim))
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", d->head_dim);
    if (d->layout != PKV_LAYOUT_NHD && d->layout != PKV_LAYOUT_HND)
        return fail(PKV_ERR_INVALID_ARG, "layout %d unknown", d->layout);
    if ((int64_t)d->num_blocks * d->block_size * d->num_heads >= (int64_t)1 << 31)
        return fail(PKV_ERR_INVALID_ARG, "num_blocks * block_size * num_heads must be < 2^31");
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
    p->ring = std::move(order);
    p->head = 0;
    p->count = N;
    p->refcount.assign(N, 0);
    p->cow_copies = 0;
    *out = p;
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
        int32_t id = ring_pop_front(pool);
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
        if (rc[ids[j]] == 0) ring_push_back(pool, ids[j]);
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
    for (int32_t r : pool->refcount) {
        if (r > 0) s.used_blocks += 1;
        if (r > 1) s.shared_blocks += 1;
        if (r > s.max_refcount) s.max_refcount = r;
    }
    s.cow_copies = pool->cow_copies;
    *out = s;
    return PKV_OK;
}

pkv_status pkv_free_queue(const pkv_pool *pool, int32_t *out, int32_t capacity, int32_t *count) {
    if (!pool || !count) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
    *count = pool->count;
    if (capacity < pool->count || (pool->count > 0 && !out))
        return fail(PKV_ERR_INVALID_ARG, "capacity %d < %d", capacity, pool->count);
    for (int32_t i = 0; i < pool->count; ++i) out[i] = pool->ring[(pool->head + i) % pool->desc.num_blocks];
    return PKV_OK;
}

pkv_status pkv_validate(const pkv_pool *pool) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const int32_t N = pool->desc.num_blocks;
    std::vector<char> inq(N, 0);
    for (int32_t i = 0; i < pool->count; ++i) {
        int32_t b = pool->ring[(pool->head + i) % N];
        if (b < 0 || b >= N || inq[b]) return fail(PKV_ERR_REFCOUNT, "free queue corrupt at %d", i);
        inq[b] = 1;
    }
    for (int32_t b = 0; b < N; ++b) {
        if (pool->refcount[b] < 0) return fail(PKV_ERR_REFCOUNT, "block %d refcount < 0", b);
        if ((pool->refcount[b] == 0) != (inq[b] != 0))
            return fail(PKV_ERR_REFCOUNT, "block %d: refcount %d but %s the free queue", b,
                        pool->refcount[b], inq[b] ? "in" : "not in");
    }
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
        *id = ring_pop_front(pool);
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
            ring_push_front(pool, allocated[j]);
        }
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
