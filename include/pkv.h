/*
 * pkv.h -- C ABI of libpkv: a paged KV cache and decode attention over it,
 * hand-written for NVIDIA GB300 (sm_103a).
 *
 * The method: K and V of every token live in a pool of fixed-size physical
 * blocks carved once at start-up; each sequence owns a block table mapping its
 * logical blocks to physical ones; blocks are shared between sequences with a
 * refcount and copied on write; the decode step appends one token per
 * sequence and attends its query over the whole cached history through the
 * table. Sources, by page address and the page's own section numbers:
 *   hnwysp.cn/news/103996    sections 1.2, 3.1-3.4, 4.1-4.4
 *   icman.com.cn/news/78786  sections 1.1, 2.1-2.4, 3.4, 4.1, 6.3
 *   m.lqnn.cn/news/240480    sections 3.1-3.3, 5.2
 *
 * Conventions (all entry points):
 *   - Every call returns a pkv_status; nothing throws across the ABI.
 *     pkv_last_error() gives a thread-local message for the last failure.
 *   - A call that fails leaves all state (pool, tables, lengths) unchanged.
 *   - Device memory (the K/V pools, q, out, tables, lengths, workspaces) is
 *     owned by the caller; the library never allocates or frees it. A pool
 *     handle owns only host metadata.
 *   - Device entry points only enqueue work on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream): no host synchronisation, no
 *     allocation. They are asynchronous; their errors found on the host are
 *     returned, errors found on the device are OR-ed into a caller-provided
 *     device status word (PKV_DEV_* bits) that the caller reads when it wants.
 *   - Kernels never trap: an out-of-range index is skipped (or clamped) and
 *     flagged in the status word; every wait in a kernel has a time limit.
 *   - A pool handle is not thread-safe: the caller serialises calls that
 *     mutate it. Distinct pools are independent.
 *   - Element types: IEEE binary16 (fp16) for q, out and the new tokens' K/V rows;
 *     the K/V pools hold fp16 or FP8 E4M3 codes with per-row fp32 scales
 *     (PKV_KV_F16 / PKV_KV_E4M3 below).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* a size, pointer or shape is outside what the call accepts */
    PKV_ERR_OUT_OF_BLOCKS = 2, /* the free queue cannot satisfy the request (nothing allocated) */
    PKV_ERR_BAD_BLOCK = 3,     /* a block id outside [0, num_blocks) */
    PKV_ERR_REFCOUNT = 4,      /* free/incref of a block whose refcount does not allow it */
    PKV_ERR_CUDA = 5,          /* a CUDA runtime call failed (message in pkv_last_error) */
    PKV_ERR_UNSUPPORTED = 6    /* a shape the kernels are not built for (e.g. head_dim 96) */
} pkv_status;

/* Block layouts within one layer's pool of N blocks (both put B*H*D contiguous
 * elements per block, so a block is one contiguous byte range):
 *   PKV_LAYOUT_NHD: [N][B][H][D] -- the order m.lqnn.cn/news/240480 §3.3 prints,
 *                   [page, slot, head, dim];
 *   PKV_LAYOUT_HND: [N][H][B][D] -- one head's tokens of a block contiguous. */
enum { PKV_LAYOUT_NHD = 0, PKV_LAYOUT_HND = 1 };

/* Element type of the K/V pools:
 *   PKV_KV_F16:  IEEE binary16;
 *   PKV_KV_E4M3: FP8 E4M3 codes (1 byte) with one fp32 scale per (token, head)
 *                row, value = code * scale, scale = amax(row) / 448 (1 for an
 *                all-zero row), codes rounded to nearest even and saturated.
 *                Quantised KV halves the bytes per token (m.lqnn.cn/news/240480
 *                §6.2; hnwysp.cn/news/103996 §5.4). Either layout, head_dim 64 or
 *                128; the scale pools are [L][N][H][B] fp32 in both layouts
 *                (pkv_pool_set_scales); the cascade's prefix pass needs HND. */
enum { PKV_KV_F16 = 0, PKV_KV_E4M3 = 1 };

/* Bits of the device status word (uint32_t) that device entry points OR into. */
#define PKV_DEV_BAD_BLOCK 0x1u   /* a block-table entry outside [0, num_blocks): clamped to 0 */
#define PKV_DEV_BAD_LENGTH 0x2u  /* a context length < 0 or > max_blocks * block_size: clamped */
#define PKV_DEV_TIMEOUT 0x4u     /* a pipeline wait hit its time limit; outputs are garbage */
#define PKV_DEV_BAD_SLOT 0x8u    /* a slot >= num_blocks * block_size: that token not written */
#define PKV_DEV_BAD_PAIR 0x10u   /* a copy pair with an id outside [0, num_blocks): skipped */

typedef struct pkv_pool_desc {
    int32_t num_layers; /* L >= 1 */
    int32_t num_blocks; /* N >= 1 physical blocks per layer */
    int32_t block_size; /* B tokens per block: 8, 16, 32, 64, 128, 256 or 512 */
    int32_t num_heads;  /* H KV heads (query heads = KV heads) */
    int32_t head_dim;   /* D: 64, 128 or 256 */
    int32_t layout;     /* PKV_LAYOUT_NHD or PKV_LAYOUT_HND */
    int32_t kv_dtype;   /* PKV_KV_F16 (0) or PKV_KV_E4M3 */
} pkv_pool_desc;

typedef struct pkv_stats {
    int32_t free_blocks;        /* blocks in the free queue */
    int32_t used_blocks;        /* blocks with refcount >= 1 */
    int32_t shared_blocks;      /* blocks with refcount >= 2 */
    int32_t max_refcount;
    int64_t cow_copies;         /* copy-on-write copies issued by pkv_prepare_append so far */
    int32_t cached_blocks;      /* blocks registered in the prefix cache (in use or free) */
    int32_t cached_free_blocks; /* of those, blocks in the free queue (revived by a hit) */
    int64_t prefix_hits;        /* blocks found by pkv_prefix_lookup so far */
    int64_t prefix_misses;      /* blocks looked up and not found */
    int64_t evictions;          /* cached blocks whose hash was dropped when reused */
} pkv_stats;

typedef struct pkv_pool pkv_pool; /* opaque host metadata */

/* Thread-local text of the last failure of this thread ("" if none). */
const char *pkv_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pkv_version(void);

/* ------------------------------------------------------------------ host: pool
 * Carve the pool: hnwysp.cn/news/103996 §3.2, §4.1 (reserve once, thread every
 * block onto the free list); icman.com.cn/news/78786 §2.3.
 *
 * k_pool, v_pool: device pointers to L * N * B * H * D fp16 elements each, laid
 *   out [L][N][block] with the block as `layout` says; 16-byte aligned. They may
 *   be NULL for a host-only pool (allocator use without a GPU); device entry
 *   points then refuse the pool. The caller keeps ownership.
 * initial_free_order: host array of N distinct ids 0..N-1 giving the free queue
 *   from head to tail, or NULL for 0, 1, ..., N-1. Copied.
 * out: receives the handle. Errors: INVALID_ARG (bad sizes, order not a
 *   permutation, N*B or L*N*B*H*D too large). Touches no CUDA state. */
pkv_status pkv_pool_create(const pkv_pool_desc *desc, void *k_pool, void *v_pool,
                           const int32_t *initial_free_order, pkv_pool **out);

/* E4M3 pools: attach the caller-owned scale pools (device fp32 [L][N][H][B]
 * each, 16-byte aligned) that pair with k_pool / v_pool. INVALID_ARG for an
 * fp16 pool. Device entry points refuse an E4M3 pool without them. */
pkv_status pkv_pool_set_scales(pkv_pool *pool, void *k_scale, void *v_scale);

/* Free the host metadata. Does not free the device pools. NULL is accepted. */
pkv_status pkv_pool_destroy(pkv_pool *pool);

/* Read back the descriptor and the device pointers given at creation. */
pkv_status pkv_pool_info(const pkv_pool *pool, pkv_pool_desc *desc, void **k_pool, void **v_pool);

/* Take n blocks from the head of the free queue, each with refcount 1, and
 * write their ids to out_ids (host, n entries) in queue order.
 * hnwysp.cn/news/103996 §3.4, §4.4 (take from the head of the free queue).
 * All-or-nothing: OUT_OF_BLOCKS if fewer than n are free, nothing taken. */
pkv_status pkv_alloc(pkv_pool *pool, int32_t n, int32_t *out_ids);

/* One more reference to each listed block (host array, n ids; repeats count
 * twice): sharing a prefix or forking a sequence, icman.com.cn/news/78786 §3.4.
 * BAD_BLOCK for an id out of range, REFCOUNT for a free block; all-or-nothing. */
pkv_status pkv_incref(pkv_pool *pool, const int32_t *ids, int32_t n);

/* Drop one reference per listed block (host array, n ids; repeats count).
 * A block reaching 0 is pushed to the tail of the free queue, in list order:
 * hnwysp.cn/news/103996 §3.3, §3.4, §4.4; icman.com.cn/news/78786 §6.3.
 * BAD_BLOCK / REFCOUNT (a count would go below 0); all-or-nothing. */
pkv_status pkv_free(pkv_pool *pool, const int32_t *ids, int32_t n);

/* Refcount of block id (0 = free). BAD_BLOCK if out of range. */
pkv_status pkv_refcount(const pkv_pool *pool, int32_t id, int32_t *out);

/* Pool counters (icman.com.cn/news/78786 §6.5 lists pool use as the first
 * figure to watch). */
pkv_status pkv_get_stats(const pkv_pool *pool, pkv_stats *out);

/* Copy the free queue, head first, into out (capacity entries); *count gets
 * its length. INVALID_ARG if capacity is too small. */
pkv_status pkv_free_queue(const pkv_pool *pool, int32_t *out, int32_t capacity, int32_t *count);

/* Check the bookkeeping: the free queue holds every block with refcount 0 once
 * and nothing else. REFCOUNT if not (never expected; a test hook). */
pkv_status pkv_validate(const pkv_pool *pool);

/* ------------------------------------------------------------- prefix cache
 * Requests that start with the same tokens share the KV blocks of those tokens
 * (icman.com.cn/news/78786 §3.2-§3.4; hnwysp.cn/news/103996 §4.3): each FULL block of
 * a prompt is keyed by a hash chained from the start of the sequence, a hit
 * takes one more reference to the cached block and writes no KV. A block whose
 * refcount drops to 0 keeps its hash while it waits in the free queue, so the
 * queue doubles as the LRU of cached blocks: a later hit takes it back out,
 * and taking it from the head for reuse drops (evicts) its hash. */

/* Hash of one block: 64-bit FNV-1a over `parent` (the previous block's hash, 0
 * for the first block; 8 bytes little-endian) followed by the n token ids (4
 * bytes little-endian each). */
uint64_t pkv_block_hash(uint64_t parent, const int32_t *token_ids, int32_t n);

/* The chained hashes of every FULL block of a prompt (icman.com.cn/news/78786 §3.2:
 * a block's key covers its tokens and, through the parent hash, every token
 * before it): out[i] = pkv_block_hash(out[i-1], tokens of block i, block_size),
 * with parent 0 for block 0. token_ids: host int32 [num_tokens]; out: host
 * uint64 [capacity]; *num_hashes = num_tokens / block_size (a partial last block
 * is not hashed). INVALID_ARG for a negative count, block_size < 1, NULL arrays
 * or capacity < num_tokens / block_size (nothing written then). */
pkv_status pkv_prompt_block_hashes(const int32_t *token_ids, int32_t num_tokens, int32_t block_size,
                                   uint64_t *out, int32_t capacity, int32_t *num_hashes);

/* For i = 0, 1, ... look hashes[i] up; stop at the first miss. Each hit gets
 * one more reference (a cached block in the free queue is taken out of it and
 * gets refcount 1) and its id goes to out_ids[i]. *num_hits = the hits.
 * Chained hashes make a later block meaningless after a miss, hence the stop. */
pkv_status pkv_prefix_lookup(pkv_pool *pool, const uint64_t *hashes, int32_t n, int32_t *out_ids,
                             int32_t *num_hits);

/* Register full blocks whose KV has been written: hashes[i] -> ids[i] (blocks in
 * use). A hash already held by another block keeps that block; a block
 * re-registered under a new hash drops the old one. BAD_BLOCK / REFCOUNT (a
 * free block) refuse the whole call. */
pkv_status pkv_prefix_register(pkv_pool *pool, const uint64_t *hashes, const int32_t *ids, int32_t n);

/* Give slots to the next tokens of a batch of sequences; the host half of the
 * decode step (m.lqnn.cn/news/240480 §3.2 step 3; hnwysp.cn/news/103996 §3.3).
 *
 * For s = 0..num_seqs-1 in order, and for each of its num_new[s] tokens in
 * order (num_new NULL = one token each), with p = context_lens[s]:
 *   - if p % B == 0: a block is taken from the free queue into
 *     block_tables[s][p / B];
 *   - else, if the block block_tables[s][p / B] has refcount > 1: a block dst
 *     is taken, the pair (that block, dst) is emitted, the old block loses one
 *     reference and dst replaces it in the table (copy-on-write);
 *   - the token's slot is block_tables[s][p / B] * B + p % B, and p grows by 1.
 * block_tables: host int32 [num_seqs][max_blocks], updated in place (entries
 *   past the sequence's blocks are not read). context_lens: host int32
 *   [num_seqs], updated in place. slot_mapping: host int64, capacity
 *   slot_capacity; *num_slots = tokens given slots, in (sequence, token) order.
 * copy_pairs: host int32 [pair_capacity][2] (src, dst); *num_pairs = pairs.
 *   The caller must run pkv_copy_blocks on these pairs before pkv_append
 *   writes the new tokens.
 * Errors (all-or-nothing, nothing changed): OUT_OF_BLOCKS; INVALID_ARG (a table
 *   too short for the new length, capacities too small, negative counts);
 *   BAD_BLOCK (a table entry that is out of range or not allocated). */
pkv_status pkv_prepare_append(pkv_pool *pool, int32_t num_seqs, int32_t *block_tables,
                              int32_t max_blocks, int32_t *context_lens, const int32_t *num_new,
                              int64_t *slot_mapping, int32_t slot_capacity, int32_t *num_slots,
                              int32_t *copy_pairs, int32_t pair_capacity, int32_t *num_pairs);

/* ---------------------------------------------------------------- device ops */

/* Write num_tokens new tokens' K and V of layer `layer` into their slots
 * ("reshape and cache"; m.lqnn.cn/news/240480 §3.2 step 3, §3.3).
 * k_new, v_new: device fp16 [num_tokens][H][D], 16-byte aligned.
 * slot_mapping: device int64 [num_tokens]; slot < 0 means "skip this token";
 *   slot >= N * B is skipped and flagged PKV_DEV_BAD_SLOT. Slots must be
 *   distinct (two tokens to one slot race).
 * status: device uint32 status word (may be NULL). Bit copy, no arithmetic.
 * Host errors: INVALID_ARG (layer out of range, host-only pool, misaligned). */
pkv_status pkv_append(const pkv_pool *pool, int32_t layer, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens, uint32_t *status,
                      void *stream);

/* Copy-on-write data move (hnwysp.cn/news/103996 §3.3): for each pair
 * (src, dst) of the device int32 array pairs[num_pairs][2], block dst <- block
 * src in every layer, K and V (B * H * D elements each). A pair with an id out
 * of range is skipped and flagged PKV_DEV_BAD_PAIR. dst blocks must be distinct
 * and must not appear as a src. num_pairs = 0 enqueues nothing. */
pkv_status pkv_copy_blocks(const pkv_pool *pool, const int32_t *pairs, int32_t num_pairs,
                           uint32_t *status, void *stream);

/* Swap (icman.com.cn/news/78786 §4.2: a preempted request's KV goes out to host
 * memory and comes back later). The library moves blocks between the pool and a
 * contiguous caller-owned buffer, and the caller frees / allocates the blocks
 * with pkv_free / pkv_alloc, all on the same stream. The buffer is either
 * device memory (the caller then moves it to and from pinned host memory with
 * one cudaMemcpyAsync each way) or pinned host memory that is mapped into the
 * device's address space (cudaHostAlloc / cudaHostRegister on a system with
 * unified addressing): the kernel then reads or writes host memory directly
 * over the host link, one pass, no staging copy. The buffer must be 16-byte
 * aligned; any other pointer (pageable host memory, an unmapped host
 * allocation) is refused with INVALID_ARG before anything is launched.
 * Buffer layout: for i = 0..n-1 and each layer: block blocks[i]'s K bytes, V
 * bytes, then (E4M3 pools) its K and V row scales; pkv_swap_bytes_per_block
 * gives the bytes per block over all layers. blocks: device int32 [n]; an id
 * outside [0, N) is skipped and flagged PKV_DEV_BAD_PAIR. Bit copies. */
size_t pkv_swap_bytes_per_block(const pkv_pool *pool);
pkv_status pkv_gather_blocks(const pkv_pool *pool, const int32_t *blocks, int32_t n, void *dst,
                             uint32_t *status, void *stream);
pkv_status pkv_scatter_blocks(const pkv_pool *pool, const int32_t *blocks, int32_t n, const void *src,
                              uint32_t *status, void *stream);

/* Paged decode attention for one layer: for every sequence s and head h,
 *   out[s][h] = softmax_t(scale * q[s][h] . K_s[t]) V_s[t],  t = 0..T_s-1,
 * where token t of sequence s is read from physical block
 * block_tables[s][t / B] at slot t % B (m.lqnn.cn/news/240480 §3.3;
 * icman.com.cn/news/78786 §2.4). Products and sums in fp32, out in fp16
 * (round to nearest even). T_s = 0 gives out[s][h] = 0.
 *
 * q: device fp16 [num_seqs][H][D]. k_cache, v_cache: device pointers to one
 *   layer's pool (N blocks in `layout`), 16-byte aligned.
 * block_tables: device int32 [num_seqs][max_blocks]. context_lens: device int32
 *   [num_seqs] (the lengths after this step's append).
 * scale: softmax scale; pass 0 or a negative value for 1/sqrt(D).
 * out: device fp16 [num_seqs][H][D].
 * workspace: device scratch of at least pkv_decode_workspace_bytes(...) bytes,
 *   16-byte aligned, ZERO-FILLED before its first use; each call leaves its
 *   counter area zero again, so one workspace serves every later call on the
 *   same stream with at most the num_seqs and num_heads it was sized for, any
 *   head_dim and either cache type (calls that overlap on the GPU must use
 *   distinct workspaces). A call that ends with PKV_DEV_TIMEOUT may leave
 *   counters set: zero the workspace again before reusing it. Its first 4
 *   bytes are the device status word of the call (PKV_DEV_* bits, sticky:
 *   clear it to reset).
 * Limits (every decode-attention entry point): num_seqs <= 4096 per launch (the
 *   kernel keeps three int32 per sequence in shared memory, and every CTA scans
 *   the lengths in its prologue); head_dim 64, 128 or 256 for an fp16 cache, 64
 *   or 128 for an E4M3 cache (either layout); block_size 8, 16,
 *   32, 64, 128, 256 or 512; num_blocks * block_size * num_heads < 2^31.
 * Errors: INVALID_ARG (sizes, alignment, workspace too small), UNSUPPORTED
 *   (head_dim or block_size not built), CUDA (launch failure). */
pkv_status pkv_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                int32_t num_blocks, int32_t block_size, int32_t num_heads,
                                int32_t head_dim, int32_t layout, const int32_t *block_tables,
                                int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs,
                                float scale, void *out, void *workspace, size_t workspace_bytes,
                                void *stream);

/* The decode step of one layer in one launch: exactly pkv_append(pool, layer,
 * k_new, v_new, slot_mapping, num_seqs) followed by pkv_pool_decode_attention
 * over the same layer, for ONE new token per sequence (m.lqnn.cn/news/240480
 * §3.2 step 3 then §3.3). Token s is sequence s's newest token: slot_mapping[s]
 * must be the slot of position context_lens[s] - 1 (what pkv_prepare_append
 * returns), and context_lens already counts it. The CTA that reads the tile
 * holding that position stores the token's K/V row (all heads handled by their
 * own CTAs) right before loading the tile, so no separate append launch runs.
 * slot_mapping[s] < 0: nothing is stored for s (the pool row is used as it is);
 * >= N * B: skipped and flagged PKV_DEV_BAD_SLOT.
 * k_new, v_new: device fp16 [num_seqs][H][D], 16-byte aligned; other arguments
 * as pkv_pool_decode_attention. */
pkv_status pkv_decode_append_attention(const pkv_pool *pool, int32_t layer, const void *q, const void *k_new,
                                       const void *v_new, const int64_t *slot_mapping,
                                       const int32_t *block_tables, int32_t max_blocks,
                                       const int32_t *context_lens, int32_t num_seqs, float scale, void *out,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* pkv_decode_attention without a caller workspace: the scratch comes from a
 * 4 MiB array compiled into the library. The method's pages have no
 * counterpart for this call; it is here for callers that cannot allocate
 * device memory -- e.g. a host framework that owns every device byte and gives
 * a plugin no workspace, or a serving loop that forbids allocation once it runs
 * because cudaMalloc can synchronise the device and stall other streams.
 *
 * Arguments and result as pkv_decode_attention, minus the workspace; status
 * (device uint32, may be NULL) receives the call's PKV_DEV_* bits OR-ed in.
 * Limit: the sizes must need at most 4 MiB of scratch (what
 * pkv_decode_workspace_bytes reports for them); larger ones return
 * PKV_ERR_INVALID_ARG with the sizes in pkv_last_error and launch nothing.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Every GPU that loads the library holds the 4 MiB until the process exits.
 * The first call on a device, made with that device current, looks the
 * array's device address up once (cudaGetSymbolAddress); make that first call
 * before any stream capture. The address is kept for the life of the process:
 * tearing the device's primary context down (cudaDeviceReset) invalidates it,
 * so do not call this entry point again on that device after such a reset.
 * All calls share the one array and each clears its counters on `stream`
 * first, so calls that overlap on the GPU (other streams, other threads) race:
 * serialise them. */
pkv_status pkv_decode_attention_static(const void *q, const void *k_cache, const void *v_cache,
                                       int32_t num_blocks, int32_t block_size, int32_t num_heads,
                                       int32_t head_dim, int32_t layout, const int32_t *block_tables,
                                       int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs,
                                       float scale, void *out, uint32_t *status, void *stream);

/* Paged prefill (chunked, causal) attention on the tensor cores: for each
 * sequence s, the chunk of its newest tokens -- rows q_start[s] .. q_start[s+1]-1
 * of q, C_s of them -- has already been appended to the pool, and
 * context_lens[s] = T_s counts it. Query i of the chunk (position
 * p = T_s - C_s + i) attends to every cached token t <= p through the block
 * table (m.lqnn.cn/news/240480 §3.3 remap, §4.3 causal prefill):
 *   out[row][h] = softmax_{t <= p}(scale * q[row][h] . K_t[h]) V_t[h].
 * q, out: device fp16 [total_q][H][D], 16-byte aligned. q_start: device int32
 * [num_seqs + 1]. max_chunk: a host bound on every C_s (sizes the grid; rows of a
 * chunk past the grid's ceil(max_chunk / 256) * 256 are not computed, and the call
 * is flagged PKV_DEV_BAD_LENGTH). status: device uint32 word (required).
 * The pool must be fp16, HND, head_dim 128. fp16 products, fp32 accumulation;
 * the softmax weights enter P V in fp16. T_s < C_s or T_s beyond the table is
 * clamped and flagged PKV_DEV_BAD_LENGTH. UNSUPPORTED for other pools. */
pkv_status pkv_prefill_attention(const pkv_pool *pool, int32_t layer, const void *q, const int32_t *q_start,
                                 int32_t total_q, int32_t num_seqs, int32_t max_chunk,
                                 const int32_t *block_tables, int32_t max_blocks,
                                 const int32_t *context_lens, float scale, void *out, uint32_t *status,
                                 void *stream);

/* ------------------------------------------------ shared-prefix (cascade) decode
 *
 * When sequences share their leading blocks (a forked prompt, or prefix-cache
 * hits: icman.com.cn/news/78786 §3.4, hnwysp.cn/news/103996 §3.3), the decode
 * attention of every one of them reads the same prefix K/V. The cascade splits
 * such a sequence's context in two: the shared prefix, attended ONCE per group
 * of sequences by pkv_prefix_attention (all the group's queries against each
 * prefix K/V tile, on the tensor cores), and the private rest, attended by
 * pkv_decode_attention_ex, whose combine step merges the prefix pieces in. The
 * result is the same attention, up to the order of rounding. */

typedef struct {
    int32_t first_seq;     /* members: sequences first_seq .. first_seq + num_seqs - 1 */
    int32_t num_seqs;      /* 2 .. PKV_MAX_GROUP_SEQS */
    int32_t prefix_tokens; /* shared leading tokens: whole blocks, the same ids in every member's table */
    int32_t reserved;      /* 0 */
} pkv_prefix_group;

#define PKV_MAX_GROUP_SEQS 128
#define PKV_ATTN_INPUTS_EARLY 0x1u     /* pkv_decode_attention_ex flag, see there */
#define PKV_ATTN_LAST_ROW_PENDING 0x2u /* pkv_decode_attention_ex flag, see there */
#define PKV_MAX_PREFIX_SPLITS 8

/* Host planner of the cascade for one step. block_tables: host int32
 * [num_seqs][max_blocks]; context_lens: host int32 [num_seqs], the lengths the
 * attention will use. A group is a run of consecutive sequences whose first
 * blocks are the same block ids; a run grows while the common prefix keeps at
 * least min_prefix_tokens tokens and the run holds at most PKV_MAX_GROUP_SEQS
 * sequences; runs of fewer than min_group (>= 2) sequences are dropped. A
 * prefix counts only blocks lying wholly inside every member's context.
 * Writes the groups (host, at most max_groups; further runs are dropped),
 * *num_groups, and seq_begin (host int32 [num_seqs]): the group's prefix_tokens
 * for a member, 0 for any other sequence. Deterministic; reads no device
 * memory. INVALID_ARG for bad sizes or NULL pointers. */
pkv_status pkv_cascade_plan(const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                            int32_t num_seqs, int32_t block_size, int32_t min_group,
                            int32_t min_prefix_tokens, pkv_prefix_group *groups, int32_t max_groups,
                            int32_t *num_groups, int32_t *seq_begin);

/* Bytes of the prefix-piece buffer for these sizes: num_seqs * num_heads *
 * PKV_MAX_PREFIX_SPLITS pieces of (head_dim + 4) fp32 (0 on bad sizes). */
size_t pkv_prefix_pieces_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim);

/* Key splits per group that pkv_prefix_attention should use on the current
 * device: enough (group, head, split) CTAs to cover the SMs once, at most one
 * split per 128 prefix tokens, within 1 .. PKV_MAX_PREFIX_SPLITS. */
int32_t pkv_prefix_splits(int32_t num_groups, int32_t num_heads, int32_t max_prefix_tokens);

/* The prefix half of the cascade for one layer. For each group g (device array
 * `groups` of num_groups), head h and split k < splits: the queries q[s][h] of
 * the group's members against the keys of split k of the prefix
 * [0, prefix_tokens) (tiles of 128 keys dealt to the splits in order), read
 * through table row first_seq. Writes, for each member s, the piece
 *   o[d] = sum_t 2^(x_t - m) V_t[d],  l = sum_t 2^(x_t - m),  m,
 * with x_t = scale * log2(e) * q[s][h] . K_t and m a reference at least as
 * large as max_t x_t - 8, as fp32 (o[0..D-1], m, l) at
 *   pieces + ((s * H + h) * PKV_MAX_PREFIX_SPLITS + k) * (D + 4);
 * a split with no keys writes m = -inf, l = 0, o = 0. q: device fp16
 * [num_seqs][H][D], 16-byte aligned. pieces: device, >=
 * pkv_prefix_pieces_bytes(num_seqs, H, D) bytes, 16-byte aligned. status:
 * device uint32 word (required): a group outside [0, num_seqs), with more
 * than PKV_MAX_GROUP_SEQS members or a prefix not in whole blocks inside the
 * table is flagged PKV_DEV_BAD_LENGTH and writes no pieces. fp16 products,
 * fp32 accumulation, weights enter P V in fp16. The pool must be HND with
 * head_dim 128, fp16 (the pass runs on tcgen05) or E4M3 (on the warp-level
 * tensor cores, K and V read as code x row scale; there m is at least
 * max_t (x_t + log2 of t's V row scale), so each weight times that scale stays
 * within fp16) -- UNSUPPORTED otherwise. flags: 0, or PKV_ATTN_INPUTS_EARLY:
 * the groups, the block tables and the prefix's cached K/V are read -- and the
 * K/V tiles' loads issued -- before the kernel that precedes it on the stream
 * has finished; q is read and the pieces written only after. The caller
 * promises that the preceding kernel writes none of the former (e.g. it is the
 * previous layer's private pass, which writes that layer's cache, out and the
 * workspace). Other flag bits: INVALID_ARG. */
pkv_status pkv_prefix_attention(const pkv_pool *pool, int32_t layer, const void *q,
                                const pkv_prefix_group *groups, int32_t num_groups, int32_t splits,
                                const int32_t *block_tables, int32_t max_blocks, int32_t num_seqs, float scale,
                                void *pieces, size_t pieces_bytes, uint32_t *status, uint32_t flags,
                                void *stream);

/* pkv_decode_append_attention and pkv_pool_decode_attention in one entry, with
 * the private half of the cascade. k_new, v_new, slot_mapping: all NULL = no
 * append (else as pkv_decode_append_attention). seq_begin, pieces: both NULL =
 * no cascade (the plain attention); the cascade needs head_dim 128
 * (UNSUPPORTED otherwise), and its prefix pass the HND layout. Otherwise seq_begin is device int32
 * [num_seqs]: sequence s attends here to its tokens [seq_begin[s], T_s) and,
 * when seq_begin[s] > 0, merges in the `splits` prefix pieces that
 * pkv_prefix_attention wrote for it earlier on the same stream. seq_begin[s]
 * must be a multiple of the block size in [0, T_s]; any other value is
 * flagged PKV_DEV_BAD_LENGTH and read as 0 (no prefix).
 * flags: 0, or PKV_ATTN_INPUTS_EARLY. With it, the kernel reads the block
 * tables, the lengths, seq_begin and the cached K/V rows -- and issues its first
 * tiles' loads -- before the kernel that precedes it on the stream has finished;
 * it touches q, k_new, v_new, the workspace, the pieces and out only after. The
 * caller promises that the preceding kernel writes none of the former (e.g. it is
 * the previous layer's attention, or the prefix pass): then the load latency at
 * the start of the launch overlaps the end of the previous one. Every libpkv
 * kernel lets its successor start only after its own inputs are final, so
 * anything launched before that preceding kernel is complete.
 * PKV_ATTN_LAST_ROW_PENDING (with PKV_ATTN_INPUTS_EARLY): the preceding kernel
 * may also write the last cached row of each sequence (it is this step's
 * pkv_append of the layer); the tiles holding those rows are then read only
 * after it has finished. Alone it changes nothing. Other flag bits:
 * INVALID_ARG. */
pkv_status pkv_decode_attention_ex(const pkv_pool *pool, int32_t layer, const void *q, const void *k_new,
                                   const void *v_new, const int64_t *slot_mapping, const int32_t *block_tables,
                                   int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs,
                                   const int32_t *seq_begin, const float *pieces, int32_t splits, float scale,
                                   void *out, void *workspace, size_t workspace_bytes, uint32_t flags,
                                   void *stream);

/* Self-test of the device wait limit (failure detection without a fault): one CTA
 * waits, with the bounded wait every pipeline stage of the attention kernels uses, on
 * an mbarrier that nothing ever completes. After the limit (1 s) it ORs
 * PKV_DEV_TIMEOUT into *status (device uint32) and exits; the context stays usable.
 * Errors: INVALID_ARG (status NULL), CUDA (launch failure). */
pkv_status pkv_check_wait_limit(uint32_t *status, void *stream);

/* Bytes of workspace pkv_decode_attention needs for these sizes on the
 * current CUDA device (0 and a pkv_last_error message on bad arguments). */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim);

/* The same attention on a pool handle's layer (pointers and shape from the
 * pool). */
pkv_status pkv_pool_decode_attention(const pkv_pool *pool, int32_t layer, const void *q,
                                     const int32_t *block_tables, int32_t max_blocks,
                                     const int32_t *context_lens, int32_t num_seqs, float scale,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Launch geometry of the decode attention kernel on the current device, for
 * reporting: CTAs per launch, CTAs per SM, and the SM count, for a cache of
 * kv_dtype (PKV_KV_F16 or PKV_KV_E4M3: the two variants differ in registers,
 * pipeline depth and so in CTAs per SM). Any output pointer may be NULL.
 * PKV_ERR_INVALID_ARG for an unsupported head_dim, a num_seqs outside
 * [0, 4096] or an unknown kv_dtype (checked before any CUDA call). */
pkv_status pkv_decode_launch_info(int32_t num_seqs, int32_t head_dim, int32_t kv_dtype, int32_t *grid_ctas,
                                  int32_t *ctas_per_sm, int32_t *num_sms);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
