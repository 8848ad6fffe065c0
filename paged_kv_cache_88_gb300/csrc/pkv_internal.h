// Internal declarations shared by the translation units of libpkv.
#pragma once

#include <cstdint>
#include <unordered_map>
#include <utility>
#include <vector>

#ifdef __CUDACC__
#include <cuda_runtime.h>
#endif

#include "pkv.h"

// Host metadata behind the opaque pkv_pool handle.
struct pkv_pool {
    pkv_pool_desc desc;
    void *k_pool;
    void *v_pool;
    float *k_scale;  // E4M3 cache: per-(token, head) scales [L][N][H][B]; else null
    float *v_scale;
    // FIFO free queue as a doubly linked list over block ids (-1 = none): O(1)
    // take from the head, return to the tail, and removal of a cached block
    // that a prefix lookup revives.
    std::vector<int32_t> next, prev;
    int32_t head, tail, count;
    std::vector<int32_t> refcount;
    int64_t cow_copies;
    // prefix cache: full blocks registered under the chained hash of their tokens
    std::vector<uint64_t> hash_of;
    std::vector<uint8_t> has_hash;
    std::unordered_map<uint64_t, int32_t> by_hash;
    int64_t prefix_hits, prefix_misses, evictions;
};

namespace pkv {

// Record the failure text for pkv_last_error() and return `st`.
pkv_status fail(pkv_status st, const char *fmt, ...);
void clear_error();

inline int64_t layer_elems(const pkv_pool_desc &d) {
    return (int64_t)d.num_blocks * d.block_size * d.num_heads * d.head_dim;
}

inline int kv_elem_bytes(const pkv_pool_desc &d) { return d.kv_dtype == PKV_KV_E4M3 ? 1 : 2; }

// One layer's device pointers of a pool.
struct PoolLayer {
    char *k;
    char *v;
    float *k_scale;  // null for an fp16 cache
    float *v_scale;
};

inline PoolLayer pool_layer(const pkv_pool *p, int32_t layer) {
    const pkv_pool_desc &d = p->desc;
    const size_t off = (size_t)layer * layer_elems(d) * kv_elem_bytes(d);
    const size_t soff = (size_t)layer * d.num_blocks * d.num_heads * d.block_size;
    PoolLayer pl;
    pl.k = static_cast<char *>(p->k_pool) + off;
    pl.v = static_cast<char *>(p->v_pool) + off;
    pl.k_scale = p->k_scale ? p->k_scale + soff : nullptr;
    pl.v_scale = p->v_scale ? p->v_scale + soff : nullptr;
    return pl;
}

inline bool supported_head_dim(int32_t d) { return d == 64 || d == 128 || d == 256; }

// The cascade's prefix pass for an E4M3 pool (HND, head_dim 128; arguments validated by
// pkv_prefix_attention). Defined in prefix_attention_q8.cu.
pkv_status prefix_attention_q8(const pkv_pool *pool, int32_t layer, const void *q, const pkv_prefix_group *groups,
                               int32_t num_groups, int32_t splits, const int32_t *block_tables, int32_t max_blocks,
                               int32_t num_seqs, float scale, void *pieces, uint32_t *status, uint32_t flags,
                               void *stream);

inline bool supported_block_size(int32_t b) {
    return b == 8 || b == 16 || b == 32 || b == 64 || b == 128 || b == 256 || b == 512;
}

// Launch `kernel` on `stream` with programmatic stream serialisation: its CTAs
// may start while the previous kernel of the stream drains; every kernel of
// libpkv calls griddepcontrol.wait before its first global-memory access, so
// stream order of memory effects is unchanged.
#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

}  // namespace pkv
