// Internal declarations shared by the translation units of libpkv.
#pragma once

#include <cstdint>
#include <vector>

#include "pkv.h"

// Host metadata behind the opaque pkv_pool handle.
struct pkv_pool {
    pkv_pool_desc desc;
    void *k_pool;
    void *v_pool;
    // FIFO free queue as a ring buffer of capacity N: head index + count.
    std::vector<int32_t> ring;
    int32_t head;
    int32_t count;
    std::vector<int32_t> refcount;
    int64_t cow_copies;
};

namespace pkv {

// Record the failure text for pkv_last_error() and return `st`.
pkv_status fail(pkv_status st, const char *fmt, ...);
void clear_error();

inline int64_t layer_elems(const pkv_pool_desc &d) {
    return (int64_t)d.num_blocks * d.block_size * d.num_heads * d.head_dim;
}

inline bool supported_head_dim(int32_t d) { return d == 64 || d == 128 || d == 256; }

inline bool supported_block_size(int32_t b) {
    return b == 8 || b == 16 || b == 32 || b == 64 || b == 128 || b == 256;
}

}  // namespace pkv
