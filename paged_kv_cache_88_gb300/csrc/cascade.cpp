// Host planner of the shared-prefix (cascade) decode.
//
// Sequences that share leading blocks -- a forked prompt whose blocks carry a
// refcount above one, or prefix-cache hits (icman.com.cn/news/78786 §3.4;
// hnwysp.cn/news/103996 §3.3) -- hold the same physical block ids at the same
// table positions. The planner finds runs of consecutive sequences with such a
// common prefix; pkv_prefix_attention then reads each group's prefix K/V once
// for all its members, and pkv_decode_attention_ex attends every member's
// private rest and merges the two halves. The plan only moves work: the
// attention it produces is the same.
#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

// Blocks lying wholly inside a context of T tokens (capped by the table width).
int32_t full_blocks(int32_t T, int32_t B, int32_t max_blocks) {
    if (T <= 0) return 0;
    return std::min(T / B, max_blocks);
}

// Length of the common run of valid ids of two table rows, up to n entries.
int32_t common_run(const int32_t *a, const int32_t *b, int32_t n) {
    int32_t k = 0;
    while (k < n && a[k] >= 0 && a[k] == b[k]) ++k;
    return k;
}

}  // namespace

extern "C" {

pkv_status pkv_cascade_plan(const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                            int32_t num_seqs, int32_t block_size, int32_t min_group, int32_t min_prefix_tokens,
                            pkv_prefix_group *groups, int32_t max_groups, int32_t *num_groups,
                            int32_t *seq_begin) {
    if (num_seqs < 0 || max_blocks < 1 || max_groups < 0 || min_group < 2)
        return pkv::fail(PKV_ERR_INVALID_ARG, "bad sizes (num_seqs >= 0, max_blocks >= 1, min_group >= 2)");
    if (!pkv::supported_block_size(block_size))
        return pkv::fail(PKV_ERR_UNSUPPORTED, "block_size %d not supported", block_size);
    if (!num_groups) return pkv::fail(PKV_ERR_INVALID_ARG, "num_groups is NULL");
    if (num_seqs > 0 && (!block_tables || !context_lens || !seq_begin))
        return pkv::fail(PKV_ERR_INVALID_ARG, "NULL table, length or seq_begin array");
    if (max_groups > 0 && !groups) return pkv::fail(PKV_ERR_INVALID_ARG, "groups is NULL");
    const int32_t B = block_size;
    // the smallest prefix worth a group, in whole blocks (at least one)
    const int32_t min_blocks = std::max<int32_t>(1, (std::max<int32_t>(min_prefix_tokens, 0) + B - 1) / B);
    for (int32_t s = 0; s < num_seqs; ++s) seq_begin[s] = 0;
    int32_t ng = 0;
    int32_t s = 0;
    while (s < num_seqs) {
        const int32_t *row0 = block_tables + (size_t)s * max_blocks;
        int32_t lcp = full_blocks(context_lens[s], B, max_blocks);
        int32_t e = s + 1;
        while (lcp >= min_blocks && e < num_seqs && e - s < PKV_MAX_GROUP_SEQS) {
            const int32_t n = std::min(lcp, full_blocks(context_lens[e], B, max_blocks));
            const int32_t k = common_run(row0, block_tables + (size_t)e * max_blocks, n);
            if (k < min_blocks) break;
            lcp = k;
            ++e;
        }
        if (e - s >= min_group && lcp >= min_blocks) {
            if (ng < max_groups) {
                groups[ng].first_seq = s;
                groups[ng].num_seqs = e - s;
                groups[ng].prefix_tokens = lcp * B;
                groups[ng].reserved = 0;
                for (int32_t m = s; m < e; ++m) seq_begin[m] = lcp * B;
                ++ng;
            }
            s = e;
        } else {
            ++s;
        }
    }
    *num_groups = ng;
    return PKV_OK;
}

size_t pkv_prefix_pieces_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim) {
    if (num_seqs < 0 || num_heads < 1 || !pkv::supported_head_dim(head_dim)) {
        pkv::fail(PKV_ERR_INVALID_ARG, "bad sizes for the prefix pieces");
        return 0;
    }
    return (size_t)num_seqs * num_heads * PKV_MAX_PREFIX_SPLITS * (head_dim + 4) * sizeof(float);
}

int32_t pkv_prefix_splits(int32_t num_groups, int32_t num_heads, int32_t max_prefix_tokens) {
    if (num_groups < 1 || num_heads < 1 || max_prefix_tokens < 1) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    const int64_t ctas = (int64_t)num_groups * num_heads;
    const int64_t want = (sms + ctas - 1) / ctas;
    const int64_t tiles = (max_prefix_tokens + 127) / 128;
    return (int32_t)std::max<int64_t>(1, std::min<int64_t>({want, tiles, (int64_t)PKV_MAX_PREFIX_SPLITS}));
}

}  // extern "C"
