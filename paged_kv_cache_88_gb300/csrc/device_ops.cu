// Data-movement kernels of libpkv for sm_103a: the append scatter ("reshape and
// cache") and the copy-on-write block copy. Both are pure bit copies bound by
// HBM bandwidth; every access is a 16-byte vector, consecutive threads touch
// consecutive 16-byte words of a row, and bad indices are skipped and flagged,
// never trapped.
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace {

using namespace pkv;

constexpr int kAppendThreads = 256;
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// Token i of the batch goes to slot slot_mapping[i]: physical block slot / B,
// offset slot % B (m.lqnn.cn/news/240480 §3.2 step 3). One thread per 16-byte
// word of the token's K (and the same word of V); a token's row for head h is
// D contiguous elements in either block layout.
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, const int64_t *__restrict__ slots,
              int32_t num_tokens, uint4 *__restrict__ k_layer, uint4 *__restrict__ v_layer, int64_t num_slots,
              int32_t B, int32_t H, int32_t words_per_row, int32_t layout, uint32_t *status) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    const int64_t words_per_token = (int64_t)H * words_per_row;
    const int64_t total = (int64_t)num_tokens * words_per_token;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / words_per_token;
        const int64_t r = idx - i * words_per_token;
        const int32_t h = (int32_t)(r / words_per_row);
        const int32_t w = (int32_t)(r - (int64_t)h * words_per_row);
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0 && status) atomicOr(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / B;
        const int64_t off = slot - blk * B;
        const int64_t row = layout == PKV_LAYOUT_NHD ? (blk * B + off) * H + h : (blk * H + h) * B + off;
        k_layer[row * words_per_row + w] = k_new[idx];
        v_layer[row * words_per_row + w] = v_new[idx];
    }
}

// Block dst <- block src in every layer, K and V (hnwysp.cn/news/103996 §3.3).
// grid.y walks (pair, layer); grid.x and the unrolled loop walk the block's words.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(const int32_t *__restrict__ pairs, int32_t num_pairs, uint4 *k_pool, uint4 *v_pool,
                   int32_t num_layers, int32_t num_blocks, int64_t block_words, uint32_t *status) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    const int64_t jobs = (int64_t)num_pairs * num_layers;
    for (int64_t y = blockIdx.y; y < jobs; y += gridDim.y) {
        const int32_t pr = (int32_t)(y / num_layers);
        const int32_t layer = (int32_t)(y - (int64_t)pr * num_layers);
        const int32_t src = pairs[2 * pr];
        const int32_t dst = pairs[2 * pr + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (status && blockIdx.x == 0 && threadIdx.x == 0 && layer == 0) atomicOr(status, PKV_DEV_BAD_PAIR);
            continue;
        }
        const int64_t sbase = ((int64_t)layer * num_blocks + src) * block_words;
        const int64_t dbase = ((int64_t)layer * num_blocks + dst) * block_words;
        const int64_t step = (int64_t)gridDim.x * blockDim.x;
        for (int64_t w0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w0 < block_words; w0 += step * kCopyUnroll) {
            uint4 kb[kCopyUnroll], vb[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const int64_t w = w0 + u * step;
                if (w < block_words) {
                    kb[u] = k_pool[sbase + w];
                    vb[u] = v_pool[sbase + w];
                }
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const int64_t w = w0 + u * step;
                if (w < block_words) {
                    k_pool[dbase + w] = kb[u];
                    v_pool[dbase + w] = vb[u];
                }
            }
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

pkv_status pkv_append(const pkv_pool *pool, int32_t layer, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens, uint32_t *status, void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (layer < 0 || layer >= d.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail(PKV_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned, slot_mapping 8-byte aligned");
    const int32_t wpr = d.head_dim / 8;
    const int64_t total = (int64_t)num_tokens * d.num_heads * wpr;
    const int64_t want = (total + kAppendThreads - 1) / kAppendThreads;
    const int grid = (int)(want < 65535 * 16 ? want : 65535 * 16);
    const size_t off = (size_t)layer * layer_elems(d) * 2;
    cudaError_t e = launch_pdl(append_kernel, dim3(grid), dim3(kAppendThreads), 0, static_cast<cudaStream_t>(stream),
                               static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
                               num_tokens, reinterpret_cast<uint4 *>(static_cast<char *>(pool->k_pool) + off),
                               reinterpret_cast<uint4 *>(static_cast<char *>(pool->v_pool) + off),
                               (int64_t)d.num_blocks * d.block_size, d.block_size, d.num_heads, wpr, d.layout, status);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

pkv_status pkv_copy_blocks(const pkv_pool *pool, const int32_t *pairs, int32_t num_pairs, uint32_t *status,
                           void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs < 0");
    if (num_pairs == 0) return PKV_OK;
    if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 3u)) return fail(PKV_ERR_INVALID_ARG, "bad pairs pointer");
    const int64_t block_words = (int64_t)d.block_size * d.num_heads * d.head_dim / 8;
    const int64_t per_row = (int64_t)kCopyThreads * kCopyUnroll;
    int gx = (int)((block_words + per_row - 1) / per_row);
    if (gx < 1) gx = 1;
    const int64_t jobs = (int64_t)num_pairs * d.num_layers;
    const int gy = (int)(jobs < 65535 ? jobs : 65535);
    cudaError_t e = launch_pdl(copy_blocks_kernel, dim3(gx, gy), dim3(kCopyThreads), 0,
                               static_cast<cudaStream_t>(stream), pairs, num_pairs,
                               static_cast<uint4 *>(pool->k_pool), static_cast<uint4 *>(pool->v_pool), d.num_layers,
                               d.num_blocks, block_words, status);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "copy launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // extern "C"
