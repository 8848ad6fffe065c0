// Data-movement kernels of libpkv for sm_103a: the append scatter ("reshape and
// cache") and the copy-on-write block copy. Both are pure bit copies bound by
// HBM bandwidth; every access is a 16-byte vector, consecutive threads touch
// consecutive 16-byte words of a row, and bad indices are skipped and flagged,
// never trapped.
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace {

using namespace pkv;

constexpr int kAppendThreads = 256;
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kSwapUnroll = 8;
constexpr int64_t kSwapChunk = (int64_t)kCopyThreads * kSwapUnroll;   // words per CTA pass

// Token i of the batch goes to slot slot_mapping[i]: physical block slot / B,
// offset slot % B (m.lqnn.cn/news/240480 §3.2 step 3). One thread per 16-byte
// word of the token's K (and the same word of V); a token's row for head h is
// D contiguous elements in either block layout.
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, const int64_t *__restrict__ slots,
              int32_t num_tokens, uint4 *__restrict__ k_layer, uint4 *__restrict__ v_layer, int64_t num_slots,
              int32_t B, int32_t H, int32_t words_per_row, int32_t layout, uint32_t *status) {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();   // successors start once this grid's inputs are final
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

// E4M3 cache: one warp per (token, head). Lanes 0..W-1 hold the K row's
// 16-byte fp16 words, lanes W..2W-1 the V row's (W = D/8 <= 16); each row's
// amax is reduced over its W lanes, then each lane stores its 8 codes and the
// first lane of a row the row's scale. The codes follow the pool's layout; the
// scales are [N][H][B] in either.
template <int D>
__global__ void __launch_bounds__(kAppendThreads)
append_q8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, const int64_t *__restrict__ slots,
                 int32_t num_tokens, unsigned char *__restrict__ k_layer, unsigned char *__restrict__ v_layer,
                 float *__restrict__ k_scale, float *__restrict__ v_scale, int64_t num_slots, int32_t B, int32_t H,
                 int32_t layout, uint32_t *status) {
    constexpr int W = D / 8;
    ptx::grid_dependency_wait();
    ptx::launch_dependents();   // successors start once this grid's inputs are final
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)num_tokens * H;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t i = r / H;
        const int32_t h = (int32_t)(r - i * H);
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (lane == 0 && h == 0 && status) atomicOr(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        uint4 w = make_uint4(0, 0, 0, 0);
        if (lane < 2 * W) w = lane < W ? k_new[r * W + lane] : v_new[r * W + lane - W];
        float m = q8::amax_word(w);
#pragma unroll
        for (int o = 1; o < W; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float scale = q8::row_scale(m);
        if (lane < 2 * W) {
            const int64_t blk = slot / B, off = slot - blk * B;
            const int64_t srow = (blk * H + h) * B + off;   // the row's scale
            const int64_t row = layout == PKV_LAYOUT_NHD ? (blk * B + off) * H + h : srow;
            reinterpret_cast<uint2 *>((lane < W ? k_layer : v_layer) + row * D)[lane % W] = q8::quantize_word(w, scale);
            if (lane % W == 0) (lane < W ? k_scale : v_scale)[srow] = scale;
        }
    }
}

// Block dst <- block src in every layer, K and V (hnwysp.cn/news/103996 §3.3).
// grid.y walks (pair, layer); grid.x and the unrolled loop walk the block's words.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(const int32_t *__restrict__ pairs, int32_t num_pairs, uint4 *k_pool, uint4 *v_pool,
                   int32_t num_layers, int32_t num_blocks, int64_t block_words, uint4 *k_scale, uint4 *v_scale,
                   int64_t scale_words, uint32_t *status) {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();   // successors start once this grid's inputs are final
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
        if (k_scale) {  // E4M3 cache: the block's row scales, H * B floats per layer
            const int64_t ss = ((int64_t)layer * num_blocks + src) * scale_words;
            const int64_t sd = ((int64_t)layer * num_blocks + dst) * scale_words;
            for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < scale_words; w += step) {
                k_scale[sd + w] = k_scale[ss + w];
                v_scale[sd + w] = v_scale[ss + w];
            }
        }
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

// Swap: blocks <-> a contiguous buffer, [n][L][K block, V block(, K scales, V scales)],
// every piece a whole number of 16-byte words. gather = pool -> buffer,
// scatter = buffer -> pool (icman.com.cn/news/78786 §4.2 swaps a preempted
// request's KV out to host memory and back).
__global__ void __launch_bounds__(kCopyThreads)
swap_blocks_kernel(const int32_t *__restrict__ blocks, int32_t n, uint4 *k_pool, uint4 *v_pool, uint4 *k_scale,
                   uint4 *v_scale, int32_t num_layers, int32_t num_blocks, int64_t block_words, int64_t scale_words,
                   uint4 *buf, int32_t to_buffer, uint32_t *status) {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();   // successors start once this grid's inputs are final
    const int64_t per = 2 * block_words + 2 * scale_words;      // words of one (block, layer) in the buffer
    const int64_t jobs = (int64_t)n * num_layers;
    for (int64_t y = blockIdx.y; y < jobs; y += gridDim.y) {
        const int32_t i = (int32_t)(y / num_layers);
        const int32_t layer = (int32_t)(y - (int64_t)i * num_layers);
        const int32_t b = blocks[i];
        if (b < 0 || b >= num_blocks) {
            if (status && blockIdx.x == 0 && threadIdx.x == 0 && layer == 0) atomicOr(status, PKV_DEV_BAD_PAIR);
            continue;
        }
        uint4 *slot = buf + y * per;
        const int64_t pb = ((int64_t)layer * num_blocks + b) * block_words;
        const int64_t ps = ((int64_t)layer * num_blocks + b) * scale_words;
        // kSwapUnroll independent 16-byte loads in flight per thread, then their stores
        // (one word per thread per CTA left too few bytes in flight to cover the latency)
        for (int64_t w0 = (int64_t)blockIdx.x * kSwapChunk + threadIdx.x; w0 < per; w0 += (int64_t)gridDim.x * kSwapChunk) {
            uint4 *pool_word[kSwapUnroll];
            uint4 val[kSwapUnroll];
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const int64_t w = w0 + u * kCopyThreads;
                pool_word[u] = nullptr;
                if (w >= per) continue;
                if (w < block_words) pool_word[u] = k_pool + pb + w;
                else if (w < 2 * block_words) pool_word[u] = v_pool + pb + (w - block_words);
                else if (w < 2 * block_words + scale_words) pool_word[u] = k_scale + ps + (w - 2 * block_words);
                else pool_word[u] = v_scale + ps + (w - 2 * block_words - scale_words);
                val[u] = to_buffer ? __ldcs(pool_word[u]) : __ldcs(slot + w);
            }
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const int64_t w = w0 + u * kCopyThreads;
                if (w < per) {
                    if (to_buffer) __stcs(slot + w, val[u]);
                    else *pool_word[u] = val[u];
                }
            }
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status swap_blocks(const pkv_pool *pool, const int32_t *blocks, int32_t n, void *buf, bool to_buffer,
                       uint32_t *status, void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (n < 0) return fail(PKV_ERR_INVALID_ARG, "n < 0");
    if (n == 0) return PKV_OK;
    if (!blocks || !buf || (reinterpret_cast<uintptr_t>(blocks) & 3u) || !aligned16(buf))
        return fail(PKV_ERR_INVALID_ARG, "blocks (4-byte aligned) and buffer (16-byte aligned) are required");
    const bool q8 = d.kv_dtype == PKV_KV_E4M3;
    if (q8 && !pool->k_scale) return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    // The buffer may be device memory or pinned host memory mapped into the device's
    // address space (the kernel then moves the blocks over the host link itself, with
    // no staging copy). Anything else would fault in the kernel, so it is refused here.
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, buf) != cudaSuccess) {
        cudaGetLastError();
        return fail(PKV_ERR_INVALID_ARG, "swap buffer: not a CUDA-visible pointer");
    }
    if (attr.type == cudaMemoryTypeHost) {
        if (!attr.devicePointer) return fail(PKV_ERR_INVALID_ARG, "swap buffer: pinned host memory not mapped to the device");
        buf = attr.devicePointer;
    } else if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) {
        return fail(PKV_ERR_INVALID_ARG, "swap buffer: must be device memory or pinned (mapped) host memory");
    }
    const int64_t block_words = (int64_t)d.block_size * d.num_heads * d.head_dim * kv_elem_bytes(d) / 16;
    const int64_t scale_words = q8 ? (int64_t)d.block_size * d.num_heads * 4 / 16 : 0;
    const int64_t per = 2 * block_words + 2 * scale_words;
    int gx = (int)((per + kSwapChunk - 1) / kSwapChunk);
    gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
    const int64_t jobs = (int64_t)n * d.num_layers;
    const int gy = (int)(jobs < 65535 ? jobs : 65535);
    cudaError_t e = launch_pdl(swap_blocks_kernel, dim3(gx, gy), dim3(kCopyThreads), 0,
                               static_cast<cudaStream_t>(stream), blocks, n, static_cast<uint4 *>(pool->k_pool),
                               static_cast<uint4 *>(pool->v_pool), reinterpret_cast<uint4 *>(pool->k_scale),
                               reinterpret_cast<uint4 *>(pool->v_scale), d.num_layers, d.num_blocks, block_words,
                               scale_words, static_cast<uint4 *>(buf), to_buffer ? 1 : 0, status);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "swap launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

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
    const PoolLayer pl = pool_layer(pool, layer);
    const int64_t nslots = (int64_t)d.num_blocks * d.block_size;
    cudaError_t e;
    if (d.kv_dtype == PKV_KV_E4M3) {
        if (!pl.k_scale) return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
        const int64_t warps = (int64_t)num_tokens * d.num_heads;
        const int64_t want = (warps * 32 + kAppendThreads - 1) / kAppendThreads;
        const int grid = (int)(want < 65535 * 16 ? want : 65535 * 16);
        auto kern = d.head_dim == 64 ? append_q8_kernel<64> : append_q8_kernel<128>;
        e = launch_pdl(kern, dim3(grid), dim3(kAppendThreads), 0, static_cast<cudaStream_t>(stream),
                       static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, num_tokens,
                       reinterpret_cast<unsigned char *>(pl.k), reinterpret_cast<unsigned char *>(pl.v), pl.k_scale,
                       pl.v_scale, nslots, d.block_size, d.num_heads, d.layout, status);
    } else {
        const int64_t total = (int64_t)num_tokens * d.num_heads * wpr;
        const int64_t want = (total + kAppendThreads - 1) / kAppendThreads;
        const int grid = (int)(want < 65535 * 16 ? want : 65535 * 16);
        e = launch_pdl(append_kernel, dim3(grid), dim3(kAppendThreads), 0, static_cast<cudaStream_t>(stream),
                       static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, num_tokens,
                       reinterpret_cast<uint4 *>(pl.k), reinterpret_cast<uint4 *>(pl.v), nslots, d.block_size,
                       d.num_heads, wpr, d.layout, status);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

size_t pkv_swap_bytes_per_block(const pkv_pool *pool) {
    if (!pool) return 0;
    const pkv_pool_desc &d = pool->desc;
    const size_t block = (size_t)d.block_size * d.num_heads * d.head_dim * kv_elem_bytes(d);
    const size_t scales = d.kv_dtype == PKV_KV_E4M3 ? (size_t)d.block_size * d.num_heads * 4 : 0;
    return (size_t)d.num_layers * 2 * (block + scales);
}

pkv_status pkv_gather_blocks(const pkv_pool *pool, const int32_t *blocks, int32_t n, void *dst, uint32_t *status,
                             void *stream) {
    return swap_blocks(pool, blocks, n, dst, true, status, stream);
}

pkv_status pkv_scatter_blocks(const pkv_pool *pool, const int32_t *blocks, int32_t n, const void *src,
                              uint32_t *status, void *stream) {
    return swap_blocks(pool, blocks, n, const_cast<void *>(src), false, status, stream);
}

pkv_status pkv_copy_blocks(const pkv_pool *pool, const int32_t *pairs, int32_t num_pairs, uint32_t *status,
                           void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs < 0");
    if (num_pairs == 0) return PKV_OK;
    if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 3u)) return fail(PKV_ERR_INVALID_ARG, "bad pairs pointer");
    const bool q8 = d.kv_dtype == PKV_KV_E4M3;
    if (q8 && !pool->k_scale) return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    const int64_t block_words = (int64_t)d.block_size * d.num_heads * d.head_dim * kv_elem_bytes(d) / 16;
    const int64_t scale_words = q8 ? (int64_t)d.block_size * d.num_heads * 4 / 16 : 0;
    const int64_t per_row = (int64_t)kCopyThreads * kCopyUnroll;
    int gx = (int)((block_words + per_row - 1) / per_row);
    if (gx < 1) gx = 1;
    const int64_t jobs = (int64_t)num_pairs * d.num_layers;
    const int gy = (int)(jobs < 65535 ? jobs : 65535);
    cudaError_t e = launch_pdl(copy_blocks_kernel, dim3(gx, gy), dim3(kCopyThreads), 0,
                               static_cast<cudaStream_t>(stream), pairs, num_pairs,
                               static_cast<uint4 *>(pool->k_pool), static_cast<uint4 *>(pool->v_pool), d.num_layers,
                               d.num_blocks, block_words, reinterpret_cast<uint4 *>(pool->k_scale),
                               reinterpret_cast<uint4 *>(pool->v_scale), scale_words, status);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "copy launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // extern "C"
