// The shared-prefix (cascade) pass for an FP8 E4M3 cache, head_dim 128, HND layout.
//
// What it computes: when sequences share their leading blocks (a forked prompt, prefix-
// cache hits: icman.com.cn/news/78786 §3.4, hnwysp.cn/news/103996 §3.3), the prefix's K/V
// are read once per group and attended by all the group's decode queries. For group g,
// head h and key split k, every member s gets the unnormalised piece
//   o[d] = sum_t 2^(x_t - m) V_t[d],  l = sum_t 2^(x_t - m),  m,
// over the split's keys t, with x_t = scale * log2(e) * q[s][h] . K_t, K_t and V_t the
// dequantised rows (code x row scale), and m the reference below. The decode kernel's
// combine merges these pieces with the attention over each member's private tokens, so
// the cascade gives the same attention up to the order of rounding (m.lqnn.cn/news/240480
// §6.2 for the quantised cache).
//
// Design: the fp16 cache's prefix pass runs on tcgen05 from fp16 tiles; here the tiles are
// E4M3 codes, converted in registers where the warp-level tensor cores (mma.sync m16n8k16,
// fp16 operands, fp32 sums) read them, as the E4M3 decode kernel does:
// * A producer warp streams 64-key tiles of K and V codes by TMA (128-byte swizzled, so
//   the fragment loads are conflict-free) and their row scales by 16-byte cp.async copies
//   into a 3-stage ring guarded by mbarriers.
// * Consumer warp w of CTA half x takes members 64 x + 16 w .. + 15 (the group's queries are
//   real rows of the products: no padding, unlike single-query decode); a group of more
//   than 64 members has its second 64 in a second CTA, which reads the same K/V tiles.
//   S = Q K^T with Q as the A operand (fp16 rows from global memory) and the codes of K as
//   B; the K row scale multiplies the scores. The softmax reference is the running max of
//   x_t + log2(V row scale), so each weight 2^(x_t - m) x scale is at most 1 and is
//   rounded to fp16; O += P V with P taken straight from the S fragments and V through
//   ldmatrix.trans (codes of two keys at one dim pair, split by a byte permute).
// * Every wait is bounded (1 s, then PKV_DEV_TIMEOUT): no trap, no hang.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace {

using namespace pkv;

constexpr int kD = 128;                           // head dim = bytes of one E4M3 row
constexpr int kTok = 64;                          // keys per tile
constexpr int kQW = 16;                           // member queries per consumer warp
constexpr int kCW = 4;                            // consumer warps: 64 members per CTA
constexpr int kHalves = PKV_MAX_GROUP_SEQS / (kQW * kCW);   // CTAs per (group, head, split)
constexpr int kThreads = (kCW + 1) * 32;          // + one producer warp
constexpr int kStages = 3;
constexpr int kTileBytes = kTok * kD;             // one K (or V) tile of codes
constexpr int kScaleOff = 2 * kTileBytes;         // then the K scales and the V scales of the tile
constexpr int kStageBytes = (2 * kTileBytes + 2 * kTok * 4 + 1023) / 1024 * 1024;   // 1024-aligned tiles
constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStages * 8 + 16 + 1024;
constexpr int kSplitKeys = 128;                   // the prefix's key splits are whole 128-key tiles
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

struct Q8PrefixParams {
    const __half *q;                 // [S][H][D]
    const pkv_prefix_group *groups;  // [gridDim.z]
    const int32_t *tables;           // [S][max_blocks]
    const float *k_scale;            // this layer's row scales [N][H][B]
    const float *v_scale;
    float *pieces;                   // [S][H][PKV_MAX_PREFIX_SPLITS][D + 4]
    uint32_t *status;
    int32_t S, H, max_blocks, B, lgB, N, splits, early;
    float scale_log2;                // scale * log2(e)
};

// Bounded wait on a phase: false (and PKV_DEV_TIMEOUT) past the limit; after one
// timeout in the CTA every later wait returns at once.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int32_t *timed_out,
                                             uint32_t *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*timed_out) return false;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*timed_out) return false;
        if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
            *timed_out = 1;
            atomicOr(status, PKV_DEV_TIMEOUT);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
prefix_attention_q8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const Q8PrefixParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
    const uint32_t st0 = ptx::smem_addr(base);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kStages * kStageBytes);
    volatile int32_t *timed_out = reinterpret_cast<volatile int32_t *>(bars + 2 * kStages);
    const uint32_t full0 = ptx::smem_addr(bars), empty0 = full0 + 8 * kStages;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t split = blockIdx.x / kHalves, half = blockIdx.x % kHalves, h = blockIdx.y;
    const int32_t H = p.H, B = p.B, lgB = p.lgB;
    const bool early = p.early != 0;
    if (!early) {
        ptx::grid_dependency_wait();
        ptx::launch_dependents();
    }
    const pkv_prefix_group grp = p.groups[blockIdx.z];
    const int32_t P = grp.prefix_tokens, n = grp.num_seqs, first = grp.first_seq;
    if (n < 1 || n > PKV_MAX_GROUP_SEQS || first < 0 || first > p.S - n || P < 0 || P > p.max_blocks * B ||
        (P & (B - 1)) != 0) {
        if (tid == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        if (early) {
            ptx::grid_dependency_wait();
            ptx::launch_dependents();
        }
        return;
    }
    const int32_t per = ((P + kSplitKeys - 1) / kSplitKeys + p.splits - 1) / p.splits;   // 128-key tiles per split
    const int32_t kv_begin = min(P, split * per * kSplitKeys);
    const int32_t kv_end = min(P, kv_begin + per * kSplitKeys);
    auto piece_of = [&](int32_t m) {
        return p.pieces + (((size_t)(first + m) * H + h) * PKV_MAX_PREFIX_SPLITS + split) * (kD + 4);
    };
    const int32_t m0 = half * kQW * kCW;               // this CTA's first member
    const int32_t nm = min(n - m0, kQW * kCW);          // and its member count
    if (kv_begin >= kv_end || nm <= 0) {
        // no keys in this split: an empty piece for each of this CTA's members (none left
        // for the second half of a group of at most 64)
        if (early) {
            ptx::grid_dependency_wait();
            ptx::launch_dependents();
        }
        for (int32_t i = tid; i < max(nm, 0) * (kD + 4); i += kThreads) {
            const int32_t m = i / (kD + 4), cc = i - m * (kD + 4);
            piece_of(m0 + m)[cc] = cc == kD ? -INFINITY : 0.f;
        }
        return;
    }
    const int32_t nt = (kv_end - kv_begin + kTok - 1) / kTok;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(full0 + 8 * i, 1);
            ptx::mbar_init(empty0 + 8 * i, kCW);
        }
        *timed_out = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();

    if (warp == kCW) {
        // ================= producer: K/V code tiles by TMA (one box per block, lane i box i),
        // the tiles' row scales by 16-byte cp.async copies
        if (lane == 0) {
            ptx::prefetch_tensormap(&kmap);
            ptx::prefetch_tensormap(&vmap);
        }
        const int32_t rows = B < kTok ? B : kTok;
        const uint32_t box_bytes = (uint32_t)rows * kD;
        const int32_t *trow = p.tables + (size_t)first * p.max_blocks;
        constexpr int KW = 4;                             // 128 table entries in registers
        int32_t win_lb0 = -1, win[KW];
        auto entry = [&](int32_t e) {
            int32_t v = 0;
#pragma unroll
            for (int jj = 0; jj < KW; ++jj) {
                const int32_t x = __shfl_sync(0xffffffffu, win[jj], e & 31);
                if ((e >> 5) == jj) v = x;
            }
            return v;
        };
        for (int32_t j = 0; j < nt; ++j) {
            const int stage = j % kStages;
            if (early && j == kStages) {
                ptx::grid_dependency_wait();
                ptx::launch_dependents();
            }
            if (j >= kStages) wait_bounded(empty0 + 8 * stage, ((j / kStages) - 1) & 1, timed_out, p.status);
            const int32_t t0 = kv_begin + j * kTok;
            const int32_t ntok = min(kTok, kv_end - t0);
            const int32_t lb = t0 >> lgB;
            const int32_t nbox = B < kTok ? (ntok + B - 1) >> lgB : 1;
            const int32_t r0 = B < kTok ? 0 : t0 & (B - 1);
            if (win_lb0 < 0 || lb < win_lb0 || lb + nbox > win_lb0 + 32 * KW) {
                win_lb0 = lb;
#pragma unroll
                for (int jj = 0; jj < KW; ++jj) {
                    const int32_t e = lb + 32 * jj + lane;
                    win[jj] = e < p.max_blocks ? __ldg(trow + e) : 0;
                }
            }
            const uint32_t dst = st0 + stage * kStageBytes;
            const uint32_t bar = full0 + 8 * stage;
            {
                // scales of tokens 4 l .. 4 l + 3 (lanes 0-15: K, 16-31: V); a run of four never
                // leaves its block (block sizes and tile starts are multiples of 4)
                const int32_t i = (lane & 15) * 4;
                const int32_t t = t0 + min(i, ntok - 1);
                int32_t blk = entry((t >> lgB) - win_lb0);
                if (blk < 0 || blk >= p.N) blk = 0;        // flagged with the boxes below
                const size_t y = ((size_t)blk * H + h) * B + (t & (B - 1));
                if (i < ntok) {
                    if (lane < 16) ptx::cp_async_16_cg(dst + kScaleOff + i * 4, p.k_scale + y);
                    else ptx::cp_async_16_cg(dst + kScaleOff + kTok * 4 + i * 4, p.v_scale + y);
                }
                ptx::cp_async_mbar_arrive(bar);
                __syncwarp();
            }
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)nbox * box_bytes * 2);
            int32_t blk = entry(lb + lane - win_lb0);
            if (lane < nbox) {
                if (blk < 0 || blk >= p.N) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    blk = 0;
                }
                const int32_t y = ((blk * H + h) << lgB) + r0;
                ptx::tma_load_2d(dst + lane * box_bytes, &kmap, 0, y, bar);
                ptx::tma_load_2d(dst + kTileBytes + lane * box_bytes, &vmap, 0, y, bar);
            }
            __syncwarp();
        }
        if (early && nt <= kStages) {
            ptx::grid_dependency_wait();
            ptx::launch_dependents();
        }
        return;
    }

    // ================= consumers: warp w attends members m0 + 16 w .. + 15
    if (early) ptx::grid_dependency_wait();   // q is read and the pieces written only after it
    const int g = lane >> 2, c = lane & 3;
    const int32_t mb = m0 + warp * kQW;
    const bool active = mb < n;
    // Q of rows g and g + 8: dims [32 c, 32 c + 32) as 16 fp16 pairs each (zero past the
    // group). k step st pairs word st of a K row's bytes [32 c, 32 c + 32) (dims
    // 32 c + 4 st .. + 3) with words 2 st, 2 st + 1 of these: a consistent order of the
    // dot product's terms.
    uint32_t qa[2][16];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int32_t m = mb + g + 8 * rr;
        const bool ok = active && m < n;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)(first + (ok ? m : 0)) * H + h) * kD + 32 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
            qa[rr][4 * i + 0] = v.x;
            qa[rr][4 * i + 1] = v.y;
            qa[rr][4 * i + 2] = v.z;
            qa[rr][4 * i + 3] = v.w;
        }
    }
    // output rows g, g + 8: n-tile 2 u + par holds dims 16 u + 2 n + par (n = 2 c, 2 c + 1)
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;

    for (int32_t j = 0; j < nt; ++j) {
        const int stage = j % kStages;
        const uint32_t kb = st0 + stage * kStageBytes, vb = kb + kTileBytes;
        wait_bounded(full0 + 8 * stage, (j / kStages) & 1, timed_out, p.status);
        if (active) {
            const int32_t ntok = min(kTok, kv_end - (kv_begin + j * kTok));
            const bool full = ntok == kTok;
            // ---- S = Q K^T, n-tile jt = keys 8 jt .. 8 jt + 7 (lane (g, c): key 8 jt + g, whose
            // (row & 7) == g picks the swizzled chunks)
            float s[8][4];
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                const uint32_t row = kb + (8 * jt + g) * kD;
                const uint4 w0 = ptx::lds128(row + (((2 * c) ^ g) << 4));
                const uint4 w1 = ptx::lds128(row + (((2 * c + 1) ^ g) << 4));
                const uint32_t kw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
                for (int st = 0; st < 8; ++st) {
                    uint32_t b0, b1;
                    q8::e4m3x4_to_half2x2(kw[st], b0, b1);
                    ptx::mma_16816(d0, d1, d2, d3, qa[0][2 * st], qa[1][2 * st], qa[0][2 * st + 1],
                                   qa[1][2 * st + 1], b0, b1, d0, d1, d2, d3);
                }
                s[jt][0] = d0;
                s[jt][1] = d1;
                s[jt][2] = d2;
                s[jt][3] = d3;
            }
            // ---- scores, reference and weights. Lane (g, c) holds keys 8 jt + 2 c + e of rows
            // g (s[.][e]) and g + 8 (s[.][2 + e]).
            float vsc[8][2];
            float tm[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                const int32_t k0 = 8 * jt + 2 * c;
                const uint2 ks = ptx::lds64(kb + kScaleOff + k0 * 4);
                const uint2 vs = ptx::lds64(kb + kScaleOff + kTok * 4 + k0 * 4);
                const float kf[2] = {__uint_as_float(ks.x), __uint_as_float(ks.y)};
                vsc[jt][0] = __uint_as_float(vs.x);
                vsc[jt][1] = __uint_as_float(vs.y);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool ok = full || k0 + e < ntok;
                    const float lv = ptx::lg2(fmaxf(vsc[jt][e], 0x1p-100f));
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const float x = ok ? s[jt][2 * rr + e] * kf[e] * sl2 : -INFINITY;
                        s[jt][2 * rr + e] = x;
                        tm[rr] = fmaxf(tm[rr], ok ? x + lv : -INFINITY);
                    }
                }
            }
            float alpha[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                tm[rr] = fmaxf(tm[rr], __shfl_xor_sync(0xffffffffu, tm[rr], 1));
                tm[rr] = fmaxf(tm[rr], __shfl_xor_sync(0xffffffffu, tm[rr], 2));
                const float mn = fmaxf(mr[rr], tm[rr]);
                alpha[rr] = mn == -INFINITY ? 1.f : ptx::ex2(mr[rr] - mn);   // mr = -inf: 0
                mr[rr] = mn;
                lr[rr] *= alpha[rr];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[0];
                o[i][2] *= alpha[1];
                o[i][3] *= alpha[1];
            }
            // weights (x weight x V scale in fp16) as the A operand of P V: k step i (keys
            // 16 i .. 16 i + 15) = n-tiles 2 i, 2 i + 1 of S
            uint32_t pa[8][2];
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                float w[4];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float x = s[jt][2 * rr + e];
                        const float pw = x == -INFINITY ? 0.f : ptx::ex2(x - mr[rr]);
                        lr[rr] += pw;
                        w[2 * rr + e] = x == -INFINITY ? 0.f : pw * vsc[jt][e];
                    }
                pa[jt][0] = ptx::pack_half2(w[0], w[1]);
                pa[jt][1] = ptx::pack_half2(w[2], w[3]);
            }
            // ---- O += P V over 4 k steps x 8 chunks of 16 dims. ldmatrix (transposed) gives
            // lane (g, c) the codes of keys 2 c, 2 c + 1 at dims 2 g, 2 g + 1 of a chunk.
            const int mi = lane >> 3;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t mk01 = 0xFFFFFFFFu, mk89 = 0xFFFFFFFFu;   // past the split: codes to 0
                if (!full) {
                    const int32_t tc = 16 * i + 2 * c;
                    mk01 = (tc < ntok ? 0x00FF00FFu : 0u) | (tc + 1 < ntok ? 0xFF00FF00u : 0u);
                    mk89 = (tc + 8 < ntok ? 0x00FF00FFu : 0u) | (tc + 9 < ntok ? 0xFF00FF00u : 0u);
                }
                const uint32_t vrow = vb + (16 * i + (mi & 1) * 8 + (lane & 7)) * kD;
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    uint32_t r[4];
                    ptx::ldmatrix_x4_trans(vrow + (((2 * hh + (mi >> 1)) ^ (lane & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        const int u = 2 * hh + uu;
                        uint32_t be0, bo0, be1, bo1;   // (even dim, odd dim) x (keys 2c.., keys 2c+8..)
                        q8::e4m3x4_to_half2x2(ptx::prmt(r[2 * uu], 0u, 0x3120u) & mk01, be0, bo0);
                        q8::e4m3x4_to_half2x2(ptx::prmt(r[2 * uu + 1], 0u, 0x3120u) & mk89, be1, bo1);
                        ptx::mma_16816(o[2 * u][0], o[2 * u][1], o[2 * u][2], o[2 * u][3], pa[2 * i][0], pa[2 * i][1],
                                       pa[2 * i + 1][0], pa[2 * i + 1][1], be0, be1, o[2 * u][0], o[2 * u][1],
                                       o[2 * u][2], o[2 * u][3]);
                        ptx::mma_16816(o[2 * u + 1][0], o[2 * u + 1][1], o[2 * u + 1][2], o[2 * u + 1][3],
                                       pa[2 * i][0], pa[2 * i][1], pa[2 * i + 1][0], pa[2 * i + 1][1], bo0, bo1,
                                       o[2 * u + 1][0], o[2 * u + 1][1], o[2 * u + 1][2], o[2 * u + 1][3]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty0 + 8 * stage);
    }
    if (!active) return;
    // ---- the pieces of rows g and g + 8: l summed over the row's four lanes
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float l = lr[rr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int32_t m = mb + g + 8 * rr;
        if (m < n) {
            float *piece = piece_of(m);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4 *>(piece + 16 * u + 4 * c) =
                    make_float4(o[2 * u][2 * rr], o[2 * u + 1][2 * rr], o[2 * u][2 * rr + 1], o[2 * u + 1][2 * rr + 1]);
            if (c == 0) *reinterpret_cast<float4 *>(piece + kD) = make_float4(mr[rr], l, 0.f, 0.f);
        }
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// [N * H * B rows][128 codes] of one pool layer; boxes of min(B, 64) rows, 128-byte swizzled.
pkv_status encode_codes(CUtensorMap *map, const void *base, const pkv_pool_desc &d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)d.num_blocks * d.num_heads * d.block_size};
    const cuuint64_t strides[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)(d.block_size < kTok ? d.block_size : kTok)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices];
cudaError_t g_attr_err[kMaxDevices];

}  // namespace

namespace pkv {

pkv_status prefix_attention_q8(const pkv_pool *pool, int32_t layer, const void *q, const pkv_prefix_group *groups,
                               int32_t num_groups, int32_t splits, const int32_t *block_tables, int32_t max_blocks,
                               int32_t num_seqs, float scale, void *pieces, uint32_t *status, uint32_t flags,
                               void *stream) {
    const pkv_pool_desc &d = pool->desc;
    const PoolLayer pl = pool_layer(pool, layer);
    if (!pl.k_scale || !pl.v_scale)
        return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    CUtensorMap kmap, vmap;
    pkv_status st = encode_codes(&kmap, pl.k, d);
    if (st != PKV_OK) return st;
    st = encode_codes(&vmap, pl.v, d);
    if (st != PKV_OK) return st;
    Q8PrefixParams prm = {};
    prm.q = static_cast<const __half *>(q);
    prm.groups = groups;
    prm.tables = block_tables;
    prm.k_scale = pl.k_scale;
    prm.v_scale = pl.v_scale;
    prm.pieces = static_cast<float *>(pieces);
    prm.status = status;
    prm.S = num_seqs;
    prm.H = d.num_heads;
    prm.max_blocks = max_blocks;
    prm.B = d.block_size;
    prm.lgB = __builtin_ctz((unsigned)d.block_size);   // a supported block size is a power of two
    prm.N = d.num_blocks;
    prm.splits = splits;
    prm.early = (flags & PKV_ATTN_INPUTS_EARLY) ? 1 : 0;
    const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)kD);
    prm.scale_log2 = (float)(sc * 1.4426950408889634);   // log2(e)

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_CUDA, "no usable CUDA device");
    std::call_once(g_attr_once[dev], [dev] {
        g_attr_err[dev] = cudaFuncSetAttribute(prefix_attention_q8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemBytes);
    });
    if (g_attr_err[dev] != cudaSuccess)
        return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(g_attr_err[dev]));
    cudaError_t e = launch_pdl(prefix_attention_q8_kernel, dim3(splits * kHalves, d.num_heads, num_groups), dim3(kThreads),
                               (size_t)kSmemBytes, static_cast<cudaStream_t>(stream), kmap, vmap, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "E4M3 prefix pass launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace pkv
