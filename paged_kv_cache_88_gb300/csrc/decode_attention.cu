// Paged decode attention for sm_103a (GB300).
//
// What it computes (per layer): for every sequence s and head h,
//   out[s][h] = softmax_t(scale * q[s][h] . K_s[t]) V_s[t],   t = 0..T_s-1,
// with token t of sequence s read from physical block table[s][t / B], slot
// t % B (m.lqnn.cn/news/240480 §3.3 remaps [batch, head, pos, dim] to
// [page, slot, head, dim] through the page table; icman.com.cn/news/78786 §2.4
// walks the block table and loads each block's K/V). Single-query decode is a
// GEMV over the cache: about 0.5 FMA per byte, so the kernel is bound by HBM
// bandwidth, not by arithmetic.
//
// Design (GB300-first; the pages' A100 kernel advice -- table in shared memory,
// vectorised loads, many heads per launch -- is prior art, not the blueprint):
//
// * Work unit = one tile of 64 tokens of one (sequence, head). All tiles of the
//   batch are numbered (s, h, t) and the launch's CTAs take equal contiguous
//   ranges of that list (a persistent grid of SMs x resident CTAs). Mixed
//   context lengths therefore cost no tail imbalance: every CTA streams the same
//   number of tiles (+-1).
// * A producer warp walks the CTA's range and issues TMA tensor loads of each
//   tile's K and V rows (one box per block, or a 64-row box inside a large
//   block; lane i issues box i) into a 2-stage shared-memory ring guarded by
//   mbarriers; it keeps a window of 128 block-table entries of the current
//   sequence in registers (one coalesced load serves every head of the
//   sequence). The query row of a new (s, h) rides along in the same stage as a
//   1-D bulk copy; an FP8 E4M3 cache's per-row scales as 16-byte cp.async copies.
// * Consumers, fp16 cache (and E4M3 at head_dim 64): four warps split each tile
//   into 16 groups of 8 lanes; a group owns four rows (tokens) of the tile, a
//   lane 8 x (D / 64) elements of the head dim. Rows are read from shared memory
//   as 16-byte words, a group covering 128 contiguous bytes per load (no bank
//   conflicts). q.K accumulates fp16 x fp16 products in fp32 (mixed-precision
//   FMA; the products are exact) and finishes with three xor-shuffles; p.V runs
//   as packed fp32 pair FMAs. Each group keeps its own online-softmax state
//   (running max m, sum l, unnormalised o), so no block-wide synchronisation
//   happens per tile.
// * Consumers, E4M3 cache at head_dim 128: the tiles land 128-byte swizzled and
//   each warp runs q.K and p.V for 16 tokens of a tile on the warp-level tensor
//   cores (mma.sync m16n8k16, codes converted to fp16 operands, fp32 sums); the
//   softmax reference covers x + log2(V row scale), so the weights x scale enter
//   p.V as fp16 <= 1.
// * When an (s, h) ends inside the CTA, the per-warp states are merged through
//   shared memory. A (s, h) that lies wholly in the CTA is written straight to
//   out; one split across CTAs writes its piece (m, l, o) to the workspace and
//   the last CTA to arrive (an atomic counter, no waiting) merges the pieces and
//   writes out -- split-KV with the combine fused into the same launch. A
//   cascade member also merges the prefix pass's pieces of its shared prefix.
// * Optional in the same launch: the step's append (the producer stores each
//   sequence's new K/V row -- quantised for an E4M3 cache -- before the tile
//   that holds it), and an early start behind the previous kernel on the stream
//   (tables, lengths and the first tiles' K/V read before the grid dependency
//   resolves).
// * Every mbarrier wait has a time limit; on expiry the CTA flags
//   PKV_DEV_TIMEOUT, stops waiting and runs to the end (no trap, no hang).
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

#ifndef PKV_ATTN_TILE
#define PKV_ATTN_TILE 64
#endif
#ifndef PKV_ATTN_WARPS
#define PKV_ATTN_WARPS 4
#endif
#ifndef PKV_ATTN_STAGES
#define PKV_ATTN_STAGES 2
#endif
#ifndef PKV_ATTN_MIN_CTAS
#define PKV_ATTN_MIN_CTAS 3
#endif
// The E4M3 tile is half the bytes of the fp16 one and its consumers are issue-bound, so
// that variant runs 4 CTAs per SM (96 registers a thread) with one more stage each.
#ifndef PKV_ATTN_MIN_CTAS_Q8
#define PKV_ATTN_MIN_CTAS_Q8 4
#endif
// The E4M3 head_dim-128 variant (tensor-core consumers) holds q and the output as MMA
// fragments.
#ifndef PKV_ATTN_MIN_CTAS_MMA
#define PKV_ATTN_MIN_CTAS_MMA 4
#endif
#ifndef PKV_ATTN_ACQREL
#define PKV_ATTN_ACQREL 1
#endif

constexpr int kTile = PKV_ATTN_TILE;              // tokens per pipeline stage
constexpr int kConsumerWarps = PKV_ATTN_WARPS;    // warps that compute
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;   // + one producer warp
constexpr int kGroups = kConsumerWarps * 4;       // 8-lane groups
constexpr int kTokPerGroup = kTile / kGroups;     // rows of a tile one group owns
constexpr int kStagesF16 = PKV_ATTN_STAGES;
#ifndef PKV_ATTN_STAGES_Q8
#define PKV_ATTN_STAGES_Q8 2
#endif
constexpr int kStagesQ8 = PKV_ATTN_STAGES_Q8;
static_assert(kTile % kGroups == 0 && kTokPerGroup >= 1 && kTokPerGroup <= 4, "tile / group split");
constexpr int kMaxSeqs = 4096;
constexpr int kMaxCtasPerSm = 8;     // bound used to size the workspace
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr int kStatusBytes = 256;

struct Params {
    const __half *q;
    __half *out;
    const int32_t *tables;
    const int32_t *lens;
    float *pieces;       // [grid][2][D + 4]
    int32_t *counters;   // [S * H]
    uint32_t *status;
    // fused append (decode step): token s's K/V row (all heads) goes to slot
    // slots[s] of the layer before the tile holding it is read; null = no append
    const uint4 *k_new;  // [S][H][D] fp16 as 16-byte words
    const uint4 *v_new;
    const int64_t *slots;  // [S]
    unsigned char *k_layer;  // this layer's pools (fp16 elements or E4M3 codes)
    unsigned char *v_layer;
    float *k_scale;      // quantised cache: this layer's per-(token, head) scales, [N][H][B]
    float *v_scale;
    // shared-prefix cascade (null = none): sequence s attends here to tokens
    // [begin[s], T_s) and merges pre_splits prefix pieces (o[D], m, l) of
    // [S][H][PKV_MAX_PREFIX_SPLITS][D + 4] when begin[s] > 0
    const int32_t *begin;
    const float *pre;
    int32_t pre_splits;
    // 1: the tables, lengths, seq_begin and cached K/V rows were final before the
    // preceding kernel on the stream started, so they are read (and the first tiles'
    // K/V loads issued) before the grid dependency resolves; q, k_new, v_new, the
    // workspace and out are touched only after it
    int32_t early;
    // 1 (with early): the preceding kernel writes each sequence's last cached row (this
    // step's append), so the tile holding it is not among the tiles loaded early
    int32_t last_pending;
    int32_t S, H, max_blocks, B, N, layout;
    int32_t lgB;         // log2(B): B is a power of two
    float scale_log2;    // scale * log2(e)
};

// Shape of one pipeline stage: [K tile][V tile][q row][K scales][V scales].
// Q8 = the cache holds E4M3 codes with a scale per (token, head) row. kMma = the E4M3
// head_dim-128 variant, whose consumers run q.K and p.V on the warp-level tensor cores:
// its K and V tiles arrive 128-byte swizzled (16-byte chunk k of token row r at chunk
// k ^ (r & 7)), which needs every tile to start on a 1024-byte boundary.
template <int D, bool Q8>
struct Stage {
    static constexpr bool kMma = Q8 && D == 128;
    static constexpr int kAlign = kMma ? 1024 : 128;
    static constexpr int kElem = Q8 ? 1 : 2;          // bytes per K/V element
    static constexpr int kRow = D * kElem;            // bytes per token row
    static constexpr int kTileBytes = kTile * kRow;   // one K (or V) tile
    static constexpr int kQ = 2 * kTileBytes;         // offset of the query row (fp16)
    static constexpr int kScales = kQ + D * 2;        // offset of the K scales, then the V scales
    static constexpr int kBytes = ((kScales + (Q8 ? 2 * kTile * 4 : 0)) + kAlign - 1) / kAlign * kAlign;
    static constexpr int kStages = Q8 ? kStagesQ8 : kStagesF16;
    static_assert(kTileBytes % kAlign == 0, "tiles start on the stage alignment");
};

__host__ __device__ constexpr int piece_stride(int D) { return D + 4; }

// Element pair e (0..3) of chunk ch of one K or V row as fp16x2: from the fp16 words
// (fp16 cache), or converted from the row's E4M3 codes, four to a word, where it is used.
template <bool Q8, int NCH>
__device__ __forceinline__ uint32_t pair_of(const uint32_t (&codes)[NCH * 2], const uint32_t (&halves)[NCH][4],
                                            int ch, int e) {
    if constexpr (Q8) return q8::e4m3x2_to_half2(codes[ch * 2 + (e >> 1)] >> (16 * (e & 1)));
    else return halves[ch][e];
}

// The cascade's prefix pieces of the current (s, h), staged in shared memory while its
// tiles stream (the cascade is built for head_dim 128).
template <int D, bool Q8>
__host__ __device__ constexpr int pre_buf_floats() { return D == 128 ? PKV_MAX_PREFIX_SPLITS * (D + 4) : 0; }

// Shared memory: [stages][prefix pieces][reduction][seq arrays][barriers + flags]
template <int D, bool Q8>
__host__ __device__ constexpr size_t smem_bytes_t(int S) {
    return ((size_t)Stage<D, Q8>::kStages * Stage<D, Q8>::kBytes + (size_t)pre_buf_floats<D, Q8>() * sizeof(float) +
            (size_t)kConsumerWarps * (D + 2) * sizeof(float) + (size_t)(3 * S + 2) * sizeof(int32_t) + 15) / 16 * 16 +
           2 * Stage<D, Q8>::kStages * sizeof(uint64_t) + 16 + Stage<D, Q8>::kAlign;  // + slack to align the base
}

struct Smem {
    unsigned char *stage;  // kStages * stage bytes
    float *pre;            // [PKV_MAX_PREFIX_SPLITS][D + 4] (head_dim 128)
    float *red_o;          // [kConsumerWarps][D]
    float *red_m;          // [kConsumerWarps]
    float *red_l;          // [kConsumerWarps]
    int32_t *len;          // [S] tokens attended here (T_s - beg[s])
    int32_t *beg;          // [S] first token attended here (the cascade's prefix length, else 0)
    int32_t *base;         // [S + 1] exclusive prefix of H * ntiles
    uint64_t *full;        // [kStages]
    uint64_t *empty;       // [kStages]
    volatile int32_t *flags;  // [0] = timed out, [1] = last-arriver flag
};

template <int D, bool Q8>
__device__ __forceinline__ Smem carve(unsigned char *raw, int S) {
    constexpr int NS = Stage<D, Q8>::kStages;
    constexpr uintptr_t A = Stage<D, Q8>::kAlign;
    Smem m;
    uintptr_t p = (reinterpret_cast<uintptr_t>(raw) + A - 1) & ~(A - 1);
    m.stage = reinterpret_cast<unsigned char *>(p);
    p += (size_t)NS * Stage<D, Q8>::kBytes;
    m.pre = reinterpret_cast<float *>(p);
    p += (size_t)pre_buf_floats<D, Q8>() * sizeof(float);
    m.red_o = reinterpret_cast<float *>(p);
    p += (size_t)kConsumerWarps * D * sizeof(float);
    m.red_m = reinterpret_cast<float *>(p);
    p += kConsumerWarps * sizeof(float);
    m.red_l = reinterpret_cast<float *>(p);
    p += kConsumerWarps * sizeof(float);
    m.len = reinterpret_cast<int32_t *>(p);
    p += (size_t)S * sizeof(int32_t);
    m.beg = reinterpret_cast<int32_t *>(p);
    p += (size_t)S * sizeof(int32_t);
    m.base = reinterpret_cast<int32_t *>(p);
    p += (size_t)(S + 1) * sizeof(int32_t);
    p = (p + 15) & ~uintptr_t(15);
    m.full = reinterpret_cast<uint64_t *>(p);
    m.empty = m.full + NS;
    m.flags = reinterpret_cast<volatile int32_t *>(m.empty + NS);
    return m;
}

// Element index of chunk ch (8 consecutive elements) of the row owned by lane j
// of a group. fp16 rows: the 8 lanes read 128 contiguous bytes per chunk; E4M3
// rows (half as many bytes): lane j owns D/8 contiguous elements, one load.
template <int D, bool Q8>
__device__ __forceinline__ int chunk_elem(int j, int ch) {
    return Q8 ? j * (D / 8) + ch * 8 : ch * 64 + j * 8;
}

// Position in the CTA's tile range: sequence, head, tile of the (s, h).
struct Cursor {
    int32_t s, h, t, nt;
};

__device__ __forceinline__ int32_t ntiles_of(int32_t T) { return (T + kTile - 1) / kTile; }

__device__ __forceinline__ Cursor locate(const Smem &sm, int32_t S, int32_t H, int32_t g) {
    // largest s with base[s] <= g (g < total, so that s has tiles)
    int32_t lo = 0, hi = S - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (sm.base[mid] <= g) lo = mid; else hi = mid - 1;
    }
    Cursor c;
    c.s = lo;
    c.nt = ntiles_of(sm.len[lo]);
    int32_t r = g - sm.base[lo];
    c.h = r / c.nt;
    c.t = r - c.h * c.nt;
    return c;
}

__device__ __forceinline__ void advance(Cursor &c, const Smem &sm, int32_t S, int32_t H) {
    if (++c.t < c.nt) return;
    c.t = 0;
    if (++c.h < H) return;
    c.h = 0;
    do {
        ++c.s;
    } while (c.s < S && sm.len[c.s] == 0);
    if (c.s < S) c.nt = ntiles_of(sm.len[c.s]);
}

// First tile index of CTA c among `total` tiles split over `grid` CTAs.
__device__ __forceinline__ int32_t range_start(int64_t total, int32_t grid, int32_t c) {
    return static_cast<int32_t>((total * c) / grid);
}

// The CTA whose range holds tile g.
__device__ __forceinline__ int32_t cta_of(int64_t total, int32_t grid, int32_t g) {
    return static_cast<int32_t>(((int64_t)(g + 1) * grid - 1) / total);
}

// Bounded wait: false (and PKV_DEV_TIMEOUT) if the phase does not complete
// within the limit; after one timeout in the CTA every later wait returns at once.
__device__ __forceinline__ bool wait_phase(const Smem &sm, uint32_t bar, uint32_t parity, uint32_t *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (sm.flags[0]) return false;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (sm.flags[0]) return false;
        if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
            sm.flags[0] = 1;
            atomicOr(status, PKV_DEV_TIMEOUT);
            return false;
        }
    }
}

// Self-test of the wait limit: one thread waits, with the attention kernels' bounded
// wait, on an mbarrier that nothing ever completes. It gives up after the limit,
// flags PKV_DEV_TIMEOUT and the CTA exits (the context stays usable).
__global__ void wait_limit_probe_kernel(uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int32_t flags[2];
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        flags[0] = flags[1] = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    Smem sm = {};
    sm.flags = flags;
    if (threadIdx.x == 0) wait_phase(sm, b, 0, status);
}

// Fold the cascade's prefix pieces of (s, h) into a combine in progress: M, L
// and this thread's output elements O[r] (element tid + r * kConsumerThreads),
// all relative to 2^M. The pieces were written by an earlier launch.
template <int D, int DPT, bool kStaged>
__device__ __forceinline__ void merge_prefix(const Params &p, const float *staged, int32_t s, int32_t h, int tid,
                                             float &M, float &L, float (&O)[DPT]) {
    const float *base = kStaged ? staged : p.pre + ((size_t)s * p.H + h) * PKV_MAX_PREFIX_SPLITS * (D + 4);
    auto ld = [](const float *a) { return kStaged ? *a : __ldcg(a); };
    // every piece's m, l and this thread's o elements in one round of loads (unrolled to
    // the largest split count, predicated on the actual one), then the arithmetic
    float pm[PKV_MAX_PREFIX_SPLITS], pl[PKV_MAX_PREFIX_SPLITS], po[PKV_MAX_PREFIX_SPLITS][DPT];
#pragma unroll
    for (int k = 0; k < PKV_MAX_PREFIX_SPLITS; ++k) {
        const bool in = k < p.pre_splits;
        const float *pc = base + k * (D + 4);
        pm[k] = in ? ld(pc + D) : -INFINITY;
        pl[k] = in ? ld(pc + D + 1) : 0.f;
#pragma unroll
        for (int r = 0; r < DPT; ++r) {
            const int d = tid + r * kConsumerThreads;
            po[k][r] = (in && d < D) ? ld(pc + d) : 0.f;
        }
    }
    float Mn = M;
#pragma unroll
    for (int k = 0; k < PKV_MAX_PREFIX_SPLITS; ++k) Mn = fmaxf(Mn, pm[k]);
    if (Mn == -INFINITY) return;
    const float a = ptx::ex2(M - Mn);          // M = -inf: 0
    L *= a;
#pragma unroll
    for (int r = 0; r < DPT; ++r) O[r] *= a;
#pragma unroll
    for (int k = 0; k < PKV_MAX_PREFIX_SPLITS; ++k) {
        if (k >= p.pre_splits) break;
        const float w = ptx::ex2(pm[k] - Mn);  // an empty piece (m = -inf): 0
        L = fmaf(w, pl[k], L);
#pragma unroll
        for (int r = 0; r < DPT; ++r) O[r] = fmaf(w, po[k][r], O[r]);
    }
    M = Mn;
}

// Resident CTAs per SM the register budget is set for.
template <int D, bool Q8>
constexpr int min_ctas() {
    return D >= 256 ? 1 : (Stage<D, Q8>::kMma ? PKV_ATTN_MIN_CTAS_MMA : (Q8 ? PKV_ATTN_MIN_CTAS_Q8 : PKV_ATTN_MIN_CTAS));
}

// A cascade member's first tile: stage its prefix pieces with cp.async, so the combine at the
// end of the (s, h) reads them from shared memory (the previous combine's last barrier has
// released the buffer).
template <int D>
__device__ __forceinline__ void stage_prefix_pieces(const Params &p, const Smem &sm, int32_t s, int32_t h, int tid) {
    if constexpr (D == 128) {
        const float *src = p.pre + ((size_t)s * p.H + h) * PKV_MAX_PREFIX_SPLITS * (D + 4);
        const int n16 = p.pre_splits * (D + 4) / 4;
        for (int i = tid; i < n16; i += kConsumerThreads)
            ptx::cp_async_16_cg(ptx::smem_addr(sm.pre) + i * 16, src + i * 4);
        ptx::cp_async_commit();
    }
}

template <int D, bool Q8>
__global__ void __launch_bounds__(kThreads, min_ctas<D, Q8>())
decode_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const Params p) {
    using St = Stage<D, Q8>;
    constexpr bool kMma = St::kMma;
    static_assert(!kMma || kTile == 16 * kConsumerWarps, "kMma: 16 tokens of the tile per consumer warp");
    constexpr int NCH = D / 64;      // chunks of 8 elements per lane per row
    constexpr int SB = St::kBytes;
    constexpr int NS = St::kStages;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const Smem sm = carve<D, Q8>(smem_raw, p.S);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int32_t S = p.S, H = p.H;
    const int32_t cap = p.max_blocks * p.B;

    // ---- set-up: barriers (before the grid dependency resolves), then lengths
    // and the tile prefix over sequences. Dependents are let launch only once this
    // grid's own dependency has resolved, so a kernel that starts early finds every
    // kernel before its predecessor complete.
    const bool early = p.early != 0;
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.empty[i]), kConsumerWarps);
        }
        sm.flags[0] = 0;
        sm.flags[1] = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        ptx::prefetch_tensormap(&kmap);
        ptx::prefetch_tensormap(&vmap);
    }
    if (!early) ptx::grid_dependency_wait();
    for (int32_t s = tid; s < S; s += kThreads) {
        int32_t T = p.lens[s];
        if (T < 0 || T > cap) {
            atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            T = T < 0 ? 0 : cap;
        }
        int32_t b0 = 0;
        if (p.begin != nullptr) {
            b0 = p.begin[s];
            if (b0 < 0 || b0 > T || b0 % p.B != 0) {   // not a prefix in whole blocks: attend all here
                atomicOr(p.status, PKV_DEV_BAD_LENGTH);
                b0 = 0;
            }
        }
        sm.len[s] = T - b0;
        sm.beg[s] = b0;
    }
    __syncthreads();
    if (warp == 0) {
        int32_t running = 0;
        for (int32_t s0 = 0; s0 < S; s0 += 32) {
            const int32_t s = s0 + lane;
            const int32_t v = s < S ? H * ntiles_of(sm.len[s]) : 0;
            int32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (s < S) sm.base[s] = running + incl - v;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) sm.base[S] = running;
    }
    __syncthreads();

    const int32_t total = sm.base[S];
    const int32_t cta = blockIdx.x;

    // The consumers touch out and the workspace: after the grid dependency.
    if (early && warp < kConsumerWarps) ptx::grid_dependency_wait();
    // Nothing to attend here: out = 0 for an empty context (softmax over no
    // tokens contributes nothing), the merged prefix pieces for a sequence the
    // cascade's prefix covers entirely.
    if (warp < kConsumerWarps) {
        for (int32_t i = cta; i < S * H; i += gridDim.x) {
            const int32_t s = i / H;
            if (sm.len[s] != 0) continue;
            if (sm.beg[s] > 0) {
                constexpr int DPT = (D + kConsumerThreads - 1) / kConsumerThreads;
                float M = -INFINITY, L = 0.f, O[DPT];
#pragma unroll
                for (int r = 0; r < DPT; ++r) O[r] = 0.f;
                merge_prefix<D, DPT, false>(p, nullptr, s, i - s * H, tid, M, L, O);
                const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
                for (int r = 0; r < DPT; ++r) {
                    const int d = tid + r * kConsumerThreads;
                    if (d < D) p.out[(size_t)i * D + d] = __float2half_rn(O[r] * inv);
                }
            } else if (tid < D / 8) {
                reinterpret_cast<uint4 *>(p.out + (size_t)i * D)[tid] = make_uint4(0, 0, 0, 0);
            }
        }
    }
    // The tile list is split over min(CTAs, tiles) CTAs so that every working CTA
    // owns at least one tile (the piece count of a split (s, h) relies on it).
    const int32_t grid = min((int32_t)gridDim.x, total);
    if (cta >= grid) return;
    const int32_t g0 = range_start(total, grid, cta);
    const int32_t g1 = range_start(total, grid, cta + 1);
    const int32_t n = g1 - g0;
    if (n <= 0) return;

    const uint32_t stage0 = ptx::smem_addr(sm.stage);
    const uint32_t full0 = ptx::smem_addr(sm.full);
    const uint32_t empty0 = ptx::smem_addr(sm.empty);

    if (warp == kConsumerWarps) {
        // ================= producer warp
        const int32_t B = p.B, lgB = p.lgB;
        const int32_t rows = B < kTile ? B : kTile;           // rows per TMA box
        const uint32_t box_bytes = (uint32_t)rows * St::kRow;
        constexpr int W = D / 8;                              // 16-byte fp16 words per new row
        constexpr int NW = (2 * W + 31) / 32;                 // words of the new K+V rows per lane
        Cursor c = locate(sm, S, H, g0);
        // a window of 32 KW block-table entries of the current sequence in registers: lane l
        // holds entry win_lb0 + 32 j + l in win[j] (one load round serves every head of the
        // sequence while the window covers the tiles)
        constexpr int KW = 4;
        int32_t win_s = -1, win_lb0 = 0, win[KW];
        uint4 nw[NW];                                         // the new token's K/V row words
        int64_t new_slot = -1;                                // pending append of the current (s, h)
        // table entry win_lb0 + e (e per lane, 0 <= e < 32 KW)
        auto entry = [&](int32_t e) {
            int32_t v = 0;
#pragma unroll
            for (int jj = 0; jj < KW; ++jj) {
                const int32_t x = __shfl_sync(0xffffffffu, win[jj], e & 31);
                if ((e >> 5) == jj) v = x;
            }
            return v;
        };
        // K/V boxes (and, for E4M3, the scales) of the tile at cursor cc into `stage`,
        // with the stage's expected bytes including the q row when `first`
        auto issue_kv = [&](const Cursor &cc, int32_t stage, bool first) {
            const int32_t tt = cc.t * kTile;                   // the tile's first token attended here
            const int32_t ntok = min(kTile, sm.len[cc.s] - tt);
            const int32_t t0 = sm.beg[cc.s] + tt;              // its position in the sequence
            const int32_t lb = t0 >> lgB;                      // first logical block of the tile
            const int32_t nbox = B < kTile ? (ntok + B - 1) >> lgB : 1;
            const int32_t r0 = B < kTile ? 0 : t0 & (B - 1);   // first row inside the block
            if (cc.s != win_s || lb < win_lb0 || lb + nbox > win_lb0 + 32 * KW) {
                win_s = cc.s;
                win_lb0 = lb;
                const int32_t *row = p.tables + (size_t)cc.s * p.max_blocks;
#pragma unroll
                for (int jj = 0; jj < KW; ++jj) {
                    const int32_t e = lb + 32 * jj + lane;
                    win[jj] = e < p.max_blocks ? __ldg(row + e) : 0;
                }
            }
            const uint32_t bytes = (uint32_t)nbox * box_bytes * 2 + (first ? D * 2 : 0);
            const uint32_t dst = stage0 + stage * SB;
            const uint32_t bar = full0 + 8 * stage;
            if constexpr (Q8) {
                // the tile's scales ([N][H][B]: token i of the tile is row y_i) as 16-byte
                // asynchronous copies of four tokens each: lanes 0-15 the K scales of tokens
                // 4l..4l+3, lanes 16-31 the V scales. A run of four never leaves its block and
                // every copy is 16-byte aligned, because the block size (8..512) and the tile
                // start (the cascade's prefix length, whole blocks, plus a multiple of 64) are
                // multiples of 4 and the host refuses scale pools that are not 16-byte aligned.
                // Issued before lane 0's arrival, so the stage's phase cannot complete without them.
                static_assert(kTile == 64, "16-byte scale copies: 16 lanes x 4 tokens per pool");
                const int32_t i = (lane & 15) * 4;
                const int32_t t = t0 + min(i, ntok - 1);
                int32_t blk = entry((t >> lgB) - win_lb0);
                if (blk < 0 || blk >= p.N) blk = 0;      // flagged with the boxes below
                const size_t y = ((size_t)blk * H + cc.h) * B + (t & (B - 1));
                if (i < ntok) {
                    if (lane < 16) ptx::cp_async_16_cg(dst + St::kScales + i * 4, p.k_scale + y);
                    else ptx::cp_async_16_cg(dst + St::kScales + kTile * 4 + i * 4, p.v_scale + y);
                }
                ptx::cp_async_mbar_arrive(bar);
                __syncwarp();
            }
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, bytes);
            // lane i < nbox loads box i (block lb + i) of K and of V
            int32_t blk = entry(lb + lane - win_lb0);
            if (lane < nbox) {
                if (blk < 0 || blk >= p.N) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    blk = 0;
                }
                int32_t x, y;
                if (p.layout == PKV_LAYOUT_NHD) {
                    x = cc.h * D;
                    y = (blk << lgB) + r0;
                } else {
                    x = 0;
                    y = ((blk * H + cc.h) << lgB) + r0;
                }
                ptx::tma_load_2d(dst + lane * box_bytes, &kmap, x, y, bar);
                ptx::tma_load_2d(dst + St::kTileBytes + lane * box_bytes, &vmap, x, y, bar);
            }
        };
        auto issue_q = [&](const Cursor &cc, int32_t stage) {
            if (lane == 0)
                ptx::bulk_load(stage0 + stage * SB + St::kQ, p.q + ((size_t)cc.s * H + cc.h) * D, D * 2,
                               full0 + 8 * stage);
        };
        int32_t k0 = 0;   // the first tile of the main loop
        if (early) {
            // the first stages' K/V before the grid dependency resolves (not a tile holding an
            // appended token: this launch stores it first, or the preceding kernel does);
            // their q rows after it
            Cursor pend[NS];
            bool pend_q[NS];
            for (; k0 < n && k0 < NS; ++k0) {
                if ((p.k_new != nullptr || p.last_pending) && c.t == c.nt - 1) break;
                const bool first = (k0 == 0) || (c.t == 0);
                issue_kv(c, k0, first);
                pend[k0] = c;
                pend_q[k0] = first;
                advance(c, sm, S, H);
            }
            ptx::grid_dependency_wait();
            if (!p.last_pending) ptx::launch_dependents();
            for (int32_t k = 0; k < k0; ++k)
                if (pend_q[k]) issue_q(pend[k], k);
            __syncwarp();
        }
        for (int32_t k = k0; k < n; ++k) {
            const int32_t stage = k % NS;
            if (p.k_new != nullptr && ((k == k0) || (c.t == 0))) {
                // a new (s, h): if its last tile is ours, fetch the appended token's rows now
                const int32_t seg_last = sm.base[c.s] + c.h * c.nt + c.nt - 1;
                new_slot = -1;
                if (seg_last < g1) {
                    new_slot = p.slots[c.s];
                    const size_t rw = ((size_t)c.s * H + c.h) * W;
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        const int wi = lane + 32 * i;
                        if (wi < 2 * W) nw[i] = wi < W ? p.k_new[rw + wi] : p.v_new[rw + wi - W];
                    }
                }
            }
            if (k >= NS) {
                const uint32_t parity = ((k / NS) - 1) & 1;
                wait_phase(sm, empty0 + 8 * stage, parity, p.status);
            }
            if (new_slot >= 0 && c.t == c.nt - 1) {
                // the tile holding the new token: store its rows (quantised for an
                // E4M3 cache), then order the generic-proxy stores before the
                // tile's TMA (async-proxy) read
                if (new_slot < (int64_t)p.N * p.B) {
                    const int64_t blk = new_slot >> lgB, off = new_slot & (p.B - 1);
                    const int64_t srow = (blk * H + c.h) * p.B + off;   // scales: [N][H][B] in either layout
                    const int64_t row = p.layout == PKV_LAYOUT_NHD ? (blk * p.B + off) * H + c.h : srow;
                    if constexpr (Q8) {
                        // one lane per 8 elements; the W lanes of a row reduce its amax
                        const int wi = lane;                   // NW == 1 for D <= 128
                        float mm = q8::amax_word(nw[0]);
#pragma unroll
                        for (int o = 1; o < W; o <<= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
                        const float scale = q8::row_scale(mm);
                        if (wi < 2 * W) {
                            const uint2 codes = q8::quantize_word(nw[0], scale);
                            unsigned char *base = wi < W ? p.k_layer : p.v_layer;
                            reinterpret_cast<uint2 *>(base + row * D)[wi % W] = codes;
                            if (wi % W == 0) (wi < W ? p.k_scale : p.v_scale)[srow] = scale;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < NW; ++i) {
                            const int wi = lane + 32 * i;
                            if (wi < 2 * W) {
                                unsigned char *base = wi < W ? p.k_layer : p.v_layer;
                                reinterpret_cast<uint4 *>(base + row * D * 2)[wi % W] = nw[i];
                            }
                        }
                    }
                    ptx::fence_proxy_async_global();
                } else if (lane == 0) {
                    atomicOr(p.status, PKV_DEV_BAD_SLOT);
                }
                new_slot = -1;
                __syncwarp();
            }
            const bool first = (k == 0) || (c.t == 0);
            issue_kv(c, stage, first);
            if (first) issue_q(c, stage);
            __syncwarp();
            advance(c, sm, S, H);
        }
        // Dependents may launch once every load is issued, not at the start: a small
        // successor (the next layer's append) launched at the start sits resident next
        // to these CTAs for the whole launch, and its waiting warps cost the
        // issue-bound E4M3 consumers about 4 us per layer (7B batch 32). In the early
        // mode the trigger above, after the first stages, stays, unless this launch
        // follows an append (last_pending), whose successor is the next layer's append.
        if (!early || p.last_pending) ptx::launch_dependents();
        return;
    }

    // ================= consumer warps
    const int grp = warp * 4 + (lane >> 3);  // 0..15
    const int j = lane & 7;
    // q of the current (s, h): this lane's 8 x NCH elements as fp16 halves
    uint16_t qlo[NCH * 4], qhi[NCH * 4];
    float2 o[NCH * 4];                        // unnormalised output, this lane's elements
    // kMma: q as the B operand (lanes 0-3: 16 fp16 pairs each, zero elsewhere) and the
    // unnormalised output, dims 16 u + 2 (lane / 4) + {0, 1} in lanes 4 (lane / 4)
    uint32_t qa[16];
    float oacc[16];
    float m = -INFINITY, l = 0.f;             // running max (log2 units) and sum
    Cursor c = locate(sm, S, H, g0);

    for (int32_t k = 0; k < n; ++k) {
        const int32_t stage = k % NS;
        const uint32_t kb = stage0 + stage * SB;             // K tile (shared address)
        const uint32_t vb = kb + St::kTileBytes;             // V tile
        wait_phase(sm, full0 + 8 * stage, (k / NS) & 1, p.status);
        const bool first = (k == 0) || (c.t == 0);
        const int32_t ntok = min(kTile, sm.len[c.s] - c.t * kTile);
        if constexpr (kMma) {
            // ---- E4M3, head_dim 128: q.K and p.V on the warp-level tensor cores (m16n8k16,
            // fp16 operands, fp32 sums). Warp w takes tokens [16 w, 16 w + 16) of the tile;
            // the query is column 0 of the products' 8 columns, the others are zero padding.
            const int g = lane >> 2, c4 = lane & 3;
            const int tok0 = warp * 16;
            const bool full = ntok == kTile;
            if (first) {
                // q dims [32 c4, 32 c4 + 32) as the B column of lanes 0-3 (zero elsewhere);
                // lanes with c4 >= 2 read the 16-byte groups of each pair in swapped order, so
                // that the four lanes' loads fall in distinct banks
                const int sw = c4 >> 1;
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = ptx::lds128(kb + St::kQ + c4 * 64 + (i ^ sw) * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 w = sw ? v[i ^ 1] : v[i];
                    qa[4 * i + 0] = g == 0 ? w.x : 0u;
                    qa[4 * i + 1] = g == 0 ? w.y : 0u;
                    qa[4 * i + 2] = g == 0 ? w.z : 0u;
                    qa[4 * i + 3] = g == 0 ? w.w : 0u;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) oacc[i] = 0.f;
                m = -INFINITY;
                l = 0.f;
                if (sm.beg[c.s] > 0) stage_prefix_pieces<D>(p, sm, c.s, c.h, tid);
            }
            // S^T = K q^T: A rows g, g + 8 = tokens tok0 + g, tok0 + g + 8 (bytes [32 c4, 32 c4 + 32)
            // of each, 128-byte swizzled: (token & 7) == g); k step st pairs their word st (dims
            // 32 c4 + 4 st .. + 3) with q's words 2 st, 2 st + 1 (the same dims), a consistent
            // order of the dot product's terms
            uint32_t kw[16];
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const uint32_t row = kb + (tok0 + 8 * r2 + g) * 128;
                const uint4 w0 = ptx::lds128(row + (((2 * c4) ^ g) << 4));
                const uint4 w1 = ptx::lds128(row + (((2 * c4 + 1) ^ g) << 4));
                kw[8 * r2 + 0] = w0.x; kw[8 * r2 + 1] = w0.y; kw[8 * r2 + 2] = w0.z; kw[8 * r2 + 3] = w0.w;
                kw[8 * r2 + 4] = w1.x; kw[8 * r2 + 5] = w1.y; kw[8 * r2 + 6] = w1.z; kw[8 * r2 + 7] = w1.w;
            }
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
            for (int st = 0; st < 8; st += 2) {       // two accumulation chains
                uint32_t a0, a1, a2, a3, e0, e1, e2, e3;
                q8::e4m3x4_to_half2x2(kw[st], a0, a2);
                q8::e4m3x4_to_half2x2(kw[8 + st], a1, a3);
                q8::e4m3x4_to_half2x2(kw[st + 1], e0, e2);
                q8::e4m3x4_to_half2x2(kw[9 + st], e1, e3);
                ptx::mma_16816(s0, s1, s2, s3, a0, a1, a2, a3, qa[2 * st], qa[2 * st + 1], s0, s1, s2, s3);
                ptx::mma_16816(t0, t1, t2, t3, e0, e1, e2, e3, qa[2 * st + 2], qa[2 * st + 3], t0, t1, t2, t3);
            }
            // lanes 4 g hold the scores of tokens tok0 + g (s0 + t0) and tok0 + g + 8 (s2 + t2)
            const int ta = tok0 + g, tb = ta + 8;
            const bool oka = full || ta < ntok, okb = full || tb < ntok;
            const float ksa = ptx::ldsf(kb + St::kScales + ta * 4), ksb = ptx::ldsf(kb + St::kScales + tb * 4);
            const float vsa = ptx::ldsf(kb + St::kScales + (kTile + ta) * 4);
            const float vsb = ptx::ldsf(kb + St::kScales + (kTile + tb) * 4);
            const float xa = oka ? (s0 + t0) * ksa * p.scale_log2 : -INFINITY;
            const float xb = okb ? (s2 + t2) * ksb * p.scale_log2 : -INFINITY;
            // the reference covers x + log2(V row scale): weight x scale <= 1 fits fp16
            float mx = fmaxf(oka ? xa + ptx::lg2(fmaxf(vsa, 0x1p-100f)) : -INFINITY,
                             okb ? xb + ptx::lg2(fmaxf(vsb, 0x1p-100f)) : -INFINITY);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            mx = __shfl_sync(0xffffffffu, mx, 0);    // lane 0's (= every 4 g lane's): warp-uniform
            if (mx > m) {
                const float alpha = ptx::ex2(m - mx);
#pragma unroll
                for (int i = 0; i < 16; ++i) oacc[i] *= alpha;
                l *= alpha;
                m = mx;
            }
            // weights; a token past the context weighs 0 whatever its stale scale holds
            const float pa = oka ? ptx::ex2(xa - m) : 0.f, pb = okb ? ptx::ex2(xb - m) : 0.f;
            l += pa + pb;
            const uint32_t pk = ptx::pack_half2(oka ? pa * vsa : 0.f, okb ? pb * vsb : 0.f);
            // B = (weight x V scale)^T, column 0 = lanes 0-3: tokens 2 c4, 2 c4 + 1 (b0) and
            // 2 c4 + 8, 2 c4 + 9 (b1), gathered from lanes 8 c4 and 8 c4 + 4
            const uint32_t xw = __shfl_sync(0xffffffffu, pk, 8 * c4);
            const uint32_t yw = __shfl_sync(0xffffffffu, pk, 8 * c4 + 4);
            const uint32_t pb0 = g == 0 ? ptx::prmt(xw, yw, 0x5410u) : 0u;
            const uint32_t pb1 = g == 0 ? ptx::prmt(xw, yw, 0x7632u) : 0u;
            // O^T += V^T P^T over 8 chunks of 16 dims. ldmatrix (transposed) gives lane (g, c4)
            // the codes of tokens 2 c4, 2 c4 + 1 at dims 2 g, 2 g + 1 of a chunk; the chunk's
            // A rows are g <-> dim 16 u + 2 g and g + 8 <-> dim 16 u + 2 g + 1
            const int mi = lane >> 3;                  // the matrix whose row this lane addresses
            const uint32_t vrow = vb + (tok0 + (mi & 1) * 8 + (lane & 7)) * 128;
            if (!full && tok0 + 16 > ntok) {
                // rows past the context may hold any codes (NaN ones included) and a zero
                // weight does not cancel a NaN in the product: zero this warp's such V rows
                const int r0 = max(ntok, tok0);
                for (int i = lane; i < (tok0 + 16 - r0) * 8; i += 32)
                    ptx::sts128(vb + (r0 + (i >> 3)) * 128 + (i & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
                ptx::fence_proxy_async_shared();       // before the stage's next TMA fill
                __syncwarp();
            }
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                uint32_t r[4];
                ptx::ldmatrix_x4_trans(vrow + (((2 * hh + (mi >> 1)) ^ (lane & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                    const int u = 2 * hh + uu;
                    // bytes [t dim, t+1 dim, t dim+1, t+1 dim+1] of tokens 0-7 and 8-15 ->
                    // [t dim, t+1 dim] (A rows g) and [t dim+1, t+1 dim+1] (A rows g + 8)
                    uint32_t a0, a1, a2, a3;
                    q8::e4m3x4_to_half2x2(ptx::prmt(r[2 * uu], 0u, 0x3120u), a0, a1);
                    q8::e4m3x4_to_half2x2(ptx::prmt(r[2 * uu + 1], 0u, 0x3120u), a2, a3);
                    float d0, d1, d2, d3;
                    ptx::mma_16816(d0, d1, d2, d3, a0, a1, a2, a3, pb0, pb1, 0.f, 0.f, 0.f, 0.f);
                    oacc[2 * u] += d0;
                    oacc[2 * u + 1] += d2;
                }
            }
        } else {
            if (first) {
    #pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const uint4 raw = ptx::lds128(kb + St::kQ + chunk_elem<D, Q8>(j, ch) * 2);
                    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
    #pragma unroll
                    for (int e = 0; e < 4; ++e) ptx::split_half2(wv[e], qlo[ch * 4 + e], qhi[ch * 4 + e]);
                }
    #pragma unroll
                for (int e = 0; e < NCH * 4; ++e) o[e] = make_float2(0.f, 0.f);
                m = -INFINITY;
                l = 0.f;
                if (sm.beg[c.s] > 0) stage_prefix_pieces<D>(p, sm, c.s, c.h, tid);
            }
            // this group's rows of the tile: grp, grp + kGroups, ...; kr/vr hold each
            // chunk's 8 elements as four fp16 pairs (fp16 cache), kcw/vcw the row's E4M3
            // codes, four to a word, converted where they are used (fewer live registers)
            const bool full = ntok == kTile;
            bool vld[kTokPerGroup];
            uint32_t kr[kTokPerGroup][NCH][4], vr[kTokPerGroup][NCH][4];
            uint32_t kcw[kTokPerGroup][NCH * 2], vcw[kTokPerGroup][NCH * 2];
            float ksc[kTokPerGroup], vsc[kTokPerGroup];
    #pragma unroll
            for (int u = 0; u < kTokPerGroup; ++u) {
                const int row = grp + kGroups * u;
                vld[u] = full || row < ntok;
                if constexpr (Q8) {
                    if constexpr (NCH == 2) {
                        const uint4 a = ptx::lds128(kb + row * St::kRow + j * 16);
                        const uint4 b = ptx::lds128(vb + row * St::kRow + j * 16);
                        kcw[u][0] = a.x; kcw[u][1] = a.y; kcw[u][2] = a.z; kcw[u][3] = a.w;
                        vcw[u][0] = b.x; vcw[u][1] = b.y; vcw[u][2] = b.z; vcw[u][3] = b.w;
                    } else {
                        const uint2 a = ptx::lds64(kb + row * St::kRow + j * 8);
                        const uint2 b = ptx::lds64(vb + row * St::kRow + j * 8);
                        kcw[u][0] = a.x; kcw[u][1] = a.y;
                        vcw[u][0] = b.x; vcw[u][1] = b.y;
                    }
                    ksc[u] = ptx::ldsf(kb + St::kScales + row * 4);
                    vsc[u] = ptx::ldsf(kb + St::kScales + kTile * 4 + row * 4);
                } else {
    #pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        const uint4 a = ptx::lds128(kb + row * St::kRow + chunk_elem<D, Q8>(j, ch) * 2);
                        const uint4 b = ptx::lds128(vb + row * St::kRow + chunk_elem<D, Q8>(j, ch) * 2);
                        kr[u][ch][0] = a.x; kr[u][ch][1] = a.y; kr[u][ch][2] = a.z; kr[u][ch][3] = a.w;
                        vr[u][ch][0] = b.x; vr[u][ch][1] = b.y; vr[u][ch][2] = b.z; vr[u][ch][3] = b.w;
                    }
                    ksc[u] = 1.f;
                    vsc[u] = 1.f;
                }
            }
            float x[kTokPerGroup];
            float mx = -INFINITY;
    #pragma unroll
            for (int u = 0; u < kTokPerGroup; ++u) {
                float a0 = 0.f, a1 = 0.f;
    #pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint16_t klo, khi;
                        ptx::split_half2(pair_of<Q8, NCH>(kcw[u], kr[u], ch, e), klo, khi);
                        a0 = ptx::fma_f16_f32(qlo[ch * 4 + e], klo, a0);
                        a1 = ptx::fma_f16_f32(qhi[ch * 4 + e], khi, a1);
                    }
                }
                float dot = a0 + a1;
                dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                if constexpr (Q8) dot *= ksc[u];
                x[u] = vld[u] ? dot * p.scale_log2 : -INFINITY;
                // E4M3: the reference max covers x + log2(V row scale), so that every weight
                // 2^(x - m) * scale is at most 1 and fits fp16 for the p.V products
                // (a scale of 0, which the quantiser never writes, counts as 2^-100)
                if constexpr (Q8) mx = fmaxf(mx, vld[u] ? x[u] + ptx::lg2(fmaxf(vsc[u], 0x1p-100f)) : -INFINITY);
                else mx = fmaxf(mx, x[u]);
            }
            if (mx > m) {                          // new running max: rescale (group-uniform branch)
                const float alpha = ptx::ex2(m - mx);
    #pragma unroll
                for (int e = 0; e < NCH * 4; ++e) o[e] = make_float2(o[e].x * alpha, o[e].y * alpha);
                l *= alpha;
                m = mx;
            }
            // rows past the context may hold any bits (NaN included): weight 0 and V skipped
            float pw[kTokPerGroup];
    #pragma unroll
            for (int u = 0; u < kTokPerGroup; ++u) {
                pw[u] = vld[u] ? ptx::ex2(x[u] - m) : 0.f;
                l += pw[u];
            }
            if constexpr (Q8) {
                // o += (weight x V row scale) in fp16 x the row's codes as fp16 (exact), one
                // mixed-precision FMA per element with fp32 accumulation
                uint16_t wh[kTokPerGroup];
    #pragma unroll
                for (int u = 0; u < kTokPerGroup; ++u) wh[u] = __half_as_ushort(__float2half_rn(pw[u] * vsc[u]));
    #pragma unroll
                for (int u = 0; u < kTokPerGroup; ++u) {
                    if (!full && !vld[u]) continue;
    #pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
    #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint16_t vlo, vhi;
                            ptx::split_half2(pair_of<Q8, NCH>(vcw[u], vr[u], ch, e), vlo, vhi);
                            o[ch * 4 + e].x = ptx::fma_f16_f32(wh[u], vlo, o[ch * 4 + e].x);
                            o[ch * 4 + e].y = ptx::fma_f16_f32(wh[u], vhi, o[ch * 4 + e].y);
                        }
                }
            } else if (full) {
    #pragma unroll
                for (int u = 0; u < kTokPerGroup; ++u)
    #pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
    #pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[ch * 4 + e] = ptx::ffma2(make_float2(pw[u], pw[u]), ptx::half2_to_float2(pair_of<Q8, NCH>(vcw[u], vr[u], ch, e)),
                                                       o[ch * 4 + e]);
            } else {
    #pragma unroll
                for (int u = 0; u < kTokPerGroup; ++u) {
                    if (!vld[u]) continue;
    #pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
    #pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[ch * 4 + e] = ptx::ffma2(make_float2(pw[u], pw[u]), ptx::half2_to_float2(pair_of<Q8, NCH>(vcw[u], vr[u], ch, e)),
                                                       o[ch * 4 + e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty0 + 8 * stage);

        const bool last = (k == n - 1) || (c.t == c.nt - 1);
        if (last) {
            if constexpr (kMma) {
                // ---- this warp's state to shared memory: l summed over lanes 4 g, output
                // dims 16 u + 2 g, + 1 from lanes 4 g
                float lw = l;                       // lanes 4 g hold the sums of their tokens
                lw += __shfl_xor_sync(0xffffffffu, lw, 4);
                lw += __shfl_xor_sync(0xffffffffu, lw, 8);
                lw += __shfl_xor_sync(0xffffffffu, lw, 16);
                if ((lane & 3) == 0) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float2 *>(sm.red_o + warp * D + 16 * u + 2 * (lane >> 2)) =
                            make_float2(oacc[2 * u], oacc[2 * u + 1]);
                }
                if (lane == 0) {
                    sm.red_m[warp] = m;
                    sm.red_l[warp] = lw;
                }
            } else {
                // ---- merge the group states of this (s, h): the 4 groups of a warp
                // by xor-shuffles, then the warps through shared memory
                float mw = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
                const float sc = mw == -INFINITY ? 0.f : ptx::ex2(m - mw);   // a warp with no row at all: 0
                float lw = l * sc;
                lw += __shfl_xor_sync(0xffffffffu, lw, 8);
                lw += __shfl_xor_sync(0xffffffffu, lw, 16);
    #pragma unroll
                for (int e = 0; e < NCH * 4; ++e) {
                    float2 v = make_float2(o[e].x * sc, o[e].y * sc);
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, 8);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, 8);
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, 16);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, 16);
                    o[e] = v;
                }
                if (lane < 8) {
    #pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        float4 *dst = reinterpret_cast<float4 *>(sm.red_o + warp * D + chunk_elem<D, Q8>(j, ch));
                        dst[0] = make_float4(o[ch * 4 + 0].x, o[ch * 4 + 0].y, o[ch * 4 + 1].x, o[ch * 4 + 1].y);
                        dst[1] = make_float4(o[ch * 4 + 2].x, o[ch * 4 + 2].y, o[ch * 4 + 3].x, o[ch * 4 + 3].y);
                    }
                    if (lane == 0) {
                        sm.red_m[warp] = mw;
                        sm.red_l[warp] = lw;
                    }
                }
            }
            if (sm.beg[c.s] > 0) ptx::cp_async_wait_all();   // this thread's staged pieces (the barrier shares them)
            ptx::named_barrier(1, kConsumerThreads);
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < kConsumerWarps; ++i) M = fmaxf(M, sm.red_m[i]);
            float w[kConsumerWarps];
            float L = 0.f;
#pragma unroll
            for (int i = 0; i < kConsumerWarps; ++i) {
                w[i] = ptx::ex2(sm.red_m[i] - M);
                L = fmaf(w[i], sm.red_l[i], L);
            }
            constexpr int DPT = (D + kConsumerThreads - 1) / kConsumerThreads;  // dims per thread
            float O[DPT];
#pragma unroll
            for (int r = 0; r < DPT; ++r) {
                const int d = tid + r * kConsumerThreads;
                float acc = 0.f;
                if (d < D) {
#pragma unroll
                    for (int i = 0; i < kConsumerWarps; ++i) acc = fmaf(w[i], sm.red_o[i * D + d], acc);
                }
                O[r] = acc;
            }
            const int32_t seg_lo = sm.base[c.s] + c.h * c.nt;   // (s, h) tiles: [seg_lo, seg_lo + nt)
            const int32_t seg_hi = seg_lo + c.nt - 1;
            const int32_t ca = cta_of(total, grid, seg_lo);    // the CTAs covering the (s, h)
            const int32_t cb = cta_of(total, grid, seg_hi);
            __half *dst_out = p.out + ((size_t)c.s * H + c.h) * D;
            if (ca == cb) {
                if (sm.beg[c.s] > 0) merge_prefix<D, DPT, true>(p, sm.pre, c.s, c.h, tid, M, L, O);
                const float inv = 1.f / L;
#pragma unroll
                for (int r = 0; r < DPT; ++r) {
                    const int d = tid + r * kConsumerThreads;
                    if (d < D) dst_out[d] = __float2half_rn(O[r] * inv);
                }
            } else {
                const int slot = seg_lo <= g0 ? 0 : 1;  // 0: the CTA's first (s, h); 1: its last
                float *piece = p.pieces + ((size_t)cta * 2 + slot) * piece_stride(D);
#pragma unroll
                for (int r = 0; r < DPT; ++r) {
                    const int d = tid + r * kConsumerThreads;
                    if (d < D) piece[d] = O[r];
                }
                if (tid == 0) {
                    piece[D] = M;
                    piece[D + 1] = L;
                }
                // piece stores -> barrier -> one acquire-release counter bump: it
                // publishes this CTA's piece and, for the last arriver, makes
                // every other piece visible (the barrier after it passes that on)
                ptx::named_barrier(1, kConsumerThreads);
                if (tid == 0) {
#if PKV_ATTN_ACQREL
                    const int32_t prev = ptx::atom_add_acq_rel_gpu(p.counters + (size_t)c.s * H + c.h, 1);
#else
                    __threadfence();
                    const int32_t prev = atomicAdd(p.counters + (size_t)c.s * H + c.h, 1);
                    __threadfence();
#endif
                    sm.flags[1] = (prev == cb - ca) ? 1 : 0;
                }
                ptx::named_barrier(1, kConsumerThreads);
                if (sm.flags[1]) {
                    const int32_t start_a = range_start(total, grid, ca);
                    auto piece_of = [&](int32_t cc) {
                        const int sl = (cc > ca || start_a == seg_lo) ? 0 : 1;
                        return p.pieces + ((size_t)cc * 2 + sl) * piece_stride(D);
                    };
                    float Mg = -INFINITY;
                    float Lg = 0.f;
                    float Og[DPT];
#pragma unroll
                    for (int r = 0; r < DPT; ++r) Og[r] = 0.f;
                    constexpr int kFew = 4;                  // pieces merged with one round of loads
                    // (fp16 caches: on an E4M3 cache the unrolled merge measured 2 % slower)
                    if (!Q8 && cb - ca < kFew) {
                        float cm[kFew], cl[kFew], co[kFew][DPT];
#pragma unroll
                        for (int u = 0; u < kFew; ++u) {
                            const bool in = u <= cb - ca;
                            const float *pc = piece_of(ca + (in ? u : 0));
                            cm[u] = in ? __ldcg(pc + D) : -INFINITY;
                            cl[u] = in ? __ldcg(pc + D + 1) : 0.f;
#pragma unroll
                            for (int r = 0; r < DPT; ++r) {
                                const int d = tid + r * kConsumerThreads;
                                co[u][r] = (in && d < D) ? __ldcg(pc + d) : 0.f;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kFew; ++u) Mg = fmaxf(Mg, cm[u]);
#pragma unroll
                        for (int u = 0; u < kFew; ++u) {
                            if (u > cb - ca) break;
                            const float wc = ptx::ex2(cm[u] - Mg);
                            Lg = fmaf(wc, cl[u], Lg);
#pragma unroll
                            for (int r = 0; r < DPT; ++r) Og[r] = fmaf(wc, co[u][r], Og[r]);
                        }
                    } else {
                        for (int32_t cc = ca; cc <= cb; ++cc) Mg = fmaxf(Mg, __ldcg(piece_of(cc) + D));
                        for (int32_t cc = ca; cc <= cb; ++cc) {
                            const float *pc = piece_of(cc);
                            const float wc = ptx::ex2(__ldcg(pc + D) - Mg);
                            Lg = fmaf(wc, __ldcg(pc + D + 1), Lg);
#pragma unroll
                            for (int r = 0; r < DPT; ++r) {
                                const int d = tid + r * kConsumerThreads;
                                if (d < D) Og[r] = fmaf(wc, __ldcg(pc + d), Og[r]);
                            }
                        }
                    }
                    if (sm.beg[c.s] > 0) merge_prefix<D, DPT, true>(p, sm.pre, c.s, c.h, tid, Mg, Lg, Og);
                    const float inv = 1.f / Lg;
#pragma unroll
                    for (int r = 0; r < DPT; ++r) {
                        const int d = tid + r * kConsumerThreads;
                        if (d < D) dst_out[d] = __float2half_rn(Og[r] * inv);
                    }
                    if (tid == 0) p.counters[(size_t)c.s * H + c.h] = 0;
                }
            }
            ptx::named_barrier(1, kConsumerThreads);
        }
        advance(c, sm, S, H);
    }
}

// ------------------------------------------------------------------ host side

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

struct DeviceInfo {
    int num_sms = 0;
    int ctas_per_sm[6] = {0, 0, 0, 0, 0, 0};  // per (head_dim 64/128/256, fp16/E4M3), at the smem size last queried
    size_t smem_for[6] = {0, 0, 0, 0, 0, 0};
    size_t smem_attr[6] = {0, 0, 0, 0, 0, 0};  // the kernel's dynamic shared memory limit as set (only grows)
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int variant_index(int D, bool q8) { return (D == 64 ? 0 : (D == 128 ? 1 : 2)) * 2 + (q8 ? 1 : 0); }

bool variant_built(int D, bool q8) { return supported_head_dim(D) && (!q8 || D <= 128); }

const void *kernel_for(int D, bool q8) {
    if (q8) return D == 64 ? reinterpret_cast<const void *>(&decode_attention_kernel<64, true>)
                           : reinterpret_cast<const void *>(&decode_attention_kernel<128, true>);
    switch (D) {
        case 64: return reinterpret_cast<const void *>(&decode_attention_kernel<64, false>);
        case 128: return reinterpret_cast<const void *>(&decode_attention_kernel<128, false>);
        default: return reinterpret_cast<const void *>(&decode_attention_kernel<256, false>);
    }
}

size_t smem_bytes(int D, bool q8, int S) {
    if (q8) return D == 64 ? smem_bytes_t<64, true>(S) : smem_bytes_t<128, true>(S);
    switch (D) {
        case 64: return smem_bytes_t<64, false>(S);
        case 128: return smem_bytes_t<128, false>(S);
        default: return smem_bytes_t<256, false>(S);
    }
}

// SMs and resident CTAs per SM for head_dim D (fp16 or E4M3 cache) with S sequences on `dev`.
pkv_status launch_shape(int dev, int D, bool q8, int S, int *grid, int *per_sm, int *sms, size_t *smem) {
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_CUDA, "device index %d", dev);
    const size_t bytes = smem_bytes(D, q8, S);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &di = g_dev[dev];
    if (di.num_sms == 0) {
        if (cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(PKV_ERR_CUDA, "cudaDeviceGetAttribute failed");
    }
    const int vi = variant_index(D, q8);
    if (di.smem_for[vi] != bytes) {
        // the limit only grows, so a launch sized for more sequences on another host thread
        // never meets a limit lowered after its own query
        if (bytes > di.smem_attr[vi]) {
            cudaError_t e = cudaFuncSetAttribute(kernel_for(D, q8), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)std::max<size_t>(bytes, 48 * 1024));
            if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            di.smem_attr[vi] = bytes;
        }
        int occ = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel_for(D, q8), kThreads, bytes);
        if (e != cudaSuccess || occ < 1)
            return fail(PKV_ERR_CUDA, "occupancy query failed (%s, %d)", cudaGetErrorString(e), occ);
        di.ctas_per_sm[vi] = std::min(occ, kMaxCtasPerSm);
        di.smem_for[vi] = bytes;
    }
    *per_sm = di.ctas_per_sm[vi];
    *sms = di.num_sms;
    *grid = di.num_sms * di.ctas_per_sm[vi];
    *smem = bytes;
    return PKV_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace layout: [status][pieces: two per CTA][last-arriver counters: one per (s, h)].
// The counters must be zero when a launch starts (each launch leaves those it used zero),
// so their place may not move between calls that share a workspace: a caller's workspace
// puts them after room for the pieces of the largest grid at the largest head_dim, so the
// same workspace serves calls with any num_seqs, head_dim and cache type it was sized for.
// The library's static scratch, whose counters are cleared on every call, packs the
// pieces of the launch's own grid instead (compact).
size_t pieces_bytes(int D, int grid) { return (size_t)grid * 2 * piece_stride(D) * sizeof(float); }

size_t counters_offset(bool compact, int D, int grid, int num_sms) {
    return kStatusBytes + round256(compact ? pieces_bytes(D, grid) : pieces_bytes(256, num_sms * kMaxCtasPerSm));
}

// Bytes of a caller's workspace for S sequences of H heads on a device with num_sms SMs.
size_t workspace_bytes_for(int S, int H, int num_sms) {
    return counters_offset(false, 0, 0, num_sms) + (size_t)S * H * sizeof(int32_t);
}

// swizzle128: the tile lands 128-byte swizzled (E4M3 head_dim 128: 128-byte rows).
pkv_status encode_map(CUtensorMap *map, const void *base, int N, int B, int H, int D, int layout, bool q8) {
    const bool swizzle128 = q8 && D == 128;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t elem = q8 ? 1 : 2;
    cuuint64_t dims[2], strides[1];
    if (layout == PKV_LAYOUT_NHD) {
        dims[0] = (cuuint64_t)H * D;
        dims[1] = (cuuint64_t)N * B;
        strides[0] = (cuuint64_t)H * D * elem;
    } else {
        dims[0] = (cuuint64_t)D;
        dims[1] = (cuuint64_t)N * H * B;
        strides[0] = (cuuint64_t)D * elem;
    }
    const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)std::min(B, kTile)};
    const cuuint32_t estr[2] = {1, 1};
    // L2 promotion no wider than what a box row reads contiguously: in NHD one head's row
    // (D elements) sits between the other heads' rows, and a wider promotion would fetch
    // a neighbour's piece with every row (an E4M3 row at head_dim 128 is 128 bytes)
    CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    if (layout == PKV_LAYOUT_NHD) {
        const cuuint64_t piece = (cuuint64_t)D * elem;
        promo = piece >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                             : (piece >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B);
    }
    CUresult r = fn(map, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    promo,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

pkv_status pkv_check_wait_limit(uint32_t *status, void *stream) {
    if (!status) return fail(PKV_ERR_INVALID_ARG, "status is NULL");
    wait_limit_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "wait-limit probe launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim) {
    if (num_seqs < 0 || num_seqs > kMaxSeqs || num_heads < 1 || !supported_head_dim(head_dim)) {
        fail(PKV_ERR_INVALID_ARG, "bad sizes for the workspace");
        return 0;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        fail(PKV_ERR_CUDA, "no CUDA device");
        return 0;
    }
    return workspace_bytes_for(num_seqs, num_heads, sms);
}

pkv_status pkv_decode_launch_info(int32_t num_seqs, int32_t head_dim, int32_t kv_dtype, int32_t *grid_ctas,
                                  int32_t *ctas_per_sm, int32_t *num_sms) {
    if (!supported_head_dim(head_dim) || num_seqs < 0 || num_seqs > kMaxSeqs)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes");
    if (kv_dtype != PKV_KV_F16 && kv_dtype != PKV_KV_E4M3) return fail(PKV_ERR_INVALID_ARG, "bad kv_dtype");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(PKV_ERR_CUDA, "no CUDA device");
    int g = 0, per = 0, sms = 0;
    size_t smem = 0;
    pkv_status st = launch_shape(dev, head_dim, kv_dtype == PKV_KV_E4M3, num_seqs, &g, &per, &sms, &smem);
    if (st != PKV_OK) return st;
    if (grid_ctas) *grid_ctas = g;
    if (ctas_per_sm) *ctas_per_sm = per;
    if (num_sms) *num_sms = sms;
    return PKV_OK;
}

}  // extern "C"

namespace {

// Shared implementation of the attention entry points; k_new / v_new / slots
// non-null = fused append of one token per sequence (decode step).
pkv_status decode_attention_impl(const void *q, const void *k_cache, const void *v_cache, int32_t num_blocks,
                                 int32_t block_size, int32_t num_heads, int32_t head_dim, int32_t layout,
                                 const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                                 int32_t num_seqs, float scale, void *out, void *workspace, size_t workspace_bytes,
                                 void *stream, const void *k_new, const void *v_new, const int64_t *slots,
                                 uint32_t *status_override = nullptr, const float *k_scale = nullptr,
                                 const float *v_scale = nullptr, const int32_t *seq_begin = nullptr,
                                 const float *pieces = nullptr, int32_t splits = 0, uint32_t flags = 0,
                                 bool compact = false) {
    const bool q8 = k_scale != nullptr;
    if ((seq_begin == nullptr) != (pieces == nullptr))
        return fail(PKV_ERR_INVALID_ARG, "seq_begin and pieces go together (both NULL: no cascade)");
    if (seq_begin) {
        if (head_dim != 128)
            return fail(PKV_ERR_UNSUPPORTED, "the cascade is built for pools with head_dim 128");
        if (splits < 1 || splits > PKV_MAX_PREFIX_SPLITS)
            return fail(PKV_ERR_INVALID_ARG, "splits %d outside 1..%d", splits, PKV_MAX_PREFIX_SPLITS);
        if ((reinterpret_cast<uintptr_t>(seq_begin) & 3u) || !aligned16(pieces))
            return fail(PKV_ERR_INVALID_ARG, "seq_begin must be 4-byte and pieces 16-byte aligned");
    }
    if (num_seqs < 0 || num_seqs > kMaxSeqs)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d outside [0, %d]", num_seqs, kMaxSeqs);
    if (num_seqs == 0) return PKV_OK;
    if (!variant_built(head_dim, q8))
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d%s", head_dim, q8 ? " with an E4M3 cache" : "");
    if (q8 && (!v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
        return fail(PKV_ERR_INVALID_ARG, "an E4M3 cache needs 16-byte aligned scale pools");
    if (!supported_block_size(block_size)) return fail(PKV_ERR_UNSUPPORTED, "block_size %d", block_size);
    if (layout != PKV_LAYOUT_NHD && layout != PKV_LAYOUT_HND) return fail(PKV_ERR_INVALID_ARG, "layout %d", layout);
    if (num_heads < 1 || num_blocks < 1 || max_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "sizes must be >= 1");
    if ((int64_t)num_blocks * block_size * num_heads >= ((int64_t)1 << 31))
        return fail(PKV_ERR_INVALID_ARG, "num_blocks * block_size * num_heads must be < 2^31");
    const int64_t tiles_bound = (int64_t)num_seqs * num_heads * (((int64_t)max_blocks * block_size + kTile - 1) / kTile);
    if (tiles_bound >= ((int64_t)1 << 31) - 1)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs * num_heads * max_context / 32 must be < 2^31");
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "misaligned pointer (q, caches, out, workspace: 16 B; tables, lens: 4 B)");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(PKV_ERR_CUDA, "no CUDA device");
    int grid = 0, per = 0, sms = 0;
    size_t smem = 0;
    pkv_status st = launch_shape(dev, head_dim, q8, num_seqs, &grid, &per, &sms, &smem);
    if (st != PKV_OK) return st;
    const size_t counters_off = counters_offset(compact, head_dim, grid, sms);
    const size_t need = counters_off + (size_t)num_seqs * num_heads * sizeof(int32_t);
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", workspace_bytes, need);

    CUtensorMap kmap, vmap;
    st = encode_map(&kmap, k_cache, num_blocks, block_size, num_heads, head_dim, layout, q8);
    if (st != PKV_OK) return st;
    st = encode_map(&vmap, v_cache, num_blocks, block_size, num_heads, head_dim, layout, q8);
    if (st != PKV_OK) return st;

    Params prm;
    prm.q = static_cast<const __half *>(q);
    prm.out = static_cast<__half *>(out);
    prm.tables = block_tables;
    prm.lens = context_lens;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    prm.status = status_override ? status_override : reinterpret_cast<uint32_t *>(ws);
    prm.pieces = reinterpret_cast<float *>(ws + kStatusBytes);
    prm.counters = reinterpret_cast<int32_t *>(ws + counters_off);
    prm.S = num_seqs;
    prm.H = num_heads;
    prm.max_blocks = max_blocks;
    prm.B = block_size;
    prm.lgB = __builtin_ctz((unsigned)block_size);   // a supported block size is a power of two
    prm.N = num_blocks;
    prm.layout = layout;
    const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)head_dim);
    prm.scale_log2 = (float)(sc * 1.4426950408889634);  // log2(e)
    prm.k_new = static_cast<const uint4 *>(k_new);
    prm.v_new = static_cast<const uint4 *>(v_new);
    prm.slots = slots;
    prm.k_layer = static_cast<unsigned char *>(const_cast<void *>(k_cache));
    prm.v_layer = static_cast<unsigned char *>(const_cast<void *>(v_cache));
    prm.k_scale = const_cast<float *>(k_scale);
    prm.v_scale = const_cast<float *>(v_scale);
    prm.begin = seq_begin;
    prm.pre = pieces;
    prm.pre_splits = seq_begin ? splits : 0;
    prm.early = (flags & PKV_ATTN_INPUTS_EARLY) ? 1 : 0;
    prm.last_pending = (flags & PKV_ATTN_LAST_ROW_PENDING) ? 1 : 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (q8) {
        e = head_dim == 64 ? launch_pdl(decode_attention_kernel<64, true>, grid, kThreads, smem, s, kmap, vmap, prm)
                           : launch_pdl(decode_attention_kernel<128, true>, grid, kThreads, smem, s, kmap, vmap, prm);
    } else {
        switch (head_dim) {
            case 64: e = launch_pdl(decode_attention_kernel<64, false>, grid, kThreads, smem, s, kmap, vmap, prm); break;
            case 128:
                e = launch_pdl(decode_attention_kernel<128, false>, grid, kThreads, smem, s, kmap, vmap, prm);
                break;
            default:
                e = launch_pdl(decode_attention_kernel<256, false>, grid, kThreads, smem, s, kmap, vmap, prm);
                break;
        }
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "decode attention launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention(const void *q, const void *k_cache, const void *v_cache, int32_t num_blocks,
                                int32_t block_size, int32_t num_heads, int32_t head_dim, int32_t layout,
                                const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                                int32_t num_seqs, float scale, void *out, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return decode_attention_impl(q, k_cache, v_cache, num_blocks, block_size, num_heads, head_dim, layout,
                                 block_tables, max_blocks, context_lens, num_seqs, scale, out, workspace,
                                 workspace_bytes, stream, nullptr, nullptr, nullptr);
}

pkv_status pkv_decode_append_attention(const pkv_pool *pool, int32_t layer, const void *q, const void *k_new,
                                       const void *v_new, const int64_t *slot_mapping, const int32_t *block_tables,
                                       int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs,
                                       float scale, void *out, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (layer < 0 || layer >= d.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
        return fail(PKV_ERR_INVALID_ARG, "NULL k_new, v_new or slot_mapping");
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail(PKV_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned, slot_mapping 8-byte aligned");
    const PoolLayer pl = pool_layer(pool, layer);
    if (pool->desc.kv_dtype == PKV_KV_E4M3 && !pl.k_scale)
        return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    return decode_attention_impl(q, pl.k, pl.v, d.num_blocks, d.block_size, d.num_heads, d.head_dim, d.layout,
                                 block_tables, max_blocks, context_lens, num_seqs, scale, out, workspace,
                                 workspace_bytes, stream, k_new, v_new, slot_mapping, nullptr, pl.k_scale,
                                 pl.v_scale);
}

pkv_status pkv_decode_attention_ex(const pkv_pool *pool, int32_t layer, const void *q, const void *k_new,
                                   const void *v_new, const int64_t *slot_mapping, const int32_t *block_tables,
                                   int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs,
                                   const int32_t *seq_begin, const float *pieces, int32_t splits, float scale,
                                   void *out, void *workspace, size_t workspace_bytes, uint32_t flags,
                                   void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    if (flags & ~(uint32_t)(PKV_ATTN_INPUTS_EARLY | PKV_ATTN_LAST_ROW_PENDING))
        return fail(PKV_ERR_INVALID_ARG, "unknown flags %#x", flags);
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (layer < 0 || layer >= d.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    const bool append = k_new || v_new || slot_mapping;
    if (append && num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
        return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and slot_mapping go together (all NULL: no append)");
    if (append && (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)))
        return fail(PKV_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned, slot_mapping 8-byte aligned");
    const PoolLayer pl = pool_layer(pool, layer);
    if (pool->desc.kv_dtype == PKV_KV_E4M3 && !pl.k_scale)
        return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    return decode_attention_impl(q, pl.k, pl.v, d.num_blocks, d.block_size, d.num_heads, d.head_dim, d.layout,
                                 block_tables, max_blocks, context_lens, num_seqs, scale, out, workspace,
                                 workspace_bytes, stream, append ? k_new : nullptr, append ? v_new : nullptr,
                                 append ? slot_mapping : nullptr, nullptr, pl.k_scale, pl.v_scale, seq_begin, pieces,
                                 splits, flags);
}

pkv_status pkv_pool_decode_attention(const pkv_pool *pool, int32_t layer, const void *q, const int32_t *block_tables,
                                     int32_t max_blocks, const int32_t *context_lens, int32_t num_seqs, float scale,
                                     void *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (layer < 0 || layer >= d.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    const PoolLayer pl = pool_layer(pool, layer);
    if (pool->desc.kv_dtype == PKV_KV_E4M3 && !pl.k_scale)
        return fail(PKV_ERR_INVALID_ARG, "E4M3 pool without scale pools (pkv_pool_set_scales)");
    return decode_attention_impl(q, pl.k, pl.v, d.num_blocks, d.block_size, d.num_heads, d.head_dim, d.layout,
                                 block_tables, max_blocks, context_lens, num_seqs, scale, out, workspace,
                                 workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr, pl.k_scale, pl.v_scale);
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free entry point
//
// pkv_decode_attention_static runs the same kernel as pkv_decode_attention but
// takes its scratch (last-arriver counters and split pieces) from a fixed array
// compiled into the library instead of a caller-provided workspace. It exists
// for callers that cannot allocate device memory: a host framework that owns
// every device byte and offers a plugin no workspace hook, or a serving loop
// that forbids allocation once it is running (cudaMalloc may synchronise the
// device and stall every other stream). Such a caller still passes its own
// inputs and outputs; only the scratch moves into the library.

namespace {

constexpr size_t kStaticScratchBytes = (size_t)4 << 20;  // 4 MiB, held by every GPU that loads libpkv

// The scratch itself. In host code this name is only a host-side stand-in for
// the symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void *g_static_scratch_addr[kMaxDevices] = {};
std::mutex g_static_scratch_mu;

// Device address of the scratch on `dev` (the current device): looked up once
// per device, on the first call made with that device current.
pkv_status static_scratch(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_CUDA, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_static_scratch_mu);
    if (!g_static_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p)
            return fail(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
        g_static_scratch_addr[dev] = p;
    }
    *out = g_static_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention_static(const void *q, const void *k_cache, const void *v_cache, int32_t num_blocks,
                                       int32_t block_size, int32_t num_heads, int32_t head_dim, int32_t layout,
                                       const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                                       int32_t num_seqs, float scale, void *out, uint32_t *status, void *stream) {
    if (num_seqs < 0 || num_seqs > kMaxSeqs)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d outside [0, %d]", num_seqs, kMaxSeqs);
    if (num_seqs == 0) return PKV_OK;
    if (num_heads < 1 || !supported_head_dim(head_dim))
        return fail(PKV_ERR_INVALID_ARG, "bad num_heads or head_dim");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(PKV_ERR_CUDA, "no CUDA device");
    int grid = 0, per = 0, sms = 0;
    size_t smem = 0;
    pkv_status st0 = launch_shape(dev, head_dim, false, num_seqs, &grid, &per, &sms, &smem);
    if (st0 != PKV_OK) return st0;
    const size_t counters_off = counters_offset(true, head_dim, grid, sms);
    const size_t counters_len = (size_t)num_seqs * num_heads * sizeof(int32_t);
    const size_t need = counters_off + counters_len;
    if (need > kStaticScratchBytes)
        return fail(PKV_ERR_INVALID_ARG,
                    "%d sequences x %d heads (head_dim %d) need %zu bytes of scratch; the static scratch holds %zu",
                    num_seqs, num_heads, head_dim, need, kStaticScratchBytes);
    void *scratch = nullptr;
    pkv_status st = static_scratch(dev, &scratch);
    if (st != PKV_OK) return st;
    // The array keeps the previous call's contents: the status word and the
    // last-arriver counters must start at zero, so clear them on the stream.
    unsigned char *sc = static_cast<unsigned char *>(scratch);
    cudaError_t e = cudaMemsetAsync(sc, 0, kStatusBytes, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaMemsetAsync(sc + counters_off, 0, counters_len, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "clearing the static scratch: %s", cudaGetErrorString(e));
    return decode_attention_impl(q, k_cache, v_cache, num_blocks, block_size, num_heads, head_dim, layout,
                                 block_tables, max_blocks, context_lens, num_seqs, scale, out, scratch,
                                 kStaticScratchBytes, stream, nullptr, nullptr, nullptr, status, nullptr, nullptr,
                                 nullptr, nullptr, 0, 0, true);
}

}  // extern "C"
