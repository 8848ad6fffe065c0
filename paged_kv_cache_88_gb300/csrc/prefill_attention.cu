// Paged prefill attention on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// What it computes: a chunk of C_s new tokens of sequence s has been appended to
// the paged cache (its K/V are in the pool; context_lens[s] = T_s counts them).
// Query i of the chunk sits at position p = T_s - C_s + i and attends causally to
// every cached token t <= p, read through the block table:
//   out[i][h] = softmax_{t <= p}(scale * q[i][h] . K_t[h]) V_t[h].
// This is the multi-query (prefill) counterpart of the decode kernel
// (m.lqnn.cn/news/240480 §3.3 remaps positions through the page table inside the
// attention kernel, §4.3 runs the causal prefill through it; icman.com.cn/news/78786
// §2.4). Dense enough for tensor cores: a 128-query tile reuses every K/V tile
// 128 times.
//
// Design (one CTA per (sequence, head, two 128-query tiles A and B); 8 softmax
// warps, one MMA-issue warp and two TMA warps; fp16 HND cache, head_dim 128):
// * One TMA warp brings the two Q tiles and the K tiles, the other the V tiles, 128
//   keys at a time (one box per block of the table, two 64-element halves each)
//   into 128-byte-swizzled shared memory: two K slots and two V slots, each
//   refilled as soon as the MMAs that read it have finished. Both query tiles use
//   every K/V tile the CTA loads, halving the K/V traffic per FLOP.
// * One elected thread issues S_x = Q_x K^T (M = N = K = 128, fp16 -> fp32) into
//   tile x's tensor-memory S, and, once the softmax warps have written P_x (fp16,
//   over S_x), O_x += P_x V onto tile x's O in tensor memory (P read from tensor
//   memory as the A operand; V read MN-major straight from its [token][dim] rows).
//   Each tile has its own four softmax warps, so the two tiles' softmax run side by
//   side while the tensor cores alternate between the tiles' P V and next S.
// * Query row r of a tile is tensor-memory lane r and one softmax thread: both
//   64-column halves of its S row come in with one wait, and its max and sum never
//   leave the thread. The causal mask is applied on the diagonal tile only. The
//   softmax reference max only moves when a row's max exceeds it by more than 2^8,
//   and only then is O rescaled in place (tcgen05.ld / st). Rows past the
//   sequence's tokens in the last key tile are zeroed in V before P V (a zero
//   weight times non-finite garbage would not be zero).
// * Every wait is bounded (1 s, then PKV_DEV_TIMEOUT); before exiting, the CTA
//   waits (bounded) for its own copies and MMAs, and frees tensor memory on
//   every path.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace {

using namespace pkv;

constexpr int kQT = 128;             // queries per CTA (MMA M)
constexpr int kKT = 128;             // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kD = 128;              // head dim (MMA K of Q K^T, N of P V)
constexpr int kHalf = 64;            // 64 fp16 = one 128-byte swizzle row
constexpr int kSub = kQT * 128;      // bytes of one [128 rows x 64 elements] swizzled sub-tile (16 KB)
constexpr int kTileBytes = 2 * kSub; // a 128 x 128 fp16 tile as two sub-tiles
constexpr int kThreads = 352;        // warps 0-7 softmax, warp 8 MMA issue, warps 9-10 TMA loads (K, V)
constexpr int kGroupThreads = 128;   // softmax threads of one query tile (one per row)
constexpr int kTiles = 2;            // query tiles per CTA (A, B: 128 positions apart)
constexpr uint32_t kTmemCols = 512;  // S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512); P_X over S_X
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// shared memory: Q_A | Q_B | K0 | K1 | V0 | V1 (each a 32 KB tile, 1024-aligned), the
// prefix pass's row-max exchange, then barriers and flags
constexpr int kSmemTiles = 6 * kTileBytes;                 // Q_A | Q_B | K0 | K1 | V0 | V1
constexpr int kXchgBytes = 2 * 2 * kQT * 4;    // prefix pass: row-max exchange [slot][half][row]
constexpr int kSmemBytes = kSmemTiles + kXchgBytes + 256 /* barriers + flags */ + 1024 /* alignment slack */;

// barrier indices (two-slot rings use index + slot)
constexpr int kQFull = 0, kKFull = 1, kVFull = 3, kKFree = 5, kVFree = 7, kSFull = 9, kPReady = 11, kOFull = 13,
              kNumBars = 15;

struct PrefillParams {
    const int32_t *q_start;   // prefill: [S + 1] chunk rows of sequence s: q_start[s] .. q_start[s+1]-1
    const int32_t *tables;    // [S][max_blocks]
    const int32_t *lens;      // prefill: [S] context lengths including the chunk
    __half *out;              // prefill: [total_q][H][D]
    const pkv_prefix_group *groups;  // prefix pass: [gridDim.z]
    float *pieces;            // prefix pass: [S][H][PKV_MAX_PREFIX_SPLITS][D + 4]
    uint32_t *status;
    int32_t S, H, max_blocks, B, N, splits;
    float scale_log2;
    int32_t early;            // prefix pass: tables, groups and K/V read before the grid dependency
};

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    // tcgen05 shared-memory matrix descriptor: start, leading and stride byte
    // offsets (16-byte units), version 1, 128-byte swizzle
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, M = N = 128;
// b_mn = 1 reads B MN-major (its rows run along K).
__device__ __forceinline__ uint32_t umma_idesc(uint32_t b_mn) {
    return (1u << 4) | ((uint32_t)(kKT >> 3) << 17) | ((uint32_t)(kQT >> 4) << 24) | (b_mn << 16);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// The same MMA with A read from tensor memory (M rows on lanes, K along columns,
// two fp16 per 32-bit column).
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Loads of 64 (32) consecutive columns of this warp's 32 lanes, completed
// before any register is used (the wait sits in the same asm statement).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr) : "memory");
}
// Two 64-column loads in flight together, then one wait (both completed before any
// register is used).
__device__ __forceinline__ void tmem_ld64x2(uint32_t ta, uint32_t tb, uint32_t (&a)[64], uint32_t (&b)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(a[32]), "=r"(a[33]), "=r"(a[34]), "=r"(a[35]), "=r"(a[36]), "=r"(a[37]), "=r"(a[38]), "=r"(a[39]), "=r"(a[40]), "=r"(a[41]), "=r"(a[42]), "=r"(a[43]), "=r"(a[44]), "=r"(a[45]), "=r"(a[46]), "=r"(a[47]), "=r"(a[48]), "=r"(a[49]), "=r"(a[50]), "=r"(a[51]), "=r"(a[52]), "=r"(a[53]), "=r"(a[54]), "=r"(a[55]), "=r"(a[56]), "=r"(a[57]), "=r"(a[58]), "=r"(a[59]), "=r"(a[60]), "=r"(a[61]), "=r"(a[62]), "=r"(a[63]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31]), "=r"(b[32]), "=r"(b[33]), "=r"(b[34]), "=r"(b[35]), "=r"(b[36]), "=r"(b[37]), "=r"(b[38]), "=r"(b[39]), "=r"(b[40]), "=r"(b[41]), "=r"(b[42]), "=r"(b[43]), "=r"(b[44]), "=r"(b[45]), "=r"(b[46]), "=r"(b[47]), "=r"(b[48]), "=r"(b[49]), "=r"(b[50]), "=r"(b[51]), "=r"(b[52]), "=r"(b[53]), "=r"(b[54]), "=r"(b[55]), "=r"(b[56]), "=r"(b[57]), "=r"(b[58]), "=r"(b[59]), "=r"(b[60]), "=r"(b[61]), "=r"(b[62]), "=r"(b[63])
        : "r"(ta), "r"(tb) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 values rounded to fp16 (nearest even), packed low = lo, high = hi.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int32_t *timed_out,
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

// Before the CTA exits: wait (bounded, whatever the timeout flag says) for an
// asynchronous operation this CTA started, so no copy or MMA outlives it.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::global_timer_ns() - t0 > kWaitLimitNs) return;
}

// One kernel, two uses:
// * prefill (kPrefix = false): CTA (pair of 128-query tiles A and B, head,
//   sequence) of a chunk, causal over the sequence's cache, normalised fp16 output;
// * the cascade's prefix pass (kPrefix = true): CTA (key split, head, group), the
//   group members' decode queries as query tile A (row r = sequence first_seq + r;
//   no tile B), every key of the split's share of the shared prefix seen by every
//   row, unnormalised fp32 pieces (o, m, l) as output.
// Tiles A and B share every K/V tile the CTA loads (B, 128 positions later, sees at
// most one key tile more), which halves the K/V traffic per FLOP. Each has its own S
// and O in tensor memory; the softmax warps take A's tile j, then B's, and while they
// work on one, the tensor cores run the other's P V and next S. Pipeline over key
// tiles j (slot b = j & 1):
//   loaders: K_j -> K[b] once both S_{j-2} are done; V_j -> V[b] once both P_{j-2} V are
//   MMA    : S_A,0, S_B,0; per j: [P_A,j] O_A += P_A,j V_j, S_A,j+1; [P_B,j] likewise for B
//   softmax: per j: S_A -> P_A,j, then S_B -> P_B,j (fp16, over S in tensor memory)
// Every barrier is waited on at most one phase behind.
template <bool kPrefix>
__global__ void __launch_bounds__(kThreads, 1)
prefill_attention_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
    const uint32_t s0 = ptx::smem_addr(base);
    auto sQ = [s0](int x) { return s0 + (uint32_t)x * kTileBytes; };
    auto sK = [s0](int b) { return s0 + (uint32_t)(2 + b) * kTileBytes; };
    auto sV = [s0](int b) { return s0 + (uint32_t)(4 + b) * kTileBytes; };
    float *xchg = reinterpret_cast<float *>(base + kSmemTiles);          // prefix pass: [2][2][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kSmemTiles + kXchgBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int32_t *timed_out = reinterpret_cast<volatile int32_t *>(bars + kNumBars + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto BAR = [bar0](int i) { return bar0 + 8 * i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t h = blockIdx.y;
    const int32_t H = p.H, B = p.B;
    const int32_t cap = p.max_blocks * B;

    // The prefix pass may start early (p.early): groups, tables and the prefix's K/V --
    // which the preceding kernel does not write -- are read, and the K/V tiles' loads
    // issued, before the grid dependency resolves; q is loaded and the pieces written
    // only after it. Dependents are let launch only once it has resolved.
    const bool early = kPrefix && p.early != 0;
    if (!early) {
        ptx::grid_dependency_wait();
        ptx::launch_dependents();   // successors start once this grid's inputs are final
    }
    // Query tile x covers query rows q0[x] .. q0[x] + rows[x] - 1 (row r: query row
    // q0[x] + r); row r of tile x sees keys t <= its limit: its own position pos0[x] + r
    // (prefill) or every key of the split (prefix). The CTA reads keys [kv_begin,
    // kv_end) through table row srow; tile x needs the first nkt_x of its key tiles.
    int32_t q0[kTiles], rows[kTiles] = {0, 0}, pos0[kTiles] = {0, 0}, kv_end_x[kTiles] = {0, 0};
    int32_t srow, kv_begin, kv_end;
    int32_t split = 0;
    if constexpr (kPrefix) {
        const pkv_prefix_group g = p.groups[blockIdx.z];
        split = blockIdx.x;
        const int32_t P = g.prefix_tokens;
        if (g.num_seqs < 1 || g.num_seqs > kQT || g.first_seq < 0 || g.first_seq > p.S - g.num_seqs || P < 0 ||
            P > cap || P % B != 0) {
            if (tid == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            if (early) {
                ptx::grid_dependency_wait();
                ptx::launch_dependents();
            }
            return;
        }
        srow = g.first_seq;
        const int32_t per = ((P + kKT - 1) / kKT + p.splits - 1) / p.splits;   // key tiles per split
        kv_begin = min(P, split * per * kKT);
        kv_end = min(P, kv_begin + per * kKT);
        q0[0] = q0[1] = g.first_seq;
        rows[0] = g.num_seqs;
        pos0[0] = kv_end - 1;
        kv_end_x[0] = kv_end;
        if (kv_begin >= kv_end) {
            // no keys in this split: an empty piece for every member
            if (early) {
                ptx::grid_dependency_wait();
                ptx::launch_dependents();
            }
            for (int32_t i = tid; i < rows[0] * (kD + 4); i += kThreads) {
                const int32_t r = i / (kD + 4), c = i - r * (kD + 4);
                p.pieces[(((size_t)(q0[0] + r) * H + h) * PKV_MAX_PREFIX_SPLITS + split) * (kD + 4) + c] =
                    c == kD ? -INFINITY : 0.f;
            }
            return;
        }
    } else {
        const int32_t s = blockIdx.z;
        const int32_t qs = p.q_start[s];
        const int32_t C = p.q_start[s + 1] - qs;
        const int32_t i0 = blockIdx.x * (kTiles * kQT);
        // a chunk longer than the grid covers (max_chunk too small): its last rows are
        // not computed, and the call is flagged
        if (blockIdx.x == gridDim.x - 1 && C > (int32_t)gridDim.x * (kTiles * kQT) && tid == 0)
            atomicOr(p.status, PKV_DEV_BAD_LENGTH);
        if (i0 >= C) return;                           // uniform: this pair of tiles has no queries
        int32_t T = p.lens[s];
        if (T < C || T > cap) {
            if (tid == 0) atomicOr(p.status, PKV_DEV_BAD_LENGTH);
            T = T < C ? C : cap;
        }
        srow = s;
        kv_begin = 0;
        for (int x = 0; x < kTiles; ++x) {
            q0[x] = qs + i0 + x * kQT;
            rows[x] = max(0, min(kQT, C - i0 - x * kQT));
            pos0[x] = T - C + i0 + x * kQT;            // position of row 0
            kv_end_x[x] = rows[x] ? pos0[x] + rows[x] : 0;
        }
        kv_end = max(kv_end_x[0], kv_end_x[1]);
    }
    int32_t nkt_x[kTiles];
    for (int x = 0; x < kTiles; ++x) nkt_x[x] = rows[x] ? (kv_end_x[x] - kv_begin + kKT - 1) / kKT : 0;
    const int32_t nkt = max(nkt_x[0], nkt_x[1]);
    const bool has_b = nkt_x[1] > 0;
    // the tile whose P V reads the CTA's last key tile first zeroes its dead V rows
    const int zero_tile = nkt_x[0] == nkt ? 0 : 1;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i)
            ptx::mbar_init(BAR(i), (i == kPReady || i == kPReady + 1) ? (kPrefix ? 8 : kGroupThreads / 32) : 1);
        *timed_out = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         ptx::smem_addr(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tS = [tmem](int x) { return tmem + (uint32_t)x * kKT; };            // P_x is written over it
    auto tO = [tmem](int x) { return tmem + (uint32_t)(2 + x) * kKT; };

    if (warp == 9 || warp == 10) {
        // ================= loaders: warp 9 brings Q and the K tiles, warp 10 the V tiles
        // (one box per block of the table, lane i box i). Separate warps, so a K tile
        // is refilled as soon as its S MMAs are done, whatever the V side waits for.
        const bool is_k = warp == 9;
        const int32_t rowsb = B < kKT ? B : kKT;       // rows per box; B is a power of two, 8..512
        auto issue_q = [&] {
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(BAR(kQFull), (has_b ? 2 : 1) * kTileBytes);
                for (int x = 0; x < kTiles; ++x)
                    if (nkt_x[x] > 0)
                        for (int half = 0; half < 2; ++half)
                            ptx::tma_load_3d(sQ(x) + half * kSub, &qmap, half * kHalf, h, q0[x], BAR(kQFull));
            }
        };
        // early: Q once the K tiles that fit the two slots are issued (before any wait
        // for a free slot, which needs Q's first S done)
        const int32_t jq = early ? min(nkt, 2) : 0;
        auto q_after_wait = [&] {
            ptx::grid_dependency_wait();
            ptx::launch_dependents();
            issue_q();
        };
        if (is_k && !early) issue_q();
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const int full0 = is_k ? kKFull : kVFull;
        const int free0 = is_k ? kKFree : kVFree;     // slot b is free once the MMAs of tile j-2 reading it are done
        for (int32_t j = 0; j < nkt; ++j) {
            if (is_k && early && j == jq) q_after_wait();
            const int b = j & 1;
            const int32_t t0 = kv_begin + j * kKT;
            const int32_t ntok = min(kKT, kv_end - t0);
            const int32_t nbox = B < kKT ? (ntok + B - 1) / B : 1;     // <= 16
            const uint32_t box_bytes = (uint32_t)nbox * rowsb * 128 * 2;
            int32_t y = 0;
            if (lane < nbox) {                          // lane i: box i of the tile
                const int32_t lb = (t0 + lane * rowsb) / B;
                int32_t blk = lb < p.max_blocks ? p.tables[(size_t)srow * p.max_blocks + lb] : -1;
                if (blk < 0 || blk >= p.N) {
                    if (is_k) atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    blk = 0;
                }
                y = (blk * H + h) * B + (B < kKT ? 0 : t0 % B);
            }
            const uint32_t off = (uint32_t)lane * rowsb * 128;
            const uint32_t dst = (is_k ? sK(b) : sV(b)) + off;
            if (j >= 2) bounded_wait(BAR(free0 + b), ((j - 2) >> 1) & 1, timed_out, p.status);
            if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(full0 + b), box_bytes);
            __syncwarp();
            if (lane < nbox)
                for (int half = 0; half < 2; ++half)
                    ptx::tma_load_2d(dst + half * kSub, map, half * kHalf, y, BAR(full0 + b));
        }
        if (is_k && early && jq == nkt) q_after_wait();
        // the last loads into each slot (and Q) have landed before the CTA may exit
        if (is_k) drain_wait(BAR(kQFull), 0);
        for (int32_t j = nkt - 2 < 0 ? 0 : nkt - 2; j < nkt; ++j) drain_wait(BAR(full0 + (j & 1)), (j >> 1) & 1);
    } else if (warp == 8) {
        // ================= MMA issue (one thread)
        if (lane == 0) {
            const uint32_t id_qk = umma_idesc(0), id_pv = umma_idesc(1);
            auto issue_s = [&](int x, int32_t j) {   // S_x = Q_x K_j^T over the head dim, 8 steps of 16
                const int b = j & 1;
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kSub + (ks & 3) * 32;
                    umma(tS(x), umma_desc(sQ(x) + koff, 16, 1024), umma_desc(sK(b) + koff, 16, 1024), id_qk,
                         ks > 0);
                }
                umma_commit(BAR(kSFull + x));
            };
            auto issue_pv = [&](int x, int32_t j) {  // O_x += P_x V_j: A = P (tensor memory), B = V (MN-major)
                const int b = j & 1;
                for (int ks = 0; ks < kKT / 16; ++ks)
                    umma_ts(tO(x), tS(x) + ks * 8, umma_desc(sV(b) + ks * 2048, kSub, 1024), id_pv,
                            (j > 0 || ks > 0) ? 1u : 0u);
                umma_commit(BAR(kOFull + x));
            };
            bounded_wait(BAR(kQFull), 0, timed_out, p.status);
            bounded_wait(BAR(kKFull), 0, timed_out, p.status);
            tc_fence_after();
            for (int x = 0; x < kTiles; ++x)
                if (nkt_x[x] > 0) issue_s(x, 0);
            umma_commit(BAR(kKFree));                    // both S of tile 0 issued
            for (int32_t j = 0; j < nkt; ++j) {
                const int b = j & 1;
                const int32_t jn = j + 1;
                bool k_next_in = false;
                bounded_wait(BAR(kVFull + b), (j >> 1) & 1, timed_out, p.status);
                for (int x = 0; x < kTiles; ++x) {
                    if (j >= nkt_x[x]) continue;
                    bounded_wait(BAR(kPReady + x), j & 1, timed_out, p.status);   // P_x,j written, S_x read
                    tc_fence_after();
                    issue_pv(x, j);
                    if (jn < nkt_x[x]) {   // S_x,j+1 overwrites P_x,j: issued after the P V that reads it
                        if (!k_next_in) {
                            bounded_wait(BAR(kKFull + (jn & 1)), (jn >> 1) & 1, timed_out, p.status);
                            tc_fence_after();
                            k_next_in = true;
                        }
                        issue_s(x, jn);
                    }
                }
                umma_commit(BAR(kVFree + b));            // both P V of tile j issued
                if (jn < nkt) umma_commit(BAR(kKFree + (jn & 1)));   // both S of tile j+1 issued
            }
            // the last commit covers every MMA issued before it
            drain_wait(BAR(kVFree + ((nkt - 1) & 1)), ((nkt - 1) >> 1) & 1);
        }
        __syncwarp();
    } else if constexpr (kPrefix) {
        // ================= prefix pass softmax: one query tile, so all eight warps work on it:
        // row r (tensor-memory lane r) is shared by warps q and q + 4 (q = r / 32), each
        // taking one 64-key half of every S tile and one 64-column half of O; the two
        // exchange their row max (and, at the end, their sums) through shared memory.
        if (early) ptx::grid_dependency_wait();    // the pieces are written only after it
        const int hf = warp >> 2, quad = warp & 3;
        const int32_t r = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float sl2 = p.scale_log2;
        constexpr float kSlack = 8.f;
        constexpr int kCols = kKT / 2;
        const int32_t nk = nkt_x[0];
        const bool valid = r < rows[0];
        float m_ref = -INFINITY, l = 0.f;
        for (int32_t j = 0; j < nk; ++j) {
            const int b = j & 1;
            bounded_wait(BAR(kSFull), j & 1, timed_out, p.status);
            tc_fence_after();
            uint32_t raw[kCols];
            tmem_ld64(tS(0) + lane_base + hf * kCols, raw);
            float xv[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) xv[i] = __uint_as_float(raw[i]);
            const int32_t t0 = kv_begin + j * kKT + hf * kCols;   // first key of this half
            if (!(valid && t0 + kCols - 1 < kv_end)) {   // a ragged last tile (or a row past the group)
#pragma unroll
                for (int i = 0; i < kCols; ++i) xv[i] = (valid && t0 + i < kv_end) ? xv[i] : -INFINITY;
            }
            float m22[22];
#pragma unroll
            for (int k = 0; k < 21; ++k) m22[k] = fmax3(xv[3 * k], xv[3 * k + 1], xv[3 * k + 2]);
            m22[21] = xv[63];
            float m8[8];
#pragma unroll
            for (int k = 0; k < 7; ++k) m8[k] = fmax3(m22[3 * k], m22[3 * k + 1], m22[3 * k + 2]);
            m8[7] = m22[21];
            float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            // a slot per parity, so a fast partner never overwrites a value not yet read
            float *xs = xchg + b * 2 * kQT;
            xs[hf * kQT + r] = mx;
            ptx::named_barrier(1 + quad, 64);
            mx = fmaxf(mx, xs[(hf ^ 1) * kQT + r]) * sl2;
            const bool move = mx > m_ref + kSlack;      // the same in both halves
            const float new_ref = move ? mx : m_ref;
            const float alpha = move ? ptx::ex2(m_ref - new_ref) : 1.f;
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                bounded_wait(BAR(kOFull), (j - 1) & 1, timed_out, p.status);
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < kCols; c0 += 32) {
                    uint32_t w[32];
                    const uint32_t ta = tO(0) + lane_base + hf * kCols + c0;
                    tmem_ld32(ta, w);
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
                    tmem_st32(ta, w);
                }
            }
            m_ref = new_ref;
            // P over S: the partner half has read its S columns before the exchange above
            const float neg = new_ref == -INFINITY ? 0.f : -new_ref;
            float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[kCols / 2];
#pragma unroll
            for (int e = 0; e < kCols / 2; ++e) {
                const float2 a = ptx::ffma2(make_float2(xv[2 * e], xv[2 * e + 1]), make_float2(sl2, sl2),
                                            make_float2(neg, neg));
                const float2 pp = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
                pk[e] = pack_half2(pp.x, pp.y);
                rs2[e & 1] = ptx::fadd2(rs2[e & 1], pp);
            }
            tmem_st32(tS(0) + lane_base + hf * (kCols / 2), pk);
            l = l * alpha + ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y));
            if (j == nk - 1) {
                // the split's last key tile: zero the V rows past the split (a prefix is
                // whole blocks, so only a ragged final tile has them)
                bounded_wait(BAR(kVFull + b), (j >> 1) & 1, timed_out, p.status);
                const int32_t first_dead = kv_end - (kv_begin + j * kKT);
                unsigned char *sVp = base + (4 + b) * kTileBytes;
                const int32_t nwords = (kKT - first_dead) * 8;
                for (int32_t w = tid; w < nwords * 2; w += 2 * kGroupThreads) {
                    const int half = w / nwords, rem = w - half * nwords;
                    const int row = first_dead + rem / 8, cc = rem & 7;
                    *reinterpret_cast<uint4 *>(sVp + half * kSub + row * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(kPReady));
        }
        if (nk > 0) {
            bounded_wait(BAR(kOFull), (nk - 1) & 1, timed_out, p.status);
            tc_fence_after();
            float *xs = xchg + (nk & 1) * 2 * kQT;   // the slot of parity nk & 1 is free by now
            xs[hf * kQT + r] = l;
            ptx::named_barrier(1 + quad, 64);
            const float lt = xs[r] + xs[kQT + r];
            uint32_t raw[kCols];
            tmem_ld64(tO(0) + lane_base + hf * kCols, raw);
            if (valid) {
                float *piece = p.pieces + (((size_t)(q0[0] + r) * H + h) * PKV_MAX_PREFIX_SPLITS + split) * (kD + 4);
                float4 *o4 = reinterpret_cast<float4 *>(piece + hf * kCols);
#pragma unroll
                for (int d = 0; d < kCols; d += 4)
                    o4[d / 4] = make_float4(__uint_as_float(raw[d]), __uint_as_float(raw[d + 1]),
                                            __uint_as_float(raw[d + 2]), __uint_as_float(raw[d + 3]));
                if (hf == 0) *reinterpret_cast<float4 *>(piece + kD) = make_float4(m_ref, lt, 0.f, 0.f);
            }
        }
    } else {
        // ================= softmax warps: warps 0-3 own query tile A, warps 4-7 tile B, one
        // thread per query row (row r = tensor-memory lane r, warp 4x + r / 32), so the two
        // tiles' softmax run side by side and a row's max and sum never leave its thread.
        // O lives in tensor memory and P V accumulates onto it. The softmax runs against a
        // reference max m_ref (log2 units) that only moves when the row's max exceeds it
        // by more than 2^8 (then O and l are rescaled), so P stays <= 256 and most tiles
        // need no O traffic at all.
        const int x = warp >> 2, quad = warp & 3;
        const int32_t r = quad * 32 + lane;
        const int gtid = tid - x * kGroupThreads;       // thread index inside the tile's group
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float sl2 = p.scale_log2;
        constexpr float kSlack = 8.f;
        constexpr int kHalfKeys = kKT / 2;              // keys of one tensor-memory load
        const int32_t nk = nkt_x[x];
        const bool valid = r < rows[x];
        const int32_t pr = pos0[x] + r;                 // the last key this row sees
        float m_ref = -INFINITY, l = 0.f;
        // row max of 64 scores: a tree of three-input maxima (64 -> 22 -> 8 -> 3 -> 1)
        auto max64 = [](const float (&v)[kHalfKeys]) {
            float m22[22];
#pragma unroll
            for (int k = 0; k < 21; ++k) m22[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
            m22[21] = v[63];
            float m8[8];
#pragma unroll
            for (int k = 0; k < 7; ++k) m8[k] = fmax3(m22[3 * k], m22[3 * k + 1], m22[3 * k + 2]);
            m8[7] = m22[21];
            return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        };
        // mask one half (64 keys from t0) of this row's scores past the row's last key
        auto mask_half = [&](int half, int32_t t0, float (&v)[kHalfKeys]) {
            const int32_t k0 = t0 + half * kHalfKeys;
            if (!(valid && k0 + kHalfKeys - 1 <= pr)) {   // the diagonal tile (or a row past the chunk)
#pragma unroll
                for (int i = 0; i < kHalfKeys; ++i) v[i] = (valid && k0 + i <= pr) ? v[i] : -INFINITY;
            }
        };
        // P = 2^(x * scale log2(e) - m_ref) of one half, pairs at a time, packed fp16 into
        // tensor-memory columns [32 half, 32 half + 32) of S; returns the half's sum
        auto store_p = [&](int half, const float (&v)[kHalfKeys], float neg) {
            float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[kHalfKeys / 2];
#pragma unroll
            for (int e = 0; e < kHalfKeys / 2; ++e) {
                const float2 a = ptx::ffma2(make_float2(v[2 * e], v[2 * e + 1]), make_float2(sl2, sl2),
                                            make_float2(neg, neg));
                const float2 pp = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
                pk[e] = pack_half2(pp.x, pp.y);
                rs2[e & 1] = ptx::fadd2(rs2[e & 1], pp);
            }
            tmem_st32(tS(x) + lane_base + half * (kHalfKeys / 2), pk);
            return (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
        };
        for (int32_t j = 0; j < nk; ++j) {
            const int b = j & 1;
            const int32_t t0 = kv_begin + j * kKT;      // first key of the tile
            bounded_wait(BAR(kSFull + x), j & 1, timed_out, p.status);
            tc_fence_after();
            // both halves of this row's scores at once
            float v0[kHalfKeys], v1[kHalfKeys];
            {
                uint32_t r0[kHalfKeys], r1[kHalfKeys];
                tmem_ld64x2(tS(x) + lane_base, tS(x) + lane_base + kHalfKeys, r0, r1);
#pragma unroll
                for (int i = 0; i < kHalfKeys; ++i) {
                    v0[i] = __uint_as_float(r0[i]);
                    v1[i] = __uint_as_float(r1[i]);
                }
            }
            mask_half(0, t0, v0);
            mask_half(1, t0, v1);
            const float mx = fmaxf(max64(v0), max64(v1)) * sl2;
            const bool move = mx > m_ref + kSlack;      // false when mx = -inf
            const float new_ref = move ? mx : m_ref;
            const float alpha = move ? ptx::ex2(m_ref - new_ref) : 1.f;   // m_ref = -inf: 0
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                // rescale this row of O once P V of the previous key tile is in it
                bounded_wait(BAR(kOFull + x), (j - 1) & 1, timed_out, p.status);
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < kD; c0 += 32) {
                    uint32_t w[32];
                    const uint32_t ta = tO(x) + lane_base + c0;
                    tmem_ld32(ta, w);
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
                    tmem_st32(ta, w);
                }
            }
            m_ref = new_ref;
            // P over S: both halves are in registers, so the columns may be overwritten. A
            // row with no live key yet (m_ref = -inf: every score is -inf) gets 0.
            const float neg = new_ref == -INFINITY ? 0.f : -new_ref;
            float rsum = store_p(0, v0, neg);            // columns [0, 32)
            rsum += store_p(1, v1, neg);                 // columns [32, 64)
            l = l * alpha + rsum;
            // the CTA's last key tile: zero the V rows no query of the CTA may see (they
            // may hold non-finite garbage), before the first P V that reads the tile
            if (j == nkt - 1 && x == zero_tile) {
                bounded_wait(BAR(kVFull + b), (j >> 1) & 1, timed_out, p.status);
                const int32_t first_dead = kv_end - t0;  // rows [first_dead, 128)
                unsigned char *sVp = base + (4 + b) * kTileBytes;
                const int32_t nwords = (kKT - first_dead) * 8;    // 16-byte words per half
                for (int32_t w = gtid; w < nwords * 2; w += kGroupThreads) {
                    const int half = w / nwords, rem = w - half * nwords;
                    const int row = first_dead + rem / 8, cc = rem & 7;
                    *reinterpret_cast<uint4 *>(sVp + half * kSub + row * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // zeroed V -> MMA
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(kPReady + x));
        }
        if (nk > 0) {
            bounded_wait(BAR(kOFull + x), (nk - 1) & 1, timed_out, p.status);
            tc_fence_after();
            const int32_t qrow = q0[x] + r;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t raw[kHalfKeys];
                tmem_ld64(tO(x) + lane_base + half * kHalfKeys, raw);
                if (valid) {
                    const float inv = 1.f / l;
                    __half *dst = p.out + ((size_t)qrow * H + h) * kD + half * kHalfKeys;
#pragma unroll
                    for (int d = 0; d < kHalfKeys; d += 8) {
                        __half2 hv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            hv[e] = __floats2half2_rn(__uint_as_float(raw[d + 2 * e]) * inv,
                                                      __uint_as_float(raw[d + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4 *>(dst + d) = *reinterpret_cast<const uint4 *>(hv);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
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

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// q ([rows][H][D] fp16) as a 3-D tensor (D, H, row), boxes of 64 x 1 x 128; the
// pool layer as rows of D, boxes of 64 x min(B, 128). 128-byte swizzle.
pkv_status encode_maps(const pkv_pool *pool, int32_t layer, const void *q, int32_t q_rows, CUtensorMap *qmap,
                       CUtensorMap *kmap, CUtensorMap *vmap) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const pkv_pool_desc &d = pool->desc;
    const PoolLayer pl = pool_layer(pool, layer);
    const int H = d.num_heads, B = d.block_size, N = d.num_blocks;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)q_rows};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
        const cuuint32_t box[3] = {kHalf, 1, kQT}, es[3] = {1, 1, 1};
        if (fn(qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(q), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(PKV_ERR_CUDA, "q tensor map");
    }
    for (int which = 0; which < 2; ++which) {
        const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)N * H * B};
        const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
        const cuuint32_t box[2] = {kHalf, (cuuint32_t)(B < kKT ? B : kKT)}, es[2] = {1, 1};
        if (fn(which ? vmap : kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, which ? pl.v : pl.k, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(PKV_ERR_CUDA, "pool tensor map");
    }
    return PKV_OK;
}

pkv_status check_pool(const pkv_pool *pool, int32_t layer, const char *what) {
    if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
    const pkv_pool_desc &d = pool->desc;
    if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
    if (layer < 0 || layer >= d.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (d.head_dim != kD || d.kv_dtype != PKV_KV_F16 || d.layout != PKV_LAYOUT_HND)
        return fail(PKV_ERR_UNSUPPORTED, "%s is built for fp16 HND pools with head_dim 128", what);
    return PKV_OK;
}

PrefillParams base_params(const pkv_pool *pool, const int32_t *block_tables, int32_t max_blocks, int32_t num_seqs,
                          float scale, uint32_t *status) {
    const pkv_pool_desc &d = pool->desc;
    PrefillParams prm = {};
    prm.tables = block_tables;
    prm.status = status;
    prm.S = num_seqs;
    prm.H = d.num_heads;
    prm.max_blocks = max_blocks;
    prm.B = d.block_size;
    prm.N = d.num_blocks;
    prm.splits = 1;
    const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)kD);
    prm.scale_log2 = (float)(sc * 1.4426950408889634);
    return prm;
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices][2];
cudaError_t g_attr_err[kMaxDevices][2];

template <bool kPrefix>
pkv_status launch_tc(dim3 grid, const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                     const PrefillParams &prm, void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_CUDA, "no usable CUDA device");
    std::call_once(g_attr_once[dev][kPrefix], [dev] {
        g_attr_err[dev][kPrefix] = cudaFuncSetAttribute(prefill_attention_kernel<kPrefix>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (g_attr_err[dev][kPrefix] != cudaSuccess)
        return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(g_attr_err[dev][kPrefix]));
    cudaError_t e = launch_pdl(prefill_attention_kernel<kPrefix>, grid, dim3(kThreads), (size_t)kSmemBytes,
                               static_cast<cudaStream_t>(stream), qmap, kmap, vmap, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s launch: %s", kPrefix ? "prefix" : "prefill",
                                      cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_prefill_attention(const pkv_pool *pool, int32_t layer, const void *q, const int32_t *q_start,
                                 int32_t total_q, int32_t num_seqs, int32_t max_chunk, const int32_t *block_tables,
                                 int32_t max_blocks, const int32_t *context_lens, float scale, void *out,
                                 uint32_t *status, void *stream) {
    pkv_status st = check_pool(pool, layer, "prefill attention");
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || total_q < 0 || max_chunk < 0 || max_blocks < 1)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes");
    if (num_seqs == 0 || total_q == 0 || max_chunk == 0) return PKV_OK;
    if (num_seqs > 65535) return fail(PKV_ERR_INVALID_ARG, "num_seqs > 65535");
    if (!q || !q_start || !block_tables || !context_lens || !out || !status)
        return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument (status is required here)");
    if (!aligned16(q) || !aligned16(out)) return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    CUtensorMap qmap, kmap, vmap;
    st = encode_maps(pool, layer, q, total_q, &qmap, &kmap, &vmap);
    if (st != PKV_OK) return st;
    PrefillParams prm = base_params(pool, block_tables, max_blocks, num_seqs, scale, status);
    prm.q_start = q_start;
    prm.lens = context_lens;
    prm.out = static_cast<__half *>(out);
    const dim3 grid((max_chunk + kTiles * kQT - 1) / (kTiles * kQT), pool->desc.num_heads, num_seqs);
    return launch_tc<false>(grid, qmap, kmap, vmap, prm, stream);
}

pkv_status pkv_prefix_attention(const pkv_pool *pool, int32_t layer, const void *q, const pkv_prefix_group *groups,
                                int32_t num_groups, int32_t splits, const int32_t *block_tables, int32_t max_blocks,
                                int32_t num_seqs, float scale, void *pieces, size_t pieces_bytes, uint32_t *status,
                                uint32_t flags, void *stream) {
    // an E4M3 pool (HND, head_dim 128) has its own prefix pass; the checks below hold for both
    const bool q8 = pool && pool->desc.kv_dtype == PKV_KV_E4M3 && pool->desc.layout == PKV_LAYOUT_HND &&
                    pool->desc.head_dim == kD;
    pkv_status st = q8 ? PKV_OK : check_pool(pool, layer, "the prefix pass");
    if (st != PKV_OK) return st;
    if (q8) {
        if (!pool->k_pool) return fail(PKV_ERR_INVALID_ARG, "pool has no device memory");
        if (layer < 0 || layer >= pool->desc.num_layers) return fail(PKV_ERR_INVALID_ARG, "layer %d out of range", layer);
        if (!pool->k_scale || !aligned16(pool->k_scale) || !aligned16(pool->v_scale))
            return fail(PKV_ERR_INVALID_ARG, "an E4M3 pool needs 16-byte aligned scale pools (pkv_pool_set_scales)");
    }
    if (flags & ~(uint32_t)PKV_ATTN_INPUTS_EARLY) return fail(PKV_ERR_INVALID_ARG, "unknown flags %#x", flags);
    if (num_groups < 0 || num_seqs < 0 || max_blocks < 1 || splits < 1 || splits > PKV_MAX_PREFIX_SPLITS)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (splits in 1..%d)", PKV_MAX_PREFIX_SPLITS);
    if (num_groups == 0 || num_seqs == 0) return PKV_OK;
    if (num_groups > 65535) return fail(PKV_ERR_INVALID_ARG, "num_groups > 65535");
    if (!q || !groups || !block_tables || !pieces || !status)
        return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument (status is required here)");
    if (!aligned16(q) || !aligned16(pieces))
        return fail(PKV_ERR_INVALID_ARG, "q and pieces must be 16-byte aligned");
    const pkv_pool_desc &d = pool->desc;
    const size_t need = (size_t)num_seqs * d.num_heads * PKV_MAX_PREFIX_SPLITS * (kD + 4) * sizeof(float);
    if (pieces_bytes < need) return fail(PKV_ERR_INVALID_ARG, "pieces: %zu bytes < %zu needed", pieces_bytes, need);
    if (q8)
        return prefix_attention_q8(pool, layer, q, groups, num_groups, splits, block_tables, max_blocks, num_seqs,
                                   scale, pieces, status, flags, stream);
    CUtensorMap qmap, kmap, vmap;
    st = encode_maps(pool, layer, q, num_seqs, &qmap, &kmap, &vmap);
    if (st != PKV_OK) return st;
    PrefillParams prm = base_params(pool, block_tables, max_blocks, num_seqs, scale, status);
    prm.groups = groups;
    prm.pieces = static_cast<float *>(pieces);
    prm.splits = splits;
    prm.early = (flags & PKV_ATTN_INPUTS_EARLY) ? 1 : 0;
    const dim3 grid(splits, d.num_heads, num_groups);
    return launch_tc<true>(grid, qmap, kmap, vmap, prm, stream);
}

}  // extern "C"
