/*
 * Decode-attention oracle in plain C, float64 (test infrastructure only).
 *
 * Same definition as oracle/ref_attn.py, written independently as loops: for
 * each (sequence s, head h), walk the tokens t = 0..T_s-1, find token t in
 * physical block table[s][t / B] at slot t % B (m.lqnn.cn/news/240480 §3.3),
 * and compute softmax(scale * q.K^T) V over all of them with the maximum
 * subtracted (icman.com.cn/news/78786 §1.1, §2.4). Inputs are IEEE binary16
 * bit patterns; every product and sum is in double. OpenMP spreads the
 * (sequence, head) pairs over the host cores; there are no SIMD intrinsics.
 *
 * This is the CPU baseline the benchmark times; it shares nothing with the
 * CUDA library.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition. */
static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)frac, -24);             /* subnormal: frac * 2^-24 */
    } else if (exp == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), exp - 25); /* (1024 + frac) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

double oracle_half_to_double(uint16_t h) { return half_to_double(h); }

/* Row of D elements holding (block, slot, head); layout 0 = [B][H][D], 1 = [H][B][D]. */
static int64_t kv_row(int layout, int64_t block, int64_t slot, int64_t head, int64_t H, int64_t B) {
    return layout == 0 ? (block * B + slot) * H + head : (block * H + head) * B + slot;
}

/*
 * q: [S][H][D] binary16; k_pool, v_pool: one layer, N blocks; tables: [S][max_blocks];
 * lens: [S]; out: [S][H][D] double. pairs (nullable): num_pairs (s, h) pairs to compute,
 * the rest of out is left untouched. Returns 0, -1 on a bad argument (a block id
 * outside [0, N) or a length beyond the table), or -2 if scratch memory ran out.
 */
int oracle_decode_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                            int layout, int64_t N, int B, int H, int D,
                            const int32_t *tables, int max_blocks, const int32_t *lens, int S,
                            double scale, double *out, const int32_t *pairs, int num_pairs,
                            int num_threads) {
    int64_t total = pairs ? (int64_t)num_pairs : (int64_t)S * H;
    int bad = 0;
    for (int s = 0; s < S; ++s) {
        if (lens[s] < 0 || (int64_t)lens[s] > (int64_t)max_blocks * B) bad = 1;
        int nb = (lens[s] + B - 1) / B;
        for (int i = 0; i < nb && !bad; ++i)
            if (tables[(int64_t)s * max_blocks + i] < 0 || tables[(int64_t)s * max_blocks + i] >= N) bad = 1;
    }
    if (bad) return -1;
    int oom = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
#pragma omp parallel
    {
        int64_t cap = 0;
        double *x = NULL;
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < total; ++w) {
            int s = pairs ? pairs[2 * w] : (int)(w / H);
            int h = pairs ? pairs[2 * w + 1] : (int)(w % H);
            int T = lens[s];
            double *o = out + ((int64_t)s * H + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (T == 0) continue;
            if (T > cap) {
                free(x);
                cap = T;
                x = (double *)malloc(sizeof(double) * (size_t)cap);
                if (!x) {
                    cap = 0;
#pragma omp atomic write
                    oom = 1;
                    continue;
                }
            }
            const uint16_t *qv = q + ((int64_t)s * H + h) * D;
            double mx = -INFINITY;
            for (int t = 0; t < T; ++t) {
                int64_t blk = tables[(int64_t)s * max_blocks + t / B];
                const uint16_t *kr = k_pool + kv_row(layout, blk, t % B, h, H, B) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += half_to_double(qv[d]) * half_to_double(kr[d]);
                x[t] = scale * dot;
                if (x[t] > mx) mx = x[t];
            }
            double denom = 0.0;
            for (int t = 0; t < T; ++t) {
                x[t] = exp(x[t] - mx);
                denom += x[t];
            }
            for (int t = 0; t < T; ++t) {
                int64_t blk = tables[(int64_t)s * max_blocks + t / B];
                const uint16_t *vr = v_pool + kv_row(layout, blk, t % B, h, H, B) * D;
                double wt = x[t] / denom;
                for (int d = 0; d < D; ++d) o[d] += wt * half_to_double(vr[d]);
            }
        }
        free(x);
    }
    return oom ? -2 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
