// FP8 E4M3 quantisation of one KV row for the quantised cache: one fp32 scale
// per (token, head) row, scale = amax / 448 (1 for an all-zero row), code =
// round-to-nearest-even(x / scale) saturated to the largest finite E4M3 value.
// Divisions are IEEE round-to-nearest so the codes are reproducible bit for bit.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstring>

namespace pkv {
namespace q8 {

constexpr float kE4M3Max = 448.f;

// Largest |x| over the 8 fp16 values of a 16-byte word.
__device__ __forceinline__ float amax_word(const uint4 &w) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h;
        memcpy(&h, &v[i], 4);
        const float2 f = __half22float2(h);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    return m;
}

__device__ __forceinline__ float row_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f; }

// 8 fp16 values -> 8 E4M3 codes (element 0 in the lowest byte).
__device__ __forceinline__ uint2 quantize_word(const uint4 &w, float scale) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h;
        memcpy(&h, &v[i], 4);
        const float2 f = __half22float2(h);
        const float2 y = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
        const uint32_t c = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
        out[i >> 1] |= (c & 0xFFFFu) << (16 * (i & 1));
    }
    return make_uint2(out[0], out[1]);
}

// Two E4M3 codes (low byte = element 0) -> their fp16 pair as a 32-bit word.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t two_codes) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu), __NV_E4M3);
    uint32_t out;
    memcpy(&out, &r, 4);
    return out;
}

// Four E4M3 codes (byte i = element i) -> two fp16 pairs: lo = elements 0, 1 and
// hi = elements 2, 3 (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t four_codes, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 c0, c1;\n\tmov.b32 {c0, c1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c0;\n\tcvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
}

}  // namespace q8
}  // namespace pkv
