// E4M3 conversion and bf16 amax helpers shared by the quantisers.
#pragma once
#include <cstdint>

namespace temx {

// 2^(127 - s) as fp32 (s <= 247 for every finite block of either recipe, so
// always a normal number).
__device__ __forceinline__ float inv_scale(uint32_t s) {
    return __uint_as_float((254u - s) << 23);
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two fp32 -> two E4M3 bytes (round to nearest even, saturate): `lo` in the
// low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four consecutive bf16 (two words) -> four E4M3 bytes in one word.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float m) {
    const uint32_t a = cvt_e4m3x2(__fmul_rn(bf16_lo(w0), m), __fmul_rn(bf16_hi(w0), m));
    const uint32_t b = cvt_e4m3x2(__fmul_rn(bf16_lo(w1), m), __fmul_rn(bf16_hi(w1), m));
    return a | (b << 16);
}

// Largest |x| of 2n words of bf16 pairs, as bf16 bits (tree of max.u16x2).
template <int kWords>
__device__ __forceinline__ uint32_t amax_words(const uint32_t* w) {
    uint32_t m[kWords / 2];
#pragma unroll
    for (int i = 0; i < kWords / 2; ++i) m[i] = max_u16x2(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
    for (int s = kWords / 4; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) m[i] = max_u16x2(m[i], m[i + s]);
    return m[0];                          // two maxima, one per 16-bit half
}

}  // namespace temx
