// ep_quant.cuh -- device helpers of the quantising dispatch kernels (sm_103a): the NVFP4 / E4M3
// hardware conversions, packed fp32 products, and exact maxima of magnitudes.
#pragma once

#include "ep_common.cuh"

namespace ep {

// ---------------------------------------------------------------------------------------
// NVFP4 element and scale formats, converted by the sm_100-family hardware instructions
// (round to nearest even, saturating to the largest finite value).
// ---------------------------------------------------------------------------------------
// Two fp32 -> two E2M1 codes in one byte: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> two E4M3 codes: `lo` in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Value of an E4M3 code held in the low byte of `c`, by the hardware conversion to f16 and then
// to fp32.  Both are exact: every finite E4M3 value (largest 448, smallest subnormal 2^-9) is
// an f16 value.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const unsigned short pair = static_cast<unsigned short>(c & 0xffu);   // upper code: 0
    float f;
    asm("{\n\t.reg .b32 h;\n\t.reg .f16 lo, hi;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, %1;\n\t"
        "mov.b32 {lo, hi}, h;\n\t"
        "cvt.f32.f16 %0, lo;\n\t}"
        : "=f"(f) : "h"(pair));
    return f;
}

// (a0 * b, a1 * b), each product rounded to nearest even in fp32 (one packed instruction).
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b, float &d0, float &d1) {
    asm("{\n\t.reg .b64 x, y, d;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %4};\n\t"
        "mul.rn.f32x2 d, x, y;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b));
}

// ---------------------------------------------------------------------------------------
// Largest magnitude of packed bf16 values, without unpacking.  With the sign bit cleared, the
// 15-bit pattern of a finite bf16 orders like its magnitude (subnormals included), so two
// 16-bit unsigned maxima per instruction give the exact maximum.  (Infinity compares above
// every finite value; a NaN, outside the method's domain, would compare above infinity.)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Per 16-bit half: the largest magnitude pattern among the word's halves at that position.
__device__ __forceinline__ uint32_t absmax_bits(uint4 v) {
    constexpr uint32_t kMag = 0x7fff7fffu;
    return max_u16x2(max_u16x2(v.x & kMag, v.y & kMag), max_u16x2(v.z & kMag, v.w & kMag));
}
// The larger of the two halves, as an fp32 value (exact: bf16 -> fp32 is a shift).
__device__ __forceinline__ float absmax_value(uint32_t m) {
    return __uint_as_float(max_u16x2(m, m >> 16) << 16);
}
// max |x| over the 16 bf16 values of two 16-byte words.
__device__ __forceinline__ float absmax16(uint4 a, uint4 b) {
    return absmax_value(max_u16x2(absmax_bits(a), absmax_bits(b)));
}

// ---------------------------------------------------------------------------------------
// Block-wide maximum of non-negative floats (all threads get the result).  `red` holds one
// slot per warp.  Non-negative floats order like their bit patterns, so each warp reduces
// with one unsigned-maximum instruction.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max_nonneg(float v) {
    return __uint_as_float(__reduce_max_sync(kFullMask, __float_as_uint(v)));
}

__device__ __forceinline__ float block_max_nonneg(float v, float *red) {
    v = warp_max_nonneg(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    float m = 0.0f;
    for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
    return m;
}

}  // namespace ep
