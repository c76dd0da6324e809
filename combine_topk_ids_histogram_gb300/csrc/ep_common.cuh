// ep_common.cuh -- device helpers shared by the dispatch / combine kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------------------
// 16-byte global accesses.  Token rows and expert-output rows are each touched once per call,
// so loads and stores use the streaming (evict-first) cache policy.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st_stream(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }

// Programmatic dependent launch.  Every kernel first waits until the kernel before it in the
// stream has completed and its memory is visible, and only then lets the next kernel start
// launching; so a kernel never reads anything before all earlier work in the stream is done,
// while the next kernel's launch and ramp-up overlap this kernel.  Both are no-ops when the
// kernel was launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Status word of the layout: read once per CTA; a non-zero word means "write nothing".
__device__ __forceinline__ int load_status(const int32_t *status) {
    return *reinterpret_cast<const volatile int32_t *>(status);
}

// ---------------------------------------------------------------------------------------
// bf16 <-> fp32.  A 32-bit word holds two bf16: element 2i in the low half.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two fp32 values to bf16 (nearest, ties to even) and pack `lo` into the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void unpack8(uint4 v, float f[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

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

// Value of a non-negative finite E4M3 code (bias 7; exponent field 0 is subnormal, m * 2^-9).
// Built bit by bit, so it is exact.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    uint32_t ex = (c >> 3) & 15u, m = c & 7u;
    if (ex == 0) return (float)m * 0.001953125f;   // m * 2^-9, exact
    return __uint_as_float(((ex + 120u) << 23) | (m << 20));
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
