// ep_common.cuh -- device helpers shared by the dispatch / combine kernels (sm_103a): streaming
// 16-byte accesses, programmatic dependent launch, the status word and bf16 <-> fp32.  The
// quantisation helpers of the dispatch kernels are in ep_quant.cuh.
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

// Programmatic dependent launch.  Every kernel first waits (griddepcontrol.wait) until the
// kernel before it in the stream has completed and its memory is visible, so it never reads
// anything before all earlier work in the stream is done.
//   pdl_begin: grids whose CTAs are all resident at once (persistent grids, the layout) then
//              let the next kernel start launching, so its launch and ramp-up overlap this
//              kernel's run.
//   pdl_wait:  grids with more CTAs than fit at once only wait; the next kernel launches as
//              their CTAs finish.  Signalled early, the next kernel's CTAs would take SM slots
//              this grid's later CTAs still need, and sit waiting for it: on GB300 a persistent
//              combine launched that way behind a 32,768-CTA per-token dispatch made the pair
//              30% slower (1157 against 886 us).
// All are no-ops when the kernel was launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_wait();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// pdl_begin for grids that fit in one wave, else pdl_wait.  `one_wave` comes from the host,
// which compares the grid with the device's SM count (the %nsmid register only bounds the SM
// ids and may exceed the count).
__device__ __forceinline__ void pdl_begin_if(int one_wave) {
    if (one_wave) pdl_begin();
    else pdl_wait();
}

// Status word of the layout: read once per CTA; a non-zero word means "write nothing".
__device__ __forceinline__ int load_status(const int32_t *status) {
    return *reinterpret_cast<const volatile int32_t *>(status);
}

// ---------------------------------------------------------------------------------------
// The bounds-checked debug build (compiled with -DEP_BOUNDS_CHECK=1) checks every index that
// comes from data against the buffer it indexes, skips an access that fails and sets
// EP_STATUS_BOUNDS in the layout's status word.  In the default build kBoundsCheck is false
// and the extra checks compile away.
// ---------------------------------------------------------------------------------------
#ifndef EP_BOUNDS_CHECK
#define EP_BOUNDS_CHECK 0
#endif
constexpr bool kBoundsCheck = EP_BOUNDS_CHECK != 0;

// The status word as one value for the whole CTA; every thread of the CTA must call it.  Only
// the layout writes the word, and it completes before any kernel that reads it starts, so in
// the default build every thread reads the same value.  In the bounds-checked build another CTA
// of the running kernel may set EP_STATUS_BOUNDS meanwhile, so the CTA agrees on one reading
// (one barrier) before it acts on it.
__device__ __forceinline__ int cta_status(const int32_t *status) {
    if (kBoundsCheck) return __syncthreads_or(load_status(status));
    return load_status(status);
}

// Records a failed check in the status word (checked build only).
__device__ __forceinline__ void bounds_fail(const int32_t *status) {
    if (kBoundsCheck) atomicOr(const_cast<int32_t *>(status), EP_STATUS_BOUNDS);
}

// Whether a row read from a layout may be used.  Both builds skip rows outside [0, R_max)
// (-1 marks an unused slot); the checked build also records any such row other than -1.
__device__ __forceinline__ bool row_ok(int r, int R_max, const int32_t *status) {
    if (r >= 0 && r < R_max) return true;
    if (r != -1) bounds_fail(status);
    return false;
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

}  // namespace ep
