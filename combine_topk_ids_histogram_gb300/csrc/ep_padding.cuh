// ep_padding.cuh -- the padding rows of a padded layout (token_dispatcher page,
// TokenDispatcherConfig.moe_router_expert_pad_multiple), written by extra CTAs that lead the
// grids of the dispatch kernels and of the combine backward kernel, so the fill runs
// alongside the per-token work instead of after it.
#pragma once

#include "ep_common.cuh"

namespace ep {

// One buffer whose padding rows a kernel fills: `row_bytes` per row, every 32-bit word of a
// padding row set to `pattern`.  Rows are written with the widest store their size and start
// allow: 16-, 4-, 2- or 1-byte stores, so a pattern must be 16-bit periodic when row_bytes is
// not a multiple of 4, and byte periodic when it is odd (the NVFP4 block-scale row, H/16 bytes,
// can be odd).  A null ptr means no buffer.
struct PadFill {
    void *ptr;
    int row_bytes;
    uint32_t pattern;
};

__device__ __forceinline__ void fill_row(const PadFill &f, int row, int lane) {
    if (!f.ptr) return;
    unsigned char *p = static_cast<unsigned char *>(f.ptr) + (size_t)row * f.row_bytes;
    if (f.row_bytes % 16 == 0) {
        const uint4 v = make_uint4(f.pattern, f.pattern, f.pattern, f.pattern);
        for (int i = lane; i < f.row_bytes / 16; i += 32) st_stream(reinterpret_cast<uint4 *>(p) + i, v);
    } else if (f.row_bytes % 4 == 0) {
        for (int i = lane; i < f.row_bytes / 4; i += 32) reinterpret_cast<uint32_t *>(p)[i] = f.pattern;
    } else if (f.row_bytes % 2 == 0) {
        for (int i = lane; i < f.row_bytes / 2; i += 32)
            reinterpret_cast<uint16_t *>(p)[i] = (uint16_t)f.pattern;
    } else {   // odd row size: rows start on any byte
        for (int i = lane; i < f.row_bytes; i += 32) p[i] = (unsigned char)f.pattern;
    }
}

// Group g's padding rows close the group: [first, row_offsets[g+1]), at most pad - 1 of them,
// where `first` is the lowest row among the group's last pad - 1 rows whose source token is -1
// (every row before it is one of the group's routed rows).  The group's rows are shared by
// `nparts` CTAs: the whole CTA finds `first`, then its warps write the rows of part `part`
// (every nparts-th warp-sized step).  Call only while the layout's status word is 0 (then every
// row is below R_max); the bounds-checked build also checks the group's rows against
// [0, R_max) and records a group outside it instead of filling it.
__device__ __forceinline__ void fill_group_padding(int g, int part, int nparts, int pad, int R_max,
                                                   const int32_t *__restrict__ row_offsets,
                                                   const int32_t *__restrict__ src_info,
                                                   const int32_t *__restrict__ status, const PadFill &f0,
                                                   const PadFill &f1, const PadFill &f2) {
    __shared__ int s_first;
    const int hi = row_offsets[g + 1];
    const int lo = max(row_offsets[g], hi - (pad - 1));
    if (kBoundsCheck && (lo < 0 || hi > R_max || lo > hi)) {
        if (threadIdx.x == 0) bounds_fail(status);
        return;
    }
    if (threadIdx.x == 0) s_first = hi;
    __syncthreads();
    for (int r = lo + threadIdx.x; r < hi; r += blockDim.x)
        if (src_info[2 * (size_t)r] < 0) atomicMin(&s_first, r);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int r = s_first + part * nw + warp; r < hi; r += nw * nparts) {
        fill_row(f0, r, lane);
        fill_row(f1, r, lane);
        fill_row(f2, r, lane);
    }
}

// The same as a separate function, for kernels whose own register allocation should not
// carry the fill's.
static __device__ __noinline__ void fill_group_padding_call(int g, int part, int nparts, int pad, int R_max,
                                                            const int32_t *__restrict__ row_offsets,
                                                            const int32_t *__restrict__ src_info,
                                                            const int32_t *__restrict__ status,
                                                            PadFill f0, PadFill f1, PadFill f2) {
    fill_group_padding(g, part, nparts, pad, R_max, row_offsets, src_info, status, f0, f1, f2);
}

// CTAs sharing one group's padding rows, for CTAs of `threads` threads: enough for about eight
// warps per group (a group has at most pad - 1 padding rows, and a lone warp's stores drain
// slowly while the token CTAs keep the memory system busy).
inline int fill_parts(const ep_layout_t *L, int threads) {
    const int warps = threads / 32 > 0 ? threads / 32 : 1;
    int parts = (8 + warps - 1) / warps;
    if (parts > L->pad_multiple - 1) parts = L->pad_multiple - 1;
    return parts > 1 ? parts : 1;
}

// Extra leading CTAs of a grid for a layout's padding rows: fill_parts per group when padded.
inline int fill_ctas(const ep_layout_t *L, int threads) {
    return L->pad_multiple > 1 ? (L->E + L->fused_shared) * fill_parts(L, threads) : 0;
}

}  // namespace ep
