// ep_dispatch.cu -- permute-scatter of token rows into the expert-major layout, as NVFP4 with
// a per-token global scale (Mojo EP dispatch page, DistributedEPDispatchBlockScaledNVDynGlobal
// Scales.execute), as plain bf16 (fused_a2a page, HybridEPDispatch.forward) or as FP8 with
// per-block scales (fused_a2a page, init_hybrid_ep_buffer, fp8_dispatch); and the padding rows
// of padded layouts (token_dispatcher page, TokenDispatcherConfig.moe_router_expert_pad_multiple).
//
// NVFP4 kernel: one CTA per token.  Each thread owns a contiguous chunk of BPT 16-element
// blocks (BPT = 2 -> 32 elements: 4 x 16-byte loads in, one 16-byte code store and one 2-byte
// scale store per destination row).  The token row is read from HBM exactly once and stays in
// registers: the row maximum is a block-wide reduction, the block maxima are per thread, the
// E4M3 and E2M1 encodings are single hardware conversions, and the same bytes are then
// stored to each of the token's K (+1 shared) rows.  The fused layout + NVFP4 calls run the
// staged kernel described further down instead, where its shape allows.
#include "ep_common.cuh"
#include "ep_async.cuh"
#include "ep_host.h"
#include "ep_padding.cuh"
#include "ep_quant.cuh"

namespace ep {
namespace {

constexpr int kMaxRowsPerToken = kMaxK + 1;

// Quantise one 16-element block held as two 16-byte words: returns the 8 code bytes
// (element 2j in the low nibble of byte j) and the E4M3 scale code.
__device__ __forceinline__ uint2 quant_block(uint4 a, uint4 b, float bmax, float g, uint32_t &scale) {
    // sf = (blockmax * g) / 6, each operation rounded once.
    const float sf = __fdiv_rn(__fmul_rn(bmax, g), 6.0f);
    const uint32_t s = cvt_e4m3x2(sf, 0.0f) & 0xffu;
    scale = s;
    const float sd = e4m3_value(s);
    if (sd == 0.0f) return make_uint2(0u, 0u);
    float r = __fdiv_rn(g, sd);
    if (isinf(r)) r = FLT_MAX;
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float p0, p1;
        mul2_rn(bf16_lo(w[q]), bf16_hi(w[q]), r, p0, p1);
        const uint32_t byte = cvt_e2m1x2(p0, p1);
        if (q < 4) lo |= byte << (8 * q);
        else hi |= byte << (8 * (q - 4));
    }
    return make_uint2(lo, hi);
}

template <int BPT, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB)
ep_dispatch_nvfp4_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int G, int R_max,
                         int early, int nfill, int fparts, int pad,
                         const int32_t *__restrict__ row_of, const int32_t *__restrict__ row_offsets,
                         const int32_t *__restrict__ src_info,
                         const int32_t *__restrict__ status, uint8_t *__restrict__ out_fp4,
                         uint8_t *__restrict__ out_scales, uint16_t *__restrict__ out_inv,
                         int32_t *__restrict__ scales_offsets, PadFill f0, PadFill f1, PadFill f2) {
    __shared__ int s_rows[kMaxRowsPerToken];
    __shared__ float s_red[32];
    // early == 0: wait for the previous kernel first; the token row, the row indices and the
    //             status word are then all requested before any is used.
    // early == 1: the kernel directly follows the layout of the same call (which let it launch
    //             only once every earlier kernel had completed), so x is read and quantised
    //             while the layout still runs, and the layout's outputs are read after the wait.
    if (!early) pdl_wait();
    if ((int)blockIdx.x < nfill) {   // leading CTAs of a padded layout: a group's padding rows
        if (!cta_status(status))
            fill_group_padding_call(blockIdx.x / fparts, blockIdx.x % fparts, fparts, pad, R_max,
                                    row_offsets, src_info, status, f0, f1, f2);
        return;
    }
    const int tid = threadIdx.x;
    const int t = blockIdx.x - nfill;
    const int nth = H / (16 * BPT);
    const bool active = tid < nth && t < T;
    uint4 v[2 * BPT];
    if (active) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H) + (size_t)tid * 2 * BPT;
#pragma unroll
        for (int i = 0; i < 2 * BPT; ++i) v[i] = ld_stream(src + i);
    } else {
#pragma unroll
        for (int i = 0; i < 2 * BPT; ++i) v[i] = make_uint4(0, 0, 0, 0);
    }
    int my_row = -1;
    if (!early && t < T) {
        if (tid < K) my_row = row_of[(size_t)t * K + tid];
        else if (tid == K && S) my_row = row_offsets[E] + t;
    }
    float bmax[BPT];
    float tmax = 0.0f;
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
        bmax[b] = absmax16(v[2 * b], v[2 * b + 1]);
        tmax = fmaxf(tmax, bmax[b]);
    }
    // Row maximum (exact) -> global scale g = 2688 / a (1 for an all-zero row).
    const float a = block_max_nonneg(tmax, s_red);
    float g = 1.0f;
    if (a != 0.0f) {
        g = __fdiv_rn(2688.0f, a);
        if (isinf(g)) g = FLT_MAX;
    }
    if (early) {
        pdl_wait();
        if (t < T) {
            if (tid < K) my_row = row_of[(size_t)t * K + tid];
            else if (tid == K && S) my_row = row_offsets[E] + t;
        }
    }
    if (cta_status(status)) return;
    if (t == 0)
        for (int gi = tid; gi <= G; gi += blockDim.x) scales_offsets[gi] = row_offsets[gi];
    if (t >= T) return;
    const int nrows = K + S;
    if (tid < nrows) s_rows[tid] = my_row;
    __syncthreads();
    if (!active) return;

    uint32_t codes[2 * BPT];
    uint32_t scl = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
        uint32_t s;
        uint2 c = quant_block(v[2 * b], v[2 * b + 1], bmax[b], g, s);
        codes[2 * b] = c.x;
        codes[2 * b + 1] = c.y;
        scl |= s << (8 * b);
    }
    uint16_t inv = 0;
    if (tid == 0) {
        __nv_bfloat16 h = __float2bfloat16_rn(__frcp_rn(g));
        inv = *reinterpret_cast<uint16_t *>(&h);
    }
    const size_t code_bytes = (size_t)H / 2, scale_bytes = (size_t)H / 16;
    for (int k = 0; k < nrows; ++k) {
        const int r = s_rows[k];
        if (!row_ok(r, R_max, status)) continue;
        uint8_t *dst = out_fp4 + (size_t)r * code_bytes + (size_t)tid * 8 * BPT;
        uint8_t *dsc = out_scales + (size_t)r * scale_bytes + (size_t)tid * BPT;
        if (BPT == 2) {
            st_stream(dst, make_uint4(codes[0], codes[1], codes[2], codes[3]));
            __stcs(reinterpret_cast<unsigned short *>(dsc), (unsigned short)scl);
        } else {
            __stcs(reinterpret_cast<uint2 *>(dst), make_uint2(codes[0], codes[1]));
            __stcs(reinterpret_cast<unsigned char *>(dsc), (unsigned char)scl);
        }
        if (tid == 0) out_inv[r] = inv;
    }
}

// BF16 dispatch: each CTA copies a run of up to kBf16Tokens consecutive tokens, as many as fill
// kBf16Chunks 16-byte chunks per thread (one token above H = 4096, two at H = 4096, four at
// H = 2048 and below), so a short row does not pay a CTA's start-up and row-index wait alone.  The
// run's rows are contiguous in x: chunk c of the run is chunk c mod H/8 of its token c div H/8.
// Every chunk a thread holds is requested before the first is stored, then stored to each of
// its token's K (+1) rows.
constexpr int kBf16Chunks = 4;   // 16-byte chunks of the run one thread holds at a time
constexpr int kBf16Tokens = 4;   // most tokens one CTA copies
constexpr int kBf16Threads = 256;

inline int bf16_tokens_per_cta(int H) {
    const int per = kBf16Chunks * kBf16Threads / (H / 8);
    return per < 1 ? 1 : (per > kBf16Tokens ? kBf16Tokens : per);
}

__global__ void __launch_bounds__(kBf16Threads)
ep_dispatch_bf16_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int R_max,
                        int nfill, int fparts, int pad, int tpc, const int32_t *__restrict__ row_of,
                        const int32_t *__restrict__ row_offsets, const int32_t *__restrict__ src_info,
                        const int32_t *__restrict__ status, uint16_t *__restrict__ out, PadFill f0) {
    __shared__ int s_rows[kBf16Tokens][kMaxRowsPerToken];
    pdl_wait();
    if (cta_status(status)) return;
    if ((int)blockIdx.x < nfill) {   // leading CTAs of a padded layout: a group's padding rows
        fill_group_padding_call(blockIdx.x / fparts, blockIdx.x % fparts, fparts, pad, R_max,
                                row_offsets, src_info, status, f0, PadFill{nullptr, 0, 0u},
                                PadFill{nullptr, 0, 0u});
        return;
    }
    const int tid = threadIdx.x;
    const int t0 = (blockIdx.x - nfill) * tpc;
    const int nt = min(tpc, T - t0);   // tokens of this run (the last run may be shorter)
    const int nrows = K + S;
    for (int j = tid; j < nt * nrows; j += blockDim.x) {
        const int g = j / nrows, k = j - g * nrows;
        s_rows[g][k] = k < K ? row_of[(size_t)(t0 + g) * K + k] : row_offsets[E] + t0 + g;
    }
    __syncthreads();
    const int nv = H / 8;          // 16-byte chunks of one token's row
    const int nrun = nt * nv;      // of the run
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t0 * H);
    for (int c0 = tid; c0 < nrun; c0 += kBf16Chunks * blockDim.x) {
        uint4 d[kBf16Chunks];
#pragma unroll
        for (int i = 0; i < kBf16Chunks; ++i) {
            const int c = c0 + i * blockDim.x;
            if (c < nrun) d[i] = ld_stream(src + c);
        }
#pragma unroll
        for (int i = 0; i < kBf16Chunks; ++i) {
            const int c = c0 + i * blockDim.x;
            if (c >= nrun) continue;
            const int g = c / nv, cc = c - g * nv;
            for (int k = 0; k < nrows; ++k) {
                const int r = s_rows[g][k];
                if (!row_ok(r, R_max, status)) continue;
                st_stream(out + (size_t)r * H + (size_t)cc * 8, d[i]);
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// FP8 dispatch: one CTA per token, one thread per 32 elements, so the four threads of a
// 128-element block share its maximum through two shuffles.  Per block, in fp32 with every
// operation rounded once: s = 448 / max|x| (1 for an all-zero block, FLT_MAX if it overflows),
// code = E4M3(x * s) by the hardware conversion, scale = 1 / s.  The row is read once.  Each
// lane's 32 code bytes are then exchanged within the warp (once per token) so that each of the
// warp's two 16-byte stores per destination row covers 512 contiguous bytes, and the same
// words are stored to each of the token's K (+1 shared) rows.
// ---------------------------------------------------------------------------------------
constexpr int kFp8Block = 128;

template <int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB)
ep_dispatch_fp8_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int R_max,
                       int nfill, int fparts, int pad, const int32_t *__restrict__ row_of,
                       const int32_t *__restrict__ row_offsets, const int32_t *__restrict__ src_info,
                       const int32_t *__restrict__ status, uint8_t *__restrict__ out_fp8,
                       float *__restrict__ out_scales, PadFill f0, PadFill f1) {
    __shared__ int s_rows[kMaxRowsPerToken];
    pdl_wait();
    if ((int)blockIdx.x < nfill) {   // leading CTAs of a padded layout: a group's padding rows
        if (!cta_status(status))
            fill_group_padding_call(blockIdx.x / fparts, blockIdx.x % fparts, fparts, pad, R_max,
                                    row_offsets, src_info, status, f0, f1, PadFill{nullptr, 0, 0u});
        return;
    }
    const int tid = threadIdx.x;
    const int t = blockIdx.x - nfill;
    const bool active = tid < H / 32;
    uint4 v[4];
    if (active) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H) + (size_t)tid * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ld_stream(src + i);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
    }
    int my_row = -1;
    if (tid < K) my_row = row_of[(size_t)t * K + tid];
    else if (tid == K && S) my_row = row_offsets[E] + t;
    if (cta_status(status)) return;
    if (tid < K + S) s_rows[tid] = my_row;
    float m = absmax_value(max_u16x2(max_u16x2(absmax_bits(v[0]), absmax_bits(v[1])),
                                     max_u16x2(absmax_bits(v[2]), absmax_bits(v[3]))));
    m = fmaxf(m, __shfl_xor_sync(kFullMask, m, 1));   // the four threads of the block
    m = fmaxf(m, __shfl_xor_sync(kFullMask, m, 2));
    __syncthreads();
    float sc = 1.0f;
    if (m != 0.0f) {
        sc = __fdiv_rn(448.0f, m);
        if (isinf(sc)) sc = FLT_MAX;
    }
    const float scale = __frcp_rn(sc);
    const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                            v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
    uint32_t c[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float p0, p1, p2, p3;
        mul2_rn(bf16_lo(w[2 * q]), bf16_hi(w[2 * q]), sc, p0, p1);
        mul2_rn(bf16_lo(w[2 * q + 1]), bf16_hi(w[2 * q + 1]), sc, p2, p3);
        c[q] = cvt_e4m3x2(p0, p1) | (cvt_e4m3x2(p2, p3) << 16);
    }
    // Lane l holds bytes [32l, 32l + 32) of its warp's 1 KiB of codes.  After the exchange, lane l
    // holds bytes [16l, 16l + 16) (w1) and [512 + 16l, 512 + 16l + 16) (w2): the 16-byte half
    // (l & 1) of lanes l/2 and 16 + l/2.
    const int lane = tid & 31;
    const bool odd = lane & 1;
    uint32_t w1[4], w2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a1 = __shfl_sync(kFullMask, c[i], lane >> 1);
        const uint32_t b1 = __shfl_sync(kFullMask, c[4 + i], lane >> 1);
        const uint32_t a2 = __shfl_sync(kFullMask, c[i], 16 + (lane >> 1));
        const uint32_t b2 = __shfl_sync(kFullMask, c[4 + i], 16 + (lane >> 1));
        w1[i] = odd ? b1 : a1;
        w2[i] = odd ? b2 : a2;
    }
    const int off1 = (tid - lane) * 32 + lane * 16;   // byte offsets in the row
    const int off2 = off1 + 512;
    const int nrows = K + S;
    const int nblk = H / kFp8Block;
    for (int k = 0; k < nrows; ++k) {
        const int r = s_rows[k];
        if (!row_ok(r, R_max, status)) continue;
        uint8_t *dst = out_fp8 + (size_t)r * H;
        if (off1 < H) st_stream(dst + off1, make_uint4(w1[0], w1[1], w1[2], w1[3]));
        if (off2 < H) st_stream(dst + off2, make_uint4(w2[0], w2[1], w2[2], w2[3]));
        if (active && (tid & 3) == 0) __stcs(out_scales + (size_t)r * nblk + (tid >> 2), scale);
    }
}

// ---------------------------------------------------------------------------------------
// Staged NVFP4 dispatch (H % 256 == 0, H <= 8192): as many CTAs as fit on the GPU (several per
// SM), each owning a contiguous range of tokens, with the per-token kernel's thread layout (one
// thread per 32 elements).  In rounds of up to kStageSlots tokens:
//   phase 1: quantise the round's tokens into shared memory (codes, block scales, inverse
//            scale per staging slot), the next token's row already loading into registers;
//   phase 2: copy every staged row to each of its K (+1) destination rows with bulk
//            asynchronous copies (shared -> global).
// With `early` set the kernel directly follows the layout kernel of the same call (which let it
// launch only once every earlier kernel had completed), so phase 1 of the first round runs
// before waiting for the layout and overlaps it; the layout's outputs are read after the wait.
// With `write_meta` set the layout kernel left src_info and expert_ids to this kernel: each lane
// that sends a row also writes that row's (token, slot) and expert, so the layout's critical
// path carries only row_of.  The metadata is written even when the status word stops the
// payload, as the layout would have written it.  For a padded layout (pad > 1), CTAs after the
// first tok_ctas write each group's padding rows as the dispatch of an all-zero token, fparts
// of them to a group.  The block scheduler places them once slots free up: on the SMs the
// layout leaves when it ends, and where token CTAs have finished.
// ---------------------------------------------------------------------------------------
constexpr int kStageSlots = 8;
constexpr int kStageMaxThreads = 256;

// (token, slot) and expert of row r of token t (slot K: the shared copy).
__device__ __forceinline__ void write_row_meta(int r, int t, int k, int K, int E,
                                               const int32_t *__restrict__ ids,
                                               int32_t *__restrict__ src_info,
                                               int32_t *__restrict__ expert_ids) {
    reinterpret_cast<int2 *>(src_info)[r] = make_int2(t, k);
    expert_ids[r] = k < K ? ids[(size_t)t * K + k] : E;
}

__global__ void __launch_bounds__(kStageMaxThreads, 4)
ep_dispatch_nvfp4_staged_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int G,
                                int R_max, int early, int write_meta, int pad, int fparts,
                                int tok_ctas, const int32_t *__restrict__ ids,
                                const int32_t *__restrict__ row_of,
                                const int32_t *__restrict__ row_offsets,
                                const int32_t *__restrict__ status, uint8_t *__restrict__ out_fp4,
                                uint8_t *__restrict__ out_scales, uint16_t *__restrict__ out_inv,
                                int32_t *__restrict__ scales_offsets, int32_t *__restrict__ src_info,
                                int32_t *__restrict__ expert_ids) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(16) float s_red[2][kStageMaxThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if ((int)blockIdx.x >= tok_ctas) {   // trailing CTAs of a padded layout: padding rows
        pdl_wait();
        if (!cta_status(status)) {      // codes 0, block scales 0, inverse scale bf16(1)
            const int q = blockIdx.x - tok_ctas;
            const PadFill f0{out_fp4, H / 2, 0u}, f1{out_scales, H / 16, 0u}, f2{out_inv, 2, 0x3F803F80u};
            fill_group_padding(q / fparts, q % fparts, fparts, pad, R_max, row_offsets, src_info, status,
                               f0, f1, f2);
        }
        return;
    }
    const int nwarps = blockDim.x >> 5;
    // The slots of absent warps (which no warp writes) hold 0, so every step reads all eight
    // with two 16-byte loads; the first step's barrier orders these stores before the reads.
    static_assert(kStageMaxThreads / 32 == 8, "two float4 per reduction step");
    if (tid < 16 && (tid & 7) >= nwarps) s_red[tid >> 3][tid & 7] = 0.0f;
    const int nth = H / 32;
    const bool active = tid < nth;
    const unsigned code_bytes = (unsigned)H / 2, scale_bytes = (unsigned)H / 16;
    const unsigned slot_bytes = code_bytes + scale_bytes;   // a multiple of 16
    unsigned char *s_stage = smem_raw;                    // [kStageSlots][slot_bytes]
    uint16_t *s_inv = reinterpret_cast<uint16_t *>(smem_raw + (size_t)kStageSlots * slot_bytes);
    // Token ranges of ceil(T / grid) or floor(T / grid) tokens: every SM gets the same number
    // of CTAs and each CTA within one token of the same work.
    const int tb = (int)((long long)blockIdx.x * T / tok_ctas);
    const int te = (int)((long long)(blockIdx.x + 1) * T / tok_ctas);
    bool waited = false;
    if (!early) {
        pdl_begin();
        waited = true;
    }
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint4 v[4], vn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = vn[i] = make_uint4(0, 0, 0, 0);
    if (active && tb < te) {
        const uint4 *src = xv + ((size_t)tb * H) / 8 + 4 * tid;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ld_stream(src + i);
    }
    for (int r0 = tb; r0 < te; r0 += kStageSlots) {
        const int r1 = min(te, r0 + kStageSlots);
        // ---- phase 1
        for (int t = r0; t < r1; ++t) {
            const int slot = t - r0, par = (t - tb) & 1;
            if (active && t + 1 < te) {
                const uint4 *src = xv + ((size_t)(t + 1) * H) / 8 + 4 * tid;
#pragma unroll
                for (int i = 0; i < 4; ++i) vn[i] = ld_stream(src + i);
            }
            const float b0 = absmax16(v[0], v[1]);
            const float b1 = absmax16(v[2], v[3]);
            const float m = warp_max_nonneg(fmaxf(b0, b1));
            if (lane == 0) s_red[par][warp] = m;
            __syncthreads();
            const float4 r0 = reinterpret_cast<const float4 *>(s_red[par])[0];
            const float4 r1 = reinterpret_cast<const float4 *>(s_red[par])[1];
            const float a = fmaxf(fmaxf(fmaxf(r0.x, r0.y), fmaxf(r0.z, r0.w)),
                                  fmaxf(fmaxf(r1.x, r1.y), fmaxf(r1.z, r1.w)));
            float g = 1.0f;
            if (a != 0.0f) {
                g = __fdiv_rn(2688.0f, a);
                if (isinf(g)) g = FLT_MAX;
            }
            unsigned char *slotp = s_stage + (size_t)slot * slot_bytes;
            if (active) {
                uint32_t s0, s1;
                const uint2 c0 = quant_block(v[0], v[1], b0, g, s0);
                const uint2 c1 = quant_block(v[2], v[3], b1, g, s1);
                *reinterpret_cast<uint4 *>(slotp + 16 * tid) = make_uint4(c0.x, c0.y, c1.x, c1.y);
                *reinterpret_cast<unsigned short *>(slotp + code_bytes + 2 * tid) =
                    (unsigned short)(s0 | (s1 << 8));
            }
            if (tid == 0) {
                __nv_bfloat16 h = __float2bfloat16_rn(__frcp_rn(g));
                s_inv[slot] = *reinterpret_cast<uint16_t *>(&h);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = vn[i];
        }
        fence_proxy_async_smem();   // the staged bytes become visible to the bulk-copy engine
        __syncthreads();
        if (!waited) {              // from here on the layout's outputs are needed
            pdl_begin();
            waited = true;
        }
        const int shared_base = S ? row_offsets[E] : 0;
        const int nrows = K + S;
        if (cta_status(status)) {         // constant per call: no copy was issued before
            if (write_meta)                // no payload, but every row's metadata
                for (int t = tb + warp; t < te; t += nwarps)
                    for (int k = lane; k < nrows; k += 32) {
                        const int r = k < K ? row_of[(size_t)t * K + k] : shared_base + t;
                        if (row_ok(r, R_max, status)) write_row_meta(r, t, k, K, E, ids, src_info, expert_ids);
                    }
            return;
        }
        if (blockIdx.x == 0 && r0 == tb)
            for (int gi = tid; gi <= G; gi += blockDim.x) scales_offsets[gi] = row_offsets[gi];
        // ---- phase 2
        for (int j = warp; j < r1 - r0; j += nwarps) {
            const int t = r0 + j;
            const unsigned char *slotp = s_stage + (size_t)j * slot_bytes;
            for (int k = lane; k < nrows; k += 32) {
                const int r = k < K ? row_of[(size_t)t * K + k] : shared_base + t;
                if (!row_ok(r, R_max, status)) continue;
                bulk_store(out_fp4 + (size_t)r * code_bytes, slotp, code_bytes);
                bulk_store(out_scales + (size_t)r * scale_bytes, slotp + code_bytes, scale_bytes);
                out_inv[r] = s_inv[j];
                if (write_meta) write_row_meta(r, t, k, K, E, ids, src_info, expert_ids);
            }
        }
        bulk_commit();
        bulk_wait_read_all();       // the staging slots may be overwritten after this
        __syncthreads();
    }
    if (!waited) pdl_begin();       // a CTA without tokens still orders itself after the layout
    bulk_wait_all();                // every copy of this thread has landed
}

// Grid of the staged dispatch (as many CTAs as fit on the SMs the layout leaves free), when
// each CTA's tokens fit two rounds of staging slots; -1 when the shape does not suit it.
inline int staged_grid(int T, int K, int H, int busy_sms) {
    if (T <= 0 || H % 256 != 0 || H / 32 > kStageMaxThreads) return -1;
    const int threads = max(H / 32, 32 * ((K + 1 + 31) / 32));
    if (threads > kStageMaxThreads) return -1;
    const size_t smem = (size_t)kStageSlots * ((size_t)H / 2 + H / 16) + 2 * kStageSlots;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(ep_dispatch_nvfp4_staged_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    int grid = resident_blocks(ep_dispatch_nvfp4_staged_kernel, threads, smem);
    if (grid <= 0) return -1;
    const int sms = device_sm_count();
    if (busy_sms > 0 && sms > busy_sms) grid = grid / sms * (sms - busy_sms);   // the SMs left free
    if (grid <= 0) return -1;
    if (grid > T) grid = T;
    const int tpc = (T + grid - 1) / grid;   // the most tokens a CTA gets
    // Beyond two rounds of staging slots per CTA the rounds alternate reading and writing inside
    // each CTA, and the per-token kernel (in early mode) is faster: on GB300, 54 tokens per CTA
    // (32,768 tokens at H = 7168) took 304 us staged against 274 us per token, while 16 tokens
    // per CTA (16,384 at H = 4096) took 41 us staged against 48 us.
    if (tpc > 2 * kStageSlots) return -1;
    return grid;
}

// The staged dispatch on `grid` CTAs (from staged_grid); with write_meta it also writes the
// layout's src_info and expert_ids (the layout kernel before it left them out), and for a padded
// layout it writes the padding rows.
inline int launch_nvfp4_staged(int grid, const uint16_t *x, int H, const int32_t *ids,
                               const ep_layout_t *L, uint8_t *out_fp4, uint8_t *out_scales,
                               uint16_t *out_inv, int32_t *scales_offsets, int early, int write_meta,
                               cudaStream_t st) {
    const int threads = max(H / 32, 32 * ((L->K + 1 + 31) / 32));
    const size_t smem = (size_t)kStageSlots * ((size_t)H / 2 + H / 16) + 2 * kStageSlots;
    const int G = L->E + L->fused_shared;
    const int R_max = layout_rows(L);
    const int pad = layout_padded(L) ? L->pad_multiple : 1;
    const int nfill = fill_ctas(L, threads);   // trailing CTAs for the padding rows
    return launch_pdl(ep_dispatch_nvfp4_staged_kernel, dim3(grid + nfill), dim3(threads), smem, st, x,
                      L->T, H, L->K, L->E, L->fused_shared, G, R_max, early, write_meta, pad,
                      fill_parts(L, threads), grid, ids,
                      (const int32_t *)L->row_of, (const int32_t *)L->row_offsets,
                      (const int32_t *)L->status, out_fp4, out_scales, out_inv, scales_offsets,
                      L->src_info, L->expert_ids);
}

__global__ void ep_cvt_kernel(const float *__restrict__ in, uint8_t *__restrict__ codes, long n, int e4m3) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const float v = in[i];
        codes[i] = (uint8_t)(e4m3 ? (cvt_e4m3x2(v, 0.0f) & 0xffu) : (cvt_e2m1x2(v, 0.0f) & 0xfu));
    }
}

inline int launch_cvt(const float *in, uint8_t *codes, long n, void *stream, int e4m3) {
    if (n < 0 || (n > 0 && (!in || !codes))) return EP_ERR_INVALID_ARG;
    if (n == 0) return EP_OK;
    long blocks = (n + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    ep_cvt_kernel<<<(int)blocks, 256, 0, as_stream(stream)>>>(in, codes, n, e4m3);
    return launch_result();
}

}  // namespace
}  // namespace ep

using namespace ep;

namespace ep {
namespace {

int launch_nvfp4(const uint16_t *input_tokens, int H, const ep_layout_t *L, uint8_t *out_fp4,
                 uint8_t *out_scales, uint16_t *out_rowwise_inv_scale, int32_t *scales_offsets,
                 int early, cudaStream_t st) {
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    const int bpt = (H % 32 == 0) ? 2 : 1;
    const int nth = H / (16 * bpt);
    if (nth > 1024) return EP_ERR_INVALID_ARG;
    if ((L->T > 0 && (!input_tokens || !out_fp4 || !out_scales || !out_rowwise_inv_scale)) ||
        !scales_offsets)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {input_tokens, out_fp4, out_scales, out_rowwise_inv_scale, scales_offsets};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    // enough threads to load the K (+1 shared) row indices of the token
    const int threads = max((nth + 31) / 32 * 32, (L->K + 1 + 31) / 32 * 32);
    // padding rows (padded layouts; the fused call's layout is never padded): codes 0, block
    // scales 0, inverse global scale bf16(1/1) = 0x3F80 -- the dispatch of an all-zero token
    const int nfill = early ? 0 : fill_ctas(L, threads);
    const int fparts = fill_parts(L, threads);
    const PadFill f0{out_fp4, H / 2, 0u}, f1{out_scales, H / 16, 0u},
        f2{out_rowwise_inv_scale, 2, 0x3F803F80u};
    const int grid = (L->T > 0 ? L->T : 1) + nfill;
    const int G = L->E + L->fused_shared;
    const int R_max = layout_rows(L);
    const int32_t *row_of = L->row_of, *row_offsets = L->row_offsets, *status = L->status;
    const int32_t *src_info = L->src_info;
#define EP_NVFP4_LAUNCH(BPT, MAXT, MINB)                                                        \
    return launch_pdl(ep_dispatch_nvfp4_kernel<BPT, MAXT, MINB>, dim3(grid), dim3(threads), 0, st, \
                      input_tokens, L->T, H, L->K, L->E, L->fused_shared, G, R_max, early, nfill, \
                      fparts, L->pad_multiple, row_of, row_offsets, src_info, status, out_fp4,   \
                      out_scales, out_rowwise_inv_scale, scales_offsets, f0, f1, f2)
    // Up to 256 threads (H <= 8192): 5 such CTAs per SM without spilling.
    if (bpt == 2 && threads <= 256) EP_NVFP4_LAUNCH(2, 256, 5);
    if (bpt == 2) EP_NVFP4_LAUNCH(2, 1024, 1);
    if (threads <= 256) EP_NVFP4_LAUNCH(1, 256, 5);
    EP_NVFP4_LAUNCH(1, 1024, 1);
#undef EP_NVFP4_LAUNCH
}

}  // namespace

}  // namespace ep

extern "C" int ep_dispatch_nvfp4(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                                 uint8_t *out_fp4, uint8_t *out_scales, uint16_t *out_rowwise_inv_scale,
                                 int32_t *scales_offsets, void *stream) {
    EP_NVTX_RANGE("ep_dispatch_nvfp4");
    return launch_nvfp4(input_tokens, hidden_size, L, out_fp4, out_scales, out_rowwise_inv_scale,
                        scales_offsets, 0, as_stream(stream));
}

extern "C" int ep_dispatch_layout_nvfp4(const int32_t *topk_ids, int T, int K, int n_experts,
                                        int n_parts, int capacity, int fused_shared,
                                        const uint16_t *input_tokens, int hidden_size,
                                        ep_layout_t *L, uint8_t *out_fp4, uint8_t *out_scales,
                                        uint16_t *out_rowwise_inv_scale, int32_t *scales_offsets,
                                        void *stream) {
    EP_NVTX_RANGE("ep_dispatch_layout_nvfp4");
    const int H = hidden_size;
    if (!hidden_ok(H) || H / 16 > 1024) return EP_ERR_INVALID_ARG;
    if ((T > 0 && (!input_tokens || !out_fp4 || !out_scales || !out_rowwise_inv_scale)) ||
        !scales_offsets)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {input_tokens, out_fp4, out_scales, out_rowwise_inv_scale, scales_offsets};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    // The dispatch kernel directly follows the layout kernel, which lets it launch only once
    // every earlier kernel of the stream has completed, so its CTAs read and quantise their
    // tokens while the layout is still running and wait for the layout only before storing.
    // When the layout takes the single-cluster kernel and the staged dispatch follows it, the
    // dispatch can write src_info and expert_ids itself, which takes them off the layout's
    // critical path.  That pays where the token rows are short for their routed slots
    // (2H <= 512 K bytes), so the layout, not the read of x, decides when the stores can start:
    // on GB300 the Qwen3-like step (H = 2048, K = 8) got 1.0 us faster (78.9 -> 78.0 us), while
    // the DSv3-like (H = 7168, K = 8) and Mixtral-like (H = 4096, K = 2) steps, whose dispatch
    // is bound by HBM, got 0.8 us slower from the extra scattered stores.
    const int planned_sms = layout_cluster_plan(T, K, n_experts, n_parts);
    const int grid = staged_grid(T, K, H, planned_sms);
    const int meta_in_dispatch = grid > 0 && planned_sms > 0 && 2 * H <= 512 * K;
    int layout_sms = 0;
    int rc = launch_layout(topk_ids, T, K, n_experts, n_parts, capacity, fused_shared, 1, 0, L, st,
                           &layout_sms, meta_in_dispatch ? 0 : 1);
    if (rc != EP_OK) return rc;
    if (grid > 0)
        return launch_nvfp4_staged(grid, input_tokens, H, topk_ids, L, out_fp4, out_scales,
                                   out_rowwise_inv_scale, scales_offsets, 1,
                                   meta_in_dispatch && layout_sms > 0, st);
    return launch_nvfp4(input_tokens, H, L, out_fp4, out_scales, out_rowwise_inv_scale,
                        scales_offsets, 1, st);
}

extern "C" int ep_dispatch_layout_padded_nvfp4(const int32_t *topk_ids, int T, int K, int n_experts,
                                               int n_parts, int capacity, int fused_shared,
                                               int pad_multiple, int num_permuted_tokens,
                                               const uint16_t *input_tokens, int hidden_size,
                                               ep_layout_t *L, uint8_t *out_fp4, uint8_t *out_scales,
                                               uint16_t *out_rowwise_inv_scale, int32_t *scales_offsets,
                                               void *stream) {
    EP_NVTX_RANGE("ep_dispatch_layout_padded_nvfp4");
    const int H = hidden_size;
    if (!hidden_ok(H) || H / 16 > 1024) return EP_ERR_INVALID_ARG;
    if ((T > 0 && (!input_tokens || !out_fp4 || !out_scales || !out_rowwise_inv_scale)) ||
        !scales_offsets)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {input_tokens, out_fp4, out_scales, out_rowwise_inv_scale, scales_offsets};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    // As in ep_dispatch_layout_nvfp4 the staged dispatch quantises while the layout runs; the
    // layout writes every row's metadata (the padding rows' too), and the dispatch writes the
    // padding rows' payload.  Without the staged kernel, the per-token kernel runs after the
    // layout with its leading padding CTAs, as ep_dispatch_nvfp4 would.
    const int grid = staged_grid(T, K, H, layout_cluster_plan(T, K, n_experts, n_parts));
    int layout_sms = 0;
    int rc = launch_layout(topk_ids, T, K, n_experts, n_parts, capacity, fused_shared, pad_multiple,
                           num_permuted_tokens, L, st, &layout_sms, 1);
    if (rc != EP_OK) return rc;
    if (grid > 0)
        return launch_nvfp4_staged(grid, input_tokens, H, topk_ids, L, out_fp4, out_scales,
                                   out_rowwise_inv_scale, scales_offsets, 1, 0, st);
    return launch_nvfp4(input_tokens, H, L, out_fp4, out_scales, out_rowwise_inv_scale,
                        scales_offsets, 0, st);
}

extern "C" int ep_dispatch_bf16(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                                uint16_t *out, void *stream) {
    EP_NVTX_RANGE("ep_dispatch_bf16");
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!input_tokens || !out)) return EP_ERR_INVALID_ARG;
    if ((input_tokens && !aligned16(input_tokens)) || (out && !aligned16(out))) return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    const int nfill = fill_ctas(L, kBf16Threads);   // padding rows: zeros
    const int tpc = bf16_tokens_per_cta(H);
    return launch_pdl(ep_dispatch_bf16_kernel, dim3((L->T + tpc - 1) / tpc + nfill), dim3(kBf16Threads), 0,
                      as_stream(stream), input_tokens, L->T, H, L->K, L->E, L->fused_shared,
                      layout_rows(L), nfill, fill_parts(L, kBf16Threads), L->pad_multiple, tpc,
                      (const int32_t *)L->row_of, (const int32_t *)L->row_offsets,
                      (const int32_t *)L->src_info, (const int32_t *)L->status, out,
                      PadFill{out, 2 * H, 0u});
}

extern "C" int ep_dispatch_fp8(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                               uint8_t *out_fp8, float *out_scales, void *stream) {
    EP_NVTX_RANGE("ep_dispatch_fp8");
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H) || H % kFp8Block != 0) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!input_tokens || !out_fp8 || !out_scales)) return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {input_tokens, out_fp8, out_scales};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    cudaStream_t st = as_stream(stream);
    const int threads = max(H / 32, 32 * ((L->K + 1 + 31) / 32));   // H % 128 == 0: whole warps
    const int R_max = layout_rows(L);
    const int nfill = fill_ctas(L, threads);
    const int fparts = fill_parts(L, threads);
    // padding rows: codes 0 and the scale of an all-zero block, 1.0f
    const PadFill f0{out_fp8, H, 0u}, f1{out_scales, 4 * (H / kFp8Block), 0x3F800000u};
    if (threads <= 256)
        return launch_pdl(ep_dispatch_fp8_kernel<256, 5>, dim3(L->T + nfill), dim3(threads), 0, st,
                          input_tokens, L->T, H, L->K, L->E, L->fused_shared, R_max, nfill, fparts,
                          L->pad_multiple, (const int32_t *)L->row_of, (const int32_t *)L->row_offsets,
                          (const int32_t *)L->src_info, (const int32_t *)L->status, out_fp8,
                          out_scales, f0, f1);
    return launch_pdl(ep_dispatch_fp8_kernel<1024, 1>, dim3(L->T + nfill), dim3(threads), 0, st,
                      input_tokens, L->T, H, L->K, L->E, L->fused_shared, R_max, nfill, fparts,
                      L->pad_multiple, (const int32_t *)L->row_of, (const int32_t *)L->row_offsets,
                      (const int32_t *)L->src_info, (const int32_t *)L->status, out_fp8, out_scales,
                      f0, f1);
}

extern "C" int ep_cvt_e2m1(const float *in, uint8_t *codes, long n, void *stream) {
    return launch_cvt(in, codes, n, stream, 0);
}

extern "C" int ep_cvt_e4m3(const float *in, uint8_t *codes, long n, void *stream) {
    return launch_cvt(in, codes, n, stream, 1);
}
