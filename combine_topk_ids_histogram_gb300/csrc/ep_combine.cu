// ep_combine.cu -- gather-reduce of expert rows back into token order (combine, and the
// dispatch backward pass with unit weights) and the combine backward pass.
//
// Combine follows the fused_a2a page (hybrid_ep_combine / HybridEPCombine.forward: expert
// outputs brought back to one row per input token, in input order) with the fp32 router
// probabilities as weights (token_dispatcher page, TokenDispatcherConfig.moe_router_dtype).
// Its backward follows HybridEPCombine.backward (the output gradient dispatched again through
// the saved layout) and the dispatch backward follows HybridEPDispatch.backward (row
// gradients combined back per token).
//
// Combine runs as many CTAs as fit on the GPU at once, each looping over tokens.  A thread owns
// column slices of the token, two adjacent 16-byte words (16 elements) at a time for K <= 8
// (one word for wider K, whose rows would not fit in registers); for a slice it issues the
// loads of all of the token's K (+1 shared) rows before accumulating, so up to 2(K+1)
// independent 16-byte loads per thread are in flight, and it already holds the next token's
// row indices.  With two words per thread a 128-thread CTA reads 4 KB of each row per step:
// on GB300 that beat 2 KB steps by 3.6% (94.5 against 98.0 us for the DSv3-shaped combine).  The
// accumulation is fp32 with one fused multiply-add per term, in ascending slot order with the
// shared row last, which makes the result deterministic.  The backward kernel keeps one CTA
// per token.
#include "ep_common.cuh"
#include "ep_host.h"
#include "ep_padding.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 128;

// Persistent: a CTA loops over tokens t = blockIdx.x, blockIdx.x + gridDim.x, ...  While it
// streams token t's rows it already holds the row indices and weights of its next token, so a
// token starts with its row loads, never with a metadata round trip.
// Resident CTAs per SM the register budget is sized for.
template <int KMAX>
constexpr int combine_min_blocks() { return KMAX <= 2 ? 8 : KMAX <= 4 ? 6 : KMAX <= 8 ? 4 : 1; }

template <int KMAX, bool WEIGHTED>
__global__ void __launch_bounds__(kCombineThreads, combine_min_blocks<KMAX>())
ep_combine_kernel(const uint16_t *__restrict__ y, const float *__restrict__ probs, int T, int H, int K,
                  int E, int S, int R_max, const int32_t *__restrict__ row_of,
                  const int32_t *__restrict__ row_offsets, const int32_t *__restrict__ status,
                  uint16_t *__restrict__ out) {
    __shared__ int s_rows[2][KMAX + 1];
    __shared__ float s_w[2][KMAX + 1];
    pdl_begin();
    if (cta_status(status)) return;
    const int tid = threadIdx.x;
    const int shared_base = S ? row_offsets[E] : 0;

    // Slot `tid` (<= KMAX) of token tt: its row (or -1) and weight.
    auto meta = [&](int tt, int &r, float &w) {
        r = -1;
        w = 1.0f;
        if (tid > KMAX || tt >= T) return;
        if (tid < K) {
            r = row_of[(size_t)tt * K + tid];
            if (WEIGHTED) w = probs[(size_t)tt * K + tid];
        } else if (tid == K && S) {
            r = shared_base + tt;
        }
        if (!row_ok(r, R_max, status)) r = -1;
    };

    int t = blockIdx.x;
    {
        int r;
        float w;
        meta(t, r, w);
        if (tid <= KMAX) {
            s_rows[0][tid] = r;
            s_w[0][tid] = w;
        }
    }
    __syncthreads();
    const int nv = H / 8;
    for (int buf = 0; t < T; t += gridDim.x, buf ^= 1) {
        int r_next;
        float w_next;
        meta(t + gridDim.x, r_next, w_next);     // in flight while this token streams
        // Row indices and weights are re-read from shared memory (broadcasts) for every slice
        // rather than held in registers, which keeps enough CTAs resident per SM.
        const int *rows = s_rows[buf];
        const float *w = s_w[buf];
        // VW adjacent words per step (H % 16 == 0, so nv is even)
        constexpr int VW = KMAX <= 8 ? 2 : 1;
        for (int c = VW * tid; c < nv; c += VW * blockDim.x) {
            uint4 d[VW][KMAX + 1];
#pragma unroll
            for (int k = 0; k <= KMAX; ++k) {
                const int r = rows[k];
                if (r >= 0) {
#pragma unroll
                    for (int j = 0; j < VW; ++j) d[j][k] = ld_stream(y + (size_t)r * H + (size_t)(c + j) * 8);
                }
            }
            float acc[VW][8];
#pragma unroll
            for (int j = 0; j < VW; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
#pragma unroll
            for (int k = 0; k <= KMAX; ++k) {
                if (rows[k] >= 0) {
                    const float wk = w[k];
#pragma unroll
                    for (int j = 0; j < VW; ++j) {
                        float f[8];
                        unpack8(d[j][k], f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(wk, f[i], acc[j][i]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < VW; ++j) st_stream(out + (size_t)t * H + (size_t)(c + j) * 8, pack8(acc[j]));
        }
        if (tid <= KMAX) {
            s_rows[buf ^ 1][tid] = r_next;
            s_w[buf ^ 1][tid] = w_next;
        }
        __syncthreads();
    }
}

template <int KMAX>
__global__ void __launch_bounds__(kCombineThreads)
ep_combine_bwd_kernel(const uint16_t *__restrict__ g, const uint16_t *__restrict__ y,
                      const float *__restrict__ probs, int T, int H, int K, int E, int S, int R_max,
                      int nfill, int fparts, int pad, const int32_t *__restrict__ row_of,
                      const int32_t *__restrict__ row_offsets, const int32_t *__restrict__ src_info,
                      const int32_t *__restrict__ status, uint16_t *__restrict__ grad_y,
                      float *__restrict__ grad_p) {
    __shared__ int s_rows[KMAX];
    __shared__ float s_p[KMAX];
    __shared__ float s_red[kCombineThreads / 32][KMAX];
    pdl_wait();
    if (cta_status(status)) return;
    if ((int)blockIdx.x < nfill) {   // leading CTAs of a padded layout: zero gradient rows
        fill_group_padding(blockIdx.x / fparts, blockIdx.x % fparts, fparts, pad, R_max, row_offsets,
                           src_info, status, PadFill{grad_y, 2 * H, 0u}, PadFill{nullptr, 0, 0u},
                           PadFill{nullptr, 0, 0u});
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = blockIdx.x - nfill;
    if (tid < KMAX) {
        int r = -1;
        float p = 0.0f;
        if (tid < K) {
            r = row_of[(size_t)t * K + tid];
            p = probs[(size_t)t * K + tid];
        }
        s_rows[tid] = row_ok(r, R_max, status) ? r : -1;
        s_p[tid] = p;
    }
    __syncthreads();
    int rows[KMAX];
    float p[KMAX], dot[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        rows[k] = s_rows[k];
        p[k] = s_p[k];
        dot[k] = 0.0f;
    }
    int shared_row = S ? row_offsets[E] + t : -1;
    if (S && !row_ok(shared_row, R_max, status)) shared_row = -1;
    const int nv = H / 8;
    for (int c = tid; c < nv; c += blockDim.x) {
        const uint4 gv = ld_stream(g + (size_t)t * H + (size_t)c * 8);
        uint4 d[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            if (rows[k] >= 0) d[k] = ld_stream(y + (size_t)rows[k] * H + (size_t)c * 8);
        float gf[8];
        unpack8(gv, gf);
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (rows[k] >= 0) {
                float f[8], o[8];
                unpack8(d[k], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    dot[k] = fmaf(gf[i], f[i], dot[k]);
                    o[i] = __fmul_rn(p[k], gf[i]);
                }
                st_stream(grad_y + (size_t)rows[k] * H + (size_t)c * 8, pack8(o));
            }
        }
        if (shared_row >= 0) st_stream(grad_y + (size_t)shared_row * H + (size_t)c * 8, gv);
    }
    // grad_p[t, k]: fixed-order tree (warp shuffle, then warps in order).
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        float v = dot[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
        if (lane == 0) s_red[warp][k] = v;
    }
    __syncthreads();
    if (tid < K) {
        float s = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += s_red[w][tid];
        grad_p[(size_t)t * K + tid] = s_rows[tid] >= 0 ? s : 0.0f;
    }
}

template <int KM, bool WEIGHTED>
int launch_combine_k(const uint16_t *y, const float *probs, int H, const ep_layout_t *L, int R_max,
                     uint16_t *out, cudaStream_t st) {
    auto kern = ep_combine_kernel<KM, WEIGHTED>;
    int grid = resident_blocks(kern, kCombineThreads, 0);
    if (grid <= 0 || grid > L->T) grid = L->T;
    return launch_pdl(kern, dim3(grid), dim3(kCombineThreads), 0, st, y, probs, L->T, H, L->K, L->E,
                      L->fused_shared, R_max, (const int32_t *)L->row_of,
                      (const int32_t *)L->row_offsets, (const int32_t *)L->status, out);
}

template <bool WEIGHTED>
int launch_combine(const uint16_t *y, const float *probs, int H, const ep_layout_t *L,
                   uint16_t *out, cudaStream_t st) {
    const int K = L->K;
    const int R_max = layout_rows(L);
    if (K <= 2) return launch_combine_k<2, WEIGHTED>(y, probs, H, L, R_max, out, st);
    if (K <= 4) return launch_combine_k<4, WEIGHTED>(y, probs, H, L, R_max, out, st);
    if (K <= 8) return launch_combine_k<8, WEIGHTED>(y, probs, H, L, R_max, out, st);
    if (K <= 16) return launch_combine_k<16, WEIGHTED>(y, probs, H, L, R_max, out, st);
    return launch_combine_k<32, WEIGHTED>(y, probs, H, L, R_max, out, st);
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" int ep_combine(const uint16_t *expert_out, const float *probs, int hidden_size,
                          const ep_layout_t *L, uint16_t *out, void *stream) {
    EP_NVTX_RANGE("ep_combine");
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!expert_out || !probs || !out)) return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {expert_out, probs, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    return launch_combine<true>(expert_out, probs, H, L, out, as_stream(stream));
}

extern "C" int ep_dispatch_bwd(const uint16_t *grad_rows, int hidden_size, const ep_layout_t *L,
                               uint16_t *grad_input, void *stream) {
    EP_NVTX_RANGE("ep_dispatch_bwd");
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!grad_rows || !grad_input)) return EP_ERR_INVALID_ARG;
    if ((grad_rows && !aligned16(grad_rows)) || (grad_input && !aligned16(grad_input)))
        return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    return launch_combine<false>(grad_rows, nullptr, H, L, grad_input, as_stream(stream));
}

extern "C" int ep_combine_bwd(const uint16_t *grad_out, const uint16_t *expert_out, const float *probs,
                              int hidden_size, const ep_layout_t *L, uint16_t *grad_expert_out,
                              float *grad_probs, void *stream) {
    EP_NVTX_RANGE("ep_combine_bwd");
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!grad_out || !expert_out || !probs || !grad_expert_out || !grad_probs))
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {grad_out, expert_out, probs, grad_expert_out, grad_probs};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    cudaStream_t st = as_stream(stream);
    const int K = L->K;
    const int R_max = layout_rows(L);
    const int nfill = fill_ctas(L, kCombineThreads);   // padding rows get a zero gradient
    const int fparts = fill_parts(L, kCombineThreads);
#define EP_BWD_CASE(KM)                                                                        \
    return launch_pdl(ep_combine_bwd_kernel<KM>, dim3(L->T + nfill), dim3(kCombineThreads), 0, st, \
                      grad_out, expert_out, probs, L->T, H, K, L->E, L->fused_shared, R_max,   \
                      nfill, fparts, L->pad_multiple, (const int32_t *)L->row_of,              \
                      (const int32_t *)L->row_offsets, (const int32_t *)L->src_info,           \
                      (const int32_t *)L->status, grad_expert_out, grad_probs)
    if (K <= 2) EP_BWD_CASE(2);
    if (K <= 4) EP_BWD_CASE(4);
    if (K <= 8) EP_BWD_CASE(8);
    if (K <= 16) EP_BWD_CASE(16);
    EP_BWD_CASE(32);
#undef EP_BWD_CASE
}
