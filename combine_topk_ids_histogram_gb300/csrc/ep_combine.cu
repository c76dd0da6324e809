// ep_combine.cu -- gather-reduce of expert rows back into token order (combine, and the
// dispatch backward pass with unit weights) and the combine backward pass.
//
// Combine follows the fused_a2a page (hybrid_ep_combine / HybridEPCombine.forward: expert
// outputs back to the original token order, [tokens, hidden]) with the fp32 router
// probabilities as weights (token_dispatcher page, TokenDispatcherConfig.moe_router_dtype).
// Its backward follows HybridEPCombine.backward (the output gradient dispatched again through
// the saved layout) and the dispatch backward follows HybridEPDispatch.backward (row
// gradients combined back per token).
//
// One CTA per token.  Each thread owns 8-element (16-byte) column slices; for a slice it
// issues the loads of all of the token's K (+1 shared) rows before accumulating, so up to
// K+1 independent 16-byte loads per thread are in flight.  Accumulation is fp32 with one
// fused multiply-add per term, in ascending slot order with the shared row last, which makes
// the result deterministic.
#include "ep_common.cuh"
#include "ep_host.h"

namespace ep {
namespace {

constexpr int kCombineThreads = 128;

template <int KMAX, bool WEIGHTED>
__global__ void __launch_bounds__(kCombineThreads)
ep_combine_kernel(const uint16_t *__restrict__ y, const float *__restrict__ probs, int T, int H, int K,
                  int E, int S, int R_max, const int32_t *__restrict__ row_of,
                  const int32_t *__restrict__ row_offsets, const int32_t *__restrict__ status,
                  uint16_t *__restrict__ out) {
    __shared__ int s_rows[KMAX + 1];
    __shared__ float s_w[KMAX + 1];
    if (load_status(status)) return;
    const int tid = threadIdx.x;
    const int t = blockIdx.x;
    if (tid <= KMAX) {
        int r = -1;
        float w = 1.0f;
        if (tid < K) {
            r = row_of[(size_t)t * K + tid];
            if (WEIGHTED) w = probs[(size_t)t * K + tid];
        } else if (tid == K && S) {
            r = row_offsets[E] + t;
        }
        s_rows[tid] = (r < R_max) ? r : -1;
        s_w[tid] = w;
    }
    __syncthreads();
    int rows[KMAX + 1];
    float w[KMAX + 1];
#pragma unroll
    for (int k = 0; k <= KMAX; ++k) {
        rows[k] = s_rows[k];
        w[k] = s_w[k];
    }
    const int nv = H / 8;
    for (int c = tid; c < nv; c += blockDim.x) {
        uint4 d[KMAX + 1];
#pragma unroll
        for (int k = 0; k <= KMAX; ++k)
            if (rows[k] >= 0) d[k] = ld_stream(y + (size_t)rows[k] * H + (size_t)c * 8);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int k = 0; k <= KMAX; ++k) {
            if (rows[k] >= 0) {
                float f[8];
                unpack8(d[k], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[k], f[i], acc[i]);
            }
        }
        st_stream(out + (size_t)t * H + (size_t)c * 8, pack8(acc));
    }
}

template <int KMAX>
__global__ void __launch_bounds__(kCombineThreads)
ep_combine_bwd_kernel(const uint16_t *__restrict__ g, const uint16_t *__restrict__ y,
                      const float *__restrict__ probs, int T, int H, int K, int E, int S, int R_max,
                      const int32_t *__restrict__ row_of, const int32_t *__restrict__ row_offsets,
                      const int32_t *__restrict__ status, uint16_t *__restrict__ grad_y,
                      float *__restrict__ grad_p) {
    __shared__ int s_rows[KMAX];
    __shared__ float s_p[KMAX];
    __shared__ float s_red[kCombineThreads / 32][KMAX];
    if (load_status(status)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = blockIdx.x;
    if (tid < KMAX) {
        int r = -1;
        float p = 0.0f;
        if (tid < K) {
            r = row_of[(size_t)t * K + tid];
            p = probs[(size_t)t * K + tid];
        }
        s_rows[tid] = (r < R_max) ? r : -1;
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
    if (shared_row >= R_max) shared_row = -1;
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

template <bool WEIGHTED>
int launch_combine(const uint16_t *y, const float *probs, int H, const ep_layout_t *L,
                   uint16_t *out, cudaStream_t st) {
    const int K = L->K;
    const int R_max = (int)rows_max(L->T, L->K, L->fused_shared);
    const int threads = kCombineThreads;
    const dim3 grid(L->T);
#define EP_COMBINE_CASE(KM)                                                                    \
    ep_combine_kernel<KM, WEIGHTED><<<grid, threads, 0, st>>>(y, probs, L->T, H, K, L->E,      \
                                                             L->fused_shared, R_max, L->row_of, \
                                                             L->row_offsets, L->status, out)
    if (K <= 2) EP_COMBINE_CASE(2);
    else if (K <= 4) EP_COMBINE_CASE(4);
    else if (K <= 8) EP_COMBINE_CASE(8);
    else if (K <= 16) EP_COMBINE_CASE(16);
    else EP_COMBINE_CASE(32);
#undef EP_COMBINE_CASE
    return launch_result();
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" int ep_combine(const uint16_t *expert_out, const float *probs, int hidden_size,
                          const ep_layout_t *L, uint16_t *out, void *stream) {
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
    const int R_max = (int)rows_max(L->T, L->K, L->fused_shared);
#define EP_BWD_CASE(KM)                                                                        \
    ep_combine_bwd_kernel<KM><<<L->T, kCombineThreads, 0, st>>>(                               \
        grad_out, expert_out, probs, L->T, H, K, L->E, L->fused_shared, R_max, L->row_of,      \
        L->row_offsets, L->status, grad_expert_out, grad_probs)
    if (K <= 2) EP_BWD_CASE(2);
    else if (K <= 4) EP_BWD_CASE(4);
    else if (K <= 8) EP_BWD_CASE(8);
    else if (K <= 16) EP_BWD_CASE(16);
    else EP_BWD_CASE(32);
#undef EP_BWD_CASE
    return launch_result();
}
