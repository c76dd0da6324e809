// ep_dispatch.cu -- permute-scatter of token rows into the expert-major layout, as NVFP4 with
// a per-token global scale (Mojo EP dispatch page, DistributedEPDispatchBlockScaledNVDynGlobal
// Scales.execute) or as plain bf16 (fused_a2a page, HybridEPDispatch.forward).
//
// NVFP4 kernel: one CTA per token.  Each thread owns a contiguous chunk of BPT 16-element
// blocks (BPT = 2 -> 32 elements: 4 x 16-byte loads in, one 16-byte code store and one 2-byte
// scale store per destination row).  The token row is read from HBM exactly once and stays in
// registers: the row maximum is a block-wide reduction, the block maxima are per thread, the
// E4M3 and E2M1 encodings are single hardware conversions, and the same bytes are then
// stored to each of the token's K (+1 shared) rows.
#include "ep_common.cuh"
#include "ep_host.h"

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
        const uint32_t byte = cvt_e2m1x2(__fmul_rn(bf16_lo(w[q]), r), __fmul_rn(bf16_hi(w[q]), r));
        if (q < 4) lo |= byte << (8 * q);
        else hi |= byte << (8 * (q - 4));
    }
    return make_uint2(lo, hi);
}

__device__ __forceinline__ float absmax8(uint4 v) {
    float f[8];
    unpack8(v, f);
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return m;
}

template <int BPT, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB)
ep_dispatch_nvfp4_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int G, int R_max,
                         int early,
                         const int32_t *__restrict__ row_of, const int32_t *__restrict__ row_offsets,
                         const int32_t *__restrict__ status, uint8_t *__restrict__ out_fp4,
                         uint8_t *__restrict__ out_scales, uint16_t *__restrict__ out_inv,
                         int32_t *__restrict__ scales_offsets) {
    __shared__ int s_rows[kMaxRowsPerToken];
    __shared__ float s_red[32];
    // early == 0: wait for the previous kernel first; the token row, the row indices and the
    //             status word are then all requested before any is used.
    // early == 1: the kernel directly follows the layout of the same call (which let it launch
    //             only once every earlier kernel had completed), so x is read and quantised
    //             while the layout still runs, and the layout's outputs are read after the wait.
    if (!early) pdl_begin();
    const int tid = threadIdx.x;
    const int t = blockIdx.x;
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
        bmax[b] = fmaxf(absmax8(v[2 * b]), absmax8(v[2 * b + 1]));
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
        pdl_begin();
        if (t < T) {
            if (tid < K) my_row = row_of[(size_t)t * K + tid];
            else if (tid == K && S) my_row = row_offsets[E] + t;
        }
    }
    if (load_status(status)) return;
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
        if (r < 0 || r >= R_max) continue;
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

__global__ void __launch_bounds__(256)
ep_dispatch_bf16_kernel(const uint16_t *__restrict__ x, int T, int H, int K, int E, int S, int R_max,
                        const int32_t *__restrict__ row_of, const int32_t *__restrict__ row_offsets,
                        const int32_t *__restrict__ status, uint16_t *__restrict__ out) {
    __shared__ int s_rows[kMaxRowsPerToken];
    pdl_begin();
    if (load_status(status)) return;
    const int tid = threadIdx.x;
    const int t = blockIdx.x;
    const int nrows = K + S;
    if (tid < K) s_rows[tid] = row_of[(size_t)t * K + tid];
    else if (tid == K && S) s_rows[K] = row_offsets[E] + t;
    __syncthreads();
    const int nv = H / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    for (int c = tid; c < nv; c += blockDim.x) {
        const uint4 d = ld_stream(src + c);
        for (int k = 0; k < nrows; ++k) {
            const int r = s_rows[k];
            if (r >= 0 && r < R_max) st_stream(out + (size_t)r * H + (size_t)c * 8, d);
        }
    }
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
    const int grid = L->T > 0 ? L->T : 1;
    const int G = L->E + L->fused_shared;
    const int R_max = (int)rows_max(L->T, L->K, L->fused_shared);
    const int32_t *row_of = L->row_of, *row_offsets = L->row_offsets, *status = L->status;
#define EP_NVFP4_LAUNCH(BPT, MAXT, MINB)                                                        \
    return launch_pdl(ep_dispatch_nvfp4_kernel<BPT, MAXT, MINB>, dim3(grid), dim3(threads), 0, st, \
                      input_tokens, L->T, H, L->K, L->E, L->fused_shared, G, R_max, early, row_of, \
                      row_offsets, status, out_fp4, out_scales, out_rowwise_inv_scale,          \
                      scales_offsets)
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
    return launch_nvfp4(input_tokens, hidden_size, L, out_fp4, out_scales, out_rowwise_inv_scale,
                        scales_offsets, 0, as_stream(stream));
}

extern "C" int ep_dispatch_layout_nvfp4(const int32_t *topk_ids, int T, int K, int n_experts,
                                        int n_parts, int capacity, int fused_shared,
                                        const uint16_t *input_tokens, int hidden_size,
                                        ep_layout_t *L, uint8_t *out_fp4, uint8_t *out_scales,
                                        uint16_t *out_rowwise_inv_scale, int32_t *scales_offsets,
                                        void *stream) {
    const int H = hidden_size;
    if (!hidden_ok(H) || H / 16 > 1024) return EP_ERR_INVALID_ARG;
    if ((T > 0 && (!input_tokens || !out_fp4 || !out_scales || !out_rowwise_inv_scale)) ||
        !scales_offsets)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {input_tokens, out_fp4, out_scales, out_rowwise_inv_scale, scales_offsets};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    int rc = launch_layout(topk_ids, T, K, n_experts, n_parts, capacity, fused_shared, L, st, nullptr);
    if (rc != EP_OK) return rc;
    // The dispatch kernel directly follows the layout kernel, which lets it launch only once
    // every earlier kernel of the stream has completed, so its CTAs read and quantise their
    // tokens while the layout is still running and wait for the layout only before storing.
    return launch_nvfp4(input_tokens, H, L, out_fp4, out_scales, out_rowwise_inv_scale,
                        scales_offsets, 1, st);
}

extern "C" int ep_dispatch_bf16(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                                uint16_t *out, void *stream) {
    const int H = hidden_size;
    if (!layout_ok(L) || !hidden_ok(H)) return EP_ERR_INVALID_ARG;
    if (L->T > 0 && (!input_tokens || !out)) return EP_ERR_INVALID_ARG;
    if ((input_tokens && !aligned16(input_tokens)) || (out && !aligned16(out))) return EP_ERR_INVALID_ARG;
    if (L->T == 0) return EP_OK;
    return launch_pdl(ep_dispatch_bf16_kernel, dim3(L->T), dim3(256), 0, as_stream(stream),
                      input_tokens, L->T, H, L->K, L->E, L->fused_shared,
                      (int)rows_max(L->T, L->K, L->fused_shared), (const int32_t *)L->row_of,
                      (const int32_t *)L->row_offsets, (const int32_t *)L->status, out);
}

extern "C" int ep_cvt_e2m1(const float *in, uint8_t *codes, long n, void *stream) {
    return launch_cvt(in, codes, n, stream, 0);
}

extern "C" int ep_cvt_e4m3(const float *in, uint8_t *codes, long n, void *stream) {
    return launch_cvt(in, codes, n, stream, 1);
}
