// ep_routing.cu -- conversions between the two routing representations: a dense routing map
// [T, E] (non-zero where token t goes to expert e) with dense probabilities, and compact top-k
// ids [T, K] (-1 for an unused slot) with per-slot probabilities (fused_a2a page,
// HybridEPDispatch.forward; token_dispatcher page, _indices_to_multihot).
//
// Both directions give one warp to each token, so a token's row of the map is read or written
// with consecutive lanes on consecutive experts.
#include "ep_common.cuh"
#include "ep_host.h"

namespace ep {
namespace {

constexpr int kRoutingThreads = 256;
constexpr int kRoutingWarps = kRoutingThreads / 32;

// Map -> compact.  First pass: count the token's experts (one ballot per 32 experts).  A
// token with more than K gets the id E in every slot.  Otherwise the second pass writes each
// set expert at its rank among the set experts (ascending id), and lanes then fill the slots
// after the last one with -1.
__global__ void __launch_bounds__(kRoutingThreads)
ep_map_to_topk_kernel(const uint8_t *__restrict__ map, const float *__restrict__ dense, int T, int E,
                      int K, int32_t *__restrict__ ids, float *__restrict__ probs) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int t = blockIdx.x * kRoutingWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kRoutingWarps) {
        const uint8_t *row = map + (size_t)t * E;
        int n = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            n += __popc(__ballot_sync(kFullMask, e < E && row[e] != 0));
        }
        int32_t *oid = ids + (size_t)t * K;
        float *op = probs ? probs + (size_t)t * K : nullptr;
        if (n > K) {
            if (lane < K) {
                oid[lane] = E;
                if (op) op[lane] = 0.0f;
            }
            continue;
        }
        int before = 0;
        for (int e0 = 0; e0 < E && before < n; e0 += 32) {
            const int e = e0 + lane;
            const bool set = e < E && row[e] != 0;
            const unsigned b = __ballot_sync(kFullMask, set);
            if (set) {
                const int slot = before + __popc(b & lt_mask);
                oid[slot] = e;
                if (op) op[slot] = dense ? dense[(size_t)t * E + e] : 0.0f;
            }
            before += __popc(b);
        }
        if (lane >= n && lane < K) {
            oid[lane] = -1;
            if (op) op[lane] = 0.0f;
        }
    }
}

// Map -> compact when E % 16 == 0: each lane reads 16 map bytes per 16-byte load (a 16-bit
// mask of set experts), a warp scan of the masks' counts gives each lane's first slot, and
// each lane writes its set experts in ascending order.  One pass of at most E/512 loads per
// lane; the ids past the token's last expert are written -1 after the total is known.
__device__ __forceinline__ unsigned byte_mask16(uint4 v) {
    unsigned m = 0;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if ((w[i >> 2] >> (8 * (i & 3))) & 0xffu) m |= 1u << i;
    return m;
}

__global__ void __launch_bounds__(kRoutingThreads)
ep_map_to_topk_wide_kernel(const uint8_t *__restrict__ map, const float *__restrict__ dense, int T,
                           int E, int K, int32_t *__restrict__ ids, float *__restrict__ probs) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nchunk = E / 16;                    // 16-byte chunks per map row
    for (int t = blockIdx.x * kRoutingWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kRoutingWarps) {
        const uint4 *row = reinterpret_cast<const uint4 *>(map + (size_t)t * E);
        unsigned m0 = 0, m1 = 0;                  // chunks lane and lane + 32 (E <= 1024)
        if (lane < nchunk) m0 = byte_mask16(__ldg(row + lane));
        if (lane + 32 < nchunk) m1 = byte_mask16(__ldg(row + lane + 32));
        const int c0 = __popc(m0), c1 = __popc(m1);
        int incl0 = c0, incl1 = c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(kFullMask, incl0, o);
            const int b = __shfl_up_sync(kFullMask, incl1, o);
            if (lane >= o) {
                incl0 += a;
                incl1 += b;
            }
        }
        const int tot0 = __shfl_sync(kFullMask, incl0, 31);
        const int n = tot0 + __shfl_sync(kFullMask, incl1, 31);
        int32_t *oid = ids + (size_t)t * K;
        float *op = probs ? probs + (size_t)t * K : nullptr;
        if (n > K) {
            if (lane < K) {
                oid[lane] = E;
                if (op) op[lane] = 0.0f;
            }
            continue;
        }
        int slot = incl0 - c0;
        for (unsigned m = m0; m; m &= m - 1) {
            const int e = 16 * lane + __ffs(m) - 1;
            oid[slot] = e;
            if (op) op[slot] = dense ? dense[(size_t)t * E + e] : 0.0f;
            ++slot;
        }
        slot = tot0 + incl1 - c1;
        for (unsigned m = m1; m; m &= m - 1) {
            const int e = 16 * (lane + 32) + __ffs(m) - 1;
            oid[slot] = e;
            if (op) op[slot] = dense ? dense[(size_t)t * E + e] : 0.0f;
            ++slot;
        }
        if (lane >= n && lane < K) {
            oid[lane] = -1;
            if (op) op[lane] = 0.0f;
        }
    }
}

// Compact -> map.  Lane k < K holds the token's slot k; for each expert of its stripe a lane
// walks the K slots (shuffles, ascending k) and adds the probabilities of the slots naming it.
__global__ void __launch_bounds__(kRoutingThreads)
ep_indices_to_multihot_kernel(const int32_t *__restrict__ ids, const float *__restrict__ probs, int T,
                              int K, int E, uint8_t *__restrict__ map, float *__restrict__ dense) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    for (int t = blockIdx.x * kRoutingWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kRoutingWarps) {
        const int my_id = lane < K ? ids[(size_t)t * K + lane] : -1;
        const float my_p = (lane < K && probs) ? probs[(size_t)t * K + lane] : 0.0f;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            bool hit = false;
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                const int id = __shfl_sync(kFullMask, my_id, k);
                const float p = __shfl_sync(kFullMask, my_p, k);
                if (id == e) {
                    hit = true;
                    acc = __fadd_rn(acc, p);
                }
            }
            if (e < E) {
                map[(size_t)t * E + e] = hit ? 1 : 0;
                if (dense) dense[(size_t)t * E + e] = acc;
            }
        }
    }
}

// Compact -> map when E % 16 == 0 (map rows 16-byte aligned, dense rows 64-byte aligned): each
// warp builds its token's map and dense rows in shared memory, then writes them with 16-byte
// stores.  The K slots are broadcast once (id and probability); each lane holding a slot keeps
// the sum, in ascending slot order, of the probabilities of the slots naming its expert, and
// the lowest such slot writes it.  About 2K shuffles and a few vector accesses per lane and
// token, against E/32 * K shuffle pairs in the kernel above.
__global__ void __launch_bounds__(kRoutingThreads)
ep_indices_to_multihot_wide_kernel(const int32_t *__restrict__ ids, const float *__restrict__ probs, int T,
                                   int K, int E, uint8_t *__restrict__ map, float *__restrict__ dense) {
    __shared__ __align__(16) float s_dense[kRoutingWarps][kMaxE];
    __shared__ __align__(16) uint8_t s_map[kRoutingWarps][kMaxE];
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float *sd = s_dense[warp];
    uint8_t *sm = s_map[warp];
    const int n16 = E / 16;   // 16-byte chunks of a map row (a dense row has 4 * n16)
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    for (int t = blockIdx.x * kRoutingWarps + warp; t < T; t += gridDim.x * kRoutingWarps) {
        const int my_id = lane < K ? ids[(size_t)t * K + lane] : -1;
        const float my_p = (lane < K && probs) ? probs[(size_t)t * K + lane] : 0.0f;
        const bool valid = my_id >= 0 && my_id < E;
        for (int c = lane; c < n16; c += 32) reinterpret_cast<uint4 *>(sm)[c] = z4;
        if (dense)
            for (int c = lane; c < 4 * n16; c += 32) reinterpret_cast<uint4 *>(sd)[c] = z4;
        bool first = valid;
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int id = __shfl_sync(kFullMask, my_id, k);
            const float p = __shfl_sync(kFullMask, my_p, k);
            if (valid && id == my_id) {
                if (k < lane) first = false;
                acc = __fadd_rn(acc, p);
            }
        }
        __syncwarp();   // the row is zero before any expert is set
        if (first) {
            sm[my_id] = 1;
            if (dense) sd[my_id] = acc;
        }
        __syncwarp();
        uint8_t *mrow = map + (size_t)t * E;
        for (int c = lane; c < n16; c += 32)
            reinterpret_cast<uint4 *>(mrow)[c] = reinterpret_cast<const uint4 *>(sm)[c];
        if (dense) {
            float *drow = dense + (size_t)t * E;
            for (int c = lane; c < 4 * n16; c += 32)
                reinterpret_cast<uint4 *>(drow)[c] = reinterpret_cast<const uint4 *>(sd)[c];
        }
        __syncwarp();   // every lane has read the row before the next token clears it
    }
}

inline int routing_grid(int T) {
    int grid = (T + kRoutingWarps - 1) / kRoutingWarps;
    const int cap = 152 * 8;
    return grid < 1 ? 1 : (grid > cap ? cap : grid);
}

}  // namespace

int launch_map_to_topk(const uint8_t *routing_map, const float *dense_probs, int T, int E, int K,
                       int32_t *topk_ids, float *topk_probs, cudaStream_t st) {
    if (T < 0 || T > kMaxT || E < 1 || E > kMaxE || K < 1 || K > kMaxK) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!routing_map || !topk_ids)) return EP_ERR_INVALID_ARG;
    if ((routing_map && !aligned16(routing_map)) || (dense_probs && !aligned16(dense_probs)) ||
        (topk_ids && !aligned16(topk_ids)) || (topk_probs && !aligned16(topk_probs)))
        return EP_ERR_INVALID_ARG;
    if (T == 0) return EP_OK;
    if (E % 16 == 0)   // every map row starts on a 16-byte boundary
        return launch_pdl(ep_map_to_topk_wide_kernel, dim3(routing_grid(T)), dim3(kRoutingThreads), 0,
                          st, routing_map, dense_probs, T, E, K, topk_ids, topk_probs);
    return launch_pdl(ep_map_to_topk_kernel, dim3(routing_grid(T)), dim3(kRoutingThreads), 0, st,
                      routing_map, dense_probs, T, E, K, topk_ids, topk_probs);
}

}  // namespace ep

using namespace ep;

extern "C" int ep_routing_map_to_topk(const uint8_t *routing_map, const float *dense_probs, int T,
                                      int n_experts, int K, int32_t *topk_ids, float *topk_probs,
                                      void *stream) {
    EP_NVTX_RANGE("ep_routing_map_to_topk");
    return launch_map_to_topk(routing_map, dense_probs, T, n_experts, K, topk_ids, topk_probs,
                              as_stream(stream));
}

extern "C" int ep_indices_to_multihot(const int32_t *topk_ids, const float *topk_probs, int T, int K,
                                      int n_experts, uint8_t *routing_map, float *dense_probs,
                                      void *stream) {
    EP_NVTX_RANGE("ep_indices_to_multihot");
    const int E = n_experts;
    if (T < 0 || T > kMaxT || E < 1 || E > kMaxE || K < 1 || K > kMaxK) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !routing_map)) return EP_ERR_INVALID_ARG;
    if ((topk_ids && !aligned16(topk_ids)) || (topk_probs && !aligned16(topk_probs)) ||
        (routing_map && !aligned16(routing_map)) || (dense_probs && !aligned16(dense_probs)))
        return EP_ERR_INVALID_ARG;
    if (T == 0) return EP_OK;
    if (E % 16 == 0)   // every map row starts on a 16-byte boundary
        return launch_pdl(ep_indices_to_multihot_wide_kernel, dim3(routing_grid(T)), dim3(kRoutingThreads),
                          0, as_stream(stream), topk_ids, topk_probs, T, K, E, routing_map, dense_probs);
    return launch_pdl(ep_indices_to_multihot_kernel, dim3(routing_grid(T)), dim3(kRoutingThreads), 0,
                      as_stream(stream), topk_ids, topk_probs, T, K, E, routing_map, dense_probs);
}
