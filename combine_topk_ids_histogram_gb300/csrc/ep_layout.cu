// ep_layout.cu -- dispatch layout: per-tile expert histogram, expert-major exclusive scan and
// stable ranks (row_offsets, expert_ids, src_info, row_of, part_tokens, status).
//
// Follows the Mojo EP dispatch page (DistributedEPDispatchBlockScaledNVDynGlobalScales.execute:
// route by top-k ids; row_offsets / expert_ids / src_info; max_token_per_rank;
// atomic_counters coordinating the thread blocks) and the fused_a2a page
// (HybridEPDispatch.forward: rows grouped by expert, -1 for unused slots).
//
// Two launches on the caller's stream:
//   1. ep_layout_count_kernel: one CTA per tile of tokens builds the tile's expert histogram
//      and partition token counts in shared memory and writes them to the workspace.  The
//      CTA that finishes last (an atomic ticket, so no CTA ever waits on another) runs the
//      exclusive scan over the [E][nTiles] count table in expert-major, tile-minor order: the
//      scanned value at (e, j) is the first row of tile j's pairs routed to expert e.  It also
//      writes row_offsets, part_tokens and the status word, and re-arms the ticket.
//   2. ep_layout_rank_kernel: one CTA per tile ranks each (t, k) inside its tile and expert,
//      stably in t*K + k order (warp __match_any_sync plus per-warp prefix counters), and
//      writes row_of, src_info and expert_ids; it also writes the shared expert's rows.
#include "ep_common.cuh"
#include "ep_host.h"

namespace ep {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kMaxTiles = 64;          // target tile count: bounds the scan of the count table
constexpr int kMaxTileIds = 8192;      // ids of one tile held in shared memory
constexpr int kScanChunk = 8192;       // count-table entries scanned per pass by the last CTA

// Tokens per tile: at least 128, a multiple of 32, enough to keep about kMaxTiles tiles, and
// at most kMaxTileIds / K so a tile's ids fit in shared memory.
inline int tile_tokens(int T, int K) {
    int want = (T + kMaxTiles - 1) / kMaxTiles;
    want = (want + 31) / 32 * 32;
    int cap = (kMaxTileIds / K) / 32 * 32;
    if (cap < 32) cap = 32;
    int tt = want < 128 ? 128 : want;
    return tt > cap ? cap : tt;
}

inline int num_tiles(int T, int tt) { return T == 0 ? 1 : (T + tt - 1) / tt; }

inline size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace: [ticket | tile_flags[nTiles] | cnt[E][nTiles] | part[E][nTiles]] (P <= E).
struct Workspace {
    int32_t *ticket, *tile_flags, *cnt, *part;
};

inline size_t workspace_bytes(int nTiles, int E) {
    return 256 + align256((size_t)nTiles * 4) + 2 * align256((size_t)E * nTiles * 4);
}

inline Workspace carve(void *base, int nTiles, int E) {
    char *p = static_cast<char *>(base);
    Workspace w;
    w.ticket = reinterpret_cast<int32_t *>(p);
    p += 256;
    w.tile_flags = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)nTiles * 4);
    w.cnt = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)E * nTiles * 4);
    w.part = reinterpret_cast<int32_t *>(p);
    return w;
}

__device__ __forceinline__ bool bad_id(int id, int E) { return id < -1 || id >= E; }

// Exclusive scan of one value per thread across the block (blockDim == kLayoutThreads).
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kLayoutWarps; ++w) {
        int t = warp_tot[w];
        if (w < warp) before += t;
        total += t;
    }
    __syncthreads();
    return before + incl - v;
}

__global__ void __launch_bounds__(kLayoutThreads)
ep_layout_count_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int P, int C, int S,
                       int tile_t, int nTiles, Workspace ws, int32_t *__restrict__ row_offsets,
                       int32_t *__restrict__ part_tokens, int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    int *s_hist = smem;          // [E]
    int *s_part = smem + E;      // [P]
    __shared__ int s_bad;
    __shared__ int s_last;
    __shared__ int s_warp[kLayoutWarps];

    const int tid = threadIdx.x, lane = tid & 31;
    const int j = blockIdx.x;
    for (int e = tid; e < E; e += blockDim.x) s_hist[e] = 0;
    for (int p = tid; p < P; p += blockDim.x) s_part[p] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    const int t0 = j * tile_t;
    const int t1 = min(T, t0 + tile_t);
    const int n = max(0, t1 - t0) * K;
    const int32_t *tid_ids = ids + (size_t)t0 * K;
    // Expert histogram; lanes holding the same id add once through their leader.
    for (int base = 0; base < n; base += blockDim.x) {
        int i = base + tid;
        int id = -1;
        if (i < n) {
            id = tid_ids[i];
            if (bad_id(id, E)) {
                s_bad = 1;
                id = -1;
            }
        }
        unsigned peers = __match_any_sync(kFullMask, id);
        if (id >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[id], __popc(peers));
    }
    // Tokens per partition: a token counts once for every partition one of its ids reaches.
    const int per = E / P;
    const int ntok = max(0, t1 - t0);
    for (int base = 0; base < ntok; base += blockDim.x) {
        int tl = base + tid;
        for (int k = 0; k < K; ++k) {
            int p = -1;
            if (tl < ntok) {
                int id = tid_ids[(size_t)tl * K + k];
                if (!bad_id(id, E) && id >= 0) {
                    p = id / per;
                    for (int k2 = 0; k2 < k; ++k2) {
                        int id2 = tid_ids[(size_t)tl * K + k2];
                        if (!bad_id(id2, E) && id2 >= 0 && id2 / per == p) {
                            p = -1;
                            break;
                        }
                    }
                }
            }
            unsigned peers = __match_any_sync(kFullMask, p);
            if (p >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_part[p], __popc(peers));
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) ws.cnt[(size_t)e * nTiles + j] = s_hist[e];
    for (int p = tid; p < P; p += blockDim.x) ws.part[(size_t)p * nTiles + j] = s_part[p];
    if (tid == 0) ws.tile_flags[j] = s_bad;

    // The last CTA to finish scans the whole table.
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(ws.ticket, 1) == nTiles - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Exclusive scan of cnt in place, kScanChunk entries per pass, through shared memory
    // (padded by one word per 32 so each thread's contiguous segment is conflict-free).
    int *s_chunk = smem;   // reuses the histogram space: kScanChunk + kScanChunk/32 ints
    const long total_n = (long)E * nTiles;
    const int seg = kScanChunk / kLayoutThreads;
    int carry = 0;
    for (long c0 = 0; c0 < total_n; c0 += kScanChunk) {
        const int len = (int)min((long)kScanChunk, total_n - c0);
        for (int i = tid; i < len; i += blockDim.x) s_chunk[i + (i >> 5)] = __ldcg(ws.cnt + c0 + i);
        __syncthreads();
        int sum = 0;
        for (int q = 0; q < seg; ++q) {
            int i = tid * seg + q;
            if (i < len) sum += s_chunk[i + (i >> 5)];
        }
        int tot;
        int run = carry + block_exclusive_scan(sum, s_warp, tot);
        for (int q = 0; q < seg; ++q) {
            int i = tid * seg + q;
            if (i < len) {
                int v = s_chunk[i + (i >> 5)];
                s_chunk[i + (i >> 5)] = run;
                run += v;
            }
        }
        __syncthreads();
        for (int i = tid; i < len; i += blockDim.x) ws.cnt[c0 + i] = s_chunk[i + (i >> 5)];
        carry += tot;
        __syncthreads();
    }
    __threadfence_block();
    // row_offsets: first row of each expert, then the shared group, then R.
    for (int e = tid; e < E; e += blockDim.x) row_offsets[e] = __ldcg(ws.cnt + (size_t)e * nTiles);
    if (tid == 0) {
        row_offsets[E] = carry;
        if (S) row_offsets[E + 1] = carry + T;
    }
    // Partition totals against the capacity, and the bad-id flags.
    int flags = 0;
    for (int p = tid; p < P; p += blockDim.x) {
        int s = 0;
        for (int jj = 0; jj < nTiles; ++jj) s += __ldcg(ws.part + (size_t)p * nTiles + jj);
        part_tokens[p] = s;
        if (s > C) flags |= EP_STATUS_OVERFLOW;
    }
    for (int jj = tid; jj < nTiles; jj += blockDim.x)
        if (__ldcg(ws.tile_flags + jj)) flags |= EP_STATUS_BAD_EXPERT;
    flags = __reduce_or_sync(kFullMask, flags);
    if (lane == 0) s_warp[tid >> 5] = flags;
    __syncthreads();
    if (tid == 0) {
        int f = 0;
        for (int w = 0; w < kLayoutWarps; ++w) f |= s_warp[w];
        *status = f;
        *ws.ticket = 0;   // ready for the next call
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
ep_layout_rank_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int S, int tile_t,
                      int nTiles, const int32_t *__restrict__ cnt,
                      const int32_t *__restrict__ row_offsets, int32_t *__restrict__ row_of,
                      int32_t *__restrict__ src_info, int32_t *__restrict__ expert_ids) {
    extern __shared__ int smem[];
    int *s_whist = smem;                       // [kLayoutWarps][E]
    int *s_ids = smem + kLayoutWarps * E;      // [tile_t * K]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x;
    const int t0 = j * tile_t;
    const int t1 = min(T, t0 + tile_t);
    const int n = max(0, t1 - t0) * K;

    for (int i = tid; i < kLayoutWarps * E; i += blockDim.x) s_whist[i] = 0;
    for (int i = tid; i < n; i += blockDim.x) {
        int id = ids[(size_t)t0 * K + i];
        s_ids[i] = bad_id(id, E) ? -1 : id;
    }
    __syncthreads();

    // Each warp owns one contiguous run of the tile's flat (t, k) indices.
    const int per_warp = ((n + kLayoutWarps - 1) / kLayoutWarps + 31) / 32 * 32;
    const int w0 = min(n, warp * per_warp), w1 = min(n, w0 + per_warp);
    int *hist = s_whist + warp * E;
    for (int base = w0; base < w1; base += 32) {
        int i = base + lane;
        int id = i < w1 ? s_ids[i] : -1;
        unsigned peers = __match_any_sync(kFullMask, id);
        if (id >= 0 && lane == __ffs(peers) - 1) hist[id] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // First row of each (warp, expert): the tile's scanned base plus earlier warps' counts.
    for (int e = tid; e < E; e += blockDim.x) {
        int run = cnt[(size_t)e * nTiles + j];
        for (int w = 0; w < kLayoutWarps; ++w) {
            int c = s_whist[w * E + e];
            s_whist[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        int i = base + lane;
        int id = i < w1 ? s_ids[i] : -1;
        unsigned peers = __match_any_sync(kFullMask, id);
        int row = -1;
        if (id >= 0) row = hist[id] + __popc(peers & lt_mask);
        __syncwarp();
        if (id >= 0 && lane == __ffs(peers) - 1) hist[id] += __popc(peers);
        __syncwarp();
        if (i < w1) {
            size_t flat = (size_t)t0 * K + i;
            if (row >= T * K) row = -1;   // only a layout raced by a concurrent writer of ids
            row_of[flat] = row;
            if (row >= 0) {
                int t = t0 + i / K;
                reinterpret_cast<int2 *>(src_info)[row] = make_int2(t, i - (i / K) * K);
                expert_ids[row] = id;
            }
        }
    }
    if (S) {
        const int rs = row_offsets[E];
        for (int t = t0 + tid; t < t1; t += blockDim.x) {
            reinterpret_cast<int2 *>(src_info)[rs + t] = make_int2(t, K);
            expert_ids[rs + t] = E;
        }
    }
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" size_t ep_layout_workspace_bytes(int T, int K, int n_experts, int fused_shared) {
    if (!sizes_ok(T, K, n_experts, fused_shared)) return 0;
    int tt = tile_tokens(T, K);
    return workspace_bytes(num_tiles(T, tt), n_experts);
}

extern "C" int ep_dispatch_layout(const int32_t *topk_ids, int T, int K, int n_experts,
                                  int n_parts, int capacity, int fused_shared, ep_layout_t *L,
                                  void *stream) {
    const int E = n_experts, P = n_parts, S = fused_shared;
    if (!L || !sizes_ok(T, K, E, S)) return EP_ERR_INVALID_ARG;
    if (P < 1 || P > E || E % P != 0 || capacity < 0) return EP_ERR_INVALID_ARG;
    if ((T > 0 && !topk_ids) || !L->row_offsets || !L->expert_ids || !L->src_info ||
        !L->row_of || !L->part_tokens || !L->status || !L->workspace)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {topk_ids, L->row_offsets, L->expert_ids, L->src_info, L->row_of,
                          L->part_tokens, L->status, L->workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    const int tt = tile_tokens(T, K);
    const int nTiles = num_tiles(T, tt);
    if (L->workspace_bytes < workspace_bytes(nTiles, E)) return EP_ERR_INVALID_ARG;

    L->T = T;
    L->K = K;
    L->E = E;
    L->P = P;
    L->capacity = capacity;
    L->fused_shared = S;

    cudaStream_t st = as_stream(stream);
    Workspace ws = carve(L->workspace, nTiles, E);
    size_t smem_count = sizeof(int) * (size_t)max(E + P, kScanChunk + kScanChunk / 32);
    ep_layout_count_kernel<<<nTiles, kLayoutThreads, smem_count, st>>>(
        topk_ids, T, K, E, P, capacity, S, tt, nTiles, ws, L->row_offsets, L->part_tokens,
        L->status);
    int rc = launch_result();
    if (rc != EP_OK) return rc;
    size_t smem_rank = sizeof(int) * ((size_t)kLayoutWarps * E + (size_t)tt * K);
    if (smem_rank > 48 * 1024 &&
        cudaFuncSetAttribute(ep_layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_rank) != cudaSuccess)
        return EP_ERR_CUDA;
    ep_layout_rank_kernel<<<nTiles, kLayoutThreads, smem_rank, st>>>(
        topk_ids, T, K, E, S, tt, nTiles, ws.cnt, L->row_offsets, L->row_of, L->src_info,
        L->expert_ids);
    return launch_result();
}

extern "C" int ep_read_status(const ep_layout_t *L, void *stream, int32_t *host_status) {
    if (!L || !L->status || !host_status) return EP_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, L->status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return EP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    *host_status = v;
    if (v & EP_STATUS_OVERFLOW) return EP_ERR_OVERFLOW;
    if (v & EP_STATUS_BAD_EXPERT) return EP_ERR_BAD_EXPERT;
    return EP_OK;
}

extern "C" const char *ep_strerror(int code) {
    switch (code) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_OVERFLOW: return "a logical partition received more tokens than its capacity";
        case EP_ERR_BAD_EXPERT: return "an expert id was outside [-1, n_experts)";
        case EP_ERR_CUDA: return "CUDA error";
        case EP_ERR_TOO_LARGE: return "the sizes need more scratch than the fixed no-allocation array holds";
        default: return "unknown error";
    }
}

// ---------------------------------------------------------------------------------------
// ep_dispatch_layout_noalloc: the same layout with its scratch in a fixed device array.
//
// For callers that must not allocate device memory at all: code running under a framework
// whose caching allocator owns the whole device, latency-critical paths where an allocation
// (and the device synchronisation cudaMalloc/cudaFree can imply) is not acceptable, or
// runtimes that hand a library only its inputs and outputs.  The scratch lives in a
// file-scope __device__ array of kNoAllocWorkspaceBytes that every GPU which loads this
// library keeps until the process exits.  Host code cannot use the array's name as a device
// address (on the host it is only a stand-in symbol), so the device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, during the first call on
// that device.  That first call also zeroes the ticket word; every later call leaves it at zero
// when it finishes.  All calls share the one array, so calls whose work overlaps on the GPU
// (other streams, other threads) race on it.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace ep {
namespace {

constexpr size_t kNoAllocWorkspaceBytes = EP_NOALLOC_WORKSPACE_BYTES;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_address[kNoAllocMaxDevices];   // device address of the array, per device

// Device address of the scratch array on the current device (set up on first use).
int noalloc_workspace(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr)
            return EP_ERR_CUDA;
        if (cudaMemset(p, 0, 256) != cudaSuccess) return EP_ERR_CUDA;   // the ticket starts at 0
        g_noalloc_address[dev] = p;
    }
    *out = g_noalloc_address[dev];
    return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" int ep_dispatch_layout_noalloc(const int32_t *topk_ids, int T, int K, int n_experts,
                                          int n_parts, int capacity, int fused_shared,
                                          ep_layout_t *L, void *stream) {
    const int E = n_experts, P = n_parts, S = fused_shared;
    if (!L || !sizes_ok(T, K, E, S)) return EP_ERR_INVALID_ARG;
    if (P < 1 || P > E || E % P != 0 || capacity < 0) return EP_ERR_INVALID_ARG;
    if ((T > 0 && !topk_ids) || !L->row_offsets || !L->expert_ids || !L->src_info ||
        !L->row_of || !L->part_tokens || !L->status)
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {topk_ids, L->row_offsets, L->expert_ids, L->src_info, L->row_of,
                          L->part_tokens, L->status};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return EP_ERR_INVALID_ARG;
    const int tt = tile_tokens(T, K);
    const int nTiles = num_tiles(T, tt);
    if (workspace_bytes(nTiles, E) > kNoAllocWorkspaceBytes) return EP_ERR_TOO_LARGE;
    void *scratch = nullptr;
    int rc = noalloc_workspace(&scratch);
    if (rc != EP_OK) return rc;

    L->T = T;
    L->K = K;
    L->E = E;
    L->P = P;
    L->capacity = capacity;
    L->fused_shared = S;

    cudaStream_t st = as_stream(stream);
    Workspace ws = carve(scratch, nTiles, E);
    size_t smem_count = sizeof(int) * (size_t)max(E + P, kScanChunk + kScanChunk / 32);
    ep_layout_count_kernel<<<nTiles, kLayoutThreads, smem_count, st>>>(
        topk_ids, T, K, E, P, capacity, S, tt, nTiles, ws, L->row_offsets, L->part_tokens,
        L->status);
    rc = launch_result();
    if (rc != EP_OK) return rc;
    size_t smem_rank = sizeof(int) * ((size_t)kLayoutWarps * E + (size_t)tt * K);
    if (smem_rank > 48 * 1024 &&
        cudaFuncSetAttribute(ep_layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_rank) != cudaSuccess)
        return EP_ERR_CUDA;
    ep_layout_rank_kernel<<<nTiles, kLayoutThreads, smem_rank, st>>>(
        topk_ids, T, K, E, S, tt, nTiles, ws.cnt, L->row_offsets, L->row_of, L->src_info,
        L->expert_ids);
    return launch_result();
}
