// ep_host.h -- host-side argument checks shared by the entry points of libep_gb300.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>
#include <utility>

#include "ep.h"

namespace ep {

// Optional NVTX range around each entry point, named after it, so that a profiler can select an
// op's kernels by range (ncu --nvtx --nvtx-include "ep_combine/", or a timeline tool).  On when
// the environment variable EP_GB300_NVTX is set to anything but "0" when the library first
// checks it; otherwise an entry point pays one test of a cached flag.  The header-only NVTX
// API does nothing unless a profiler is attached.
inline bool nvtx_enabled() {
    static const bool on = [] {
        const char *v = getenv("EP_GB300_NVTX");
        return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
    }();
    return on;
}
struct NvtxScope {
    bool on;
    explicit NvtxScope(const char *name) : on(nvtx_enabled()) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxScope() {
        if (on) nvtxRangePop();
    }
    NvtxScope(const NvtxScope &) = delete;
    NvtxScope &operator=(const NvtxScope &) = delete;
};
#define EP_NVTX_RANGE(name) ::ep::NvtxScope ep_nvtx_range_(name)

constexpr int kMaxK = 32;
constexpr int kMaxE = 1024;
constexpr int kMaxT = 1 << 24;
constexpr int kMaxH = 32768;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr int kMaxPad = 65536;

// Rows every dispatched buffer holds: T*K routed rows plus one shared row per token.
inline long long rows_max(int T, int K, int S) { return (long long)T * K + (long long)S * T; }

// Rows every dispatched buffer holds for a padded layout: the static row capacity when one is
// set, else the routed and shared rows plus at most pad - 1 padding rows per group.
inline long long rows_max(int T, int K, int E, int S, int pad, int row_capacity) {
    if (row_capacity > 0) return row_capacity;
    const long long p = pad > 1 ? pad : 1;
    return rows_max(T, K, S) + (long long)(E + S) * (p - 1);
}

inline bool sizes_ok(int T, int K, int E, int S) {
    if (T < 0 || T > kMaxT || K < 1 || K > kMaxK || E < 1 || E > kMaxE) return false;
    if (S != 0 && S != 1) return false;
    return rows_max(T, K, S) < (1ll << 31);
}

// Padding multiple and row capacity of a layout call (pad 1 / capacity 0: none).
inline bool padding_ok(int T, int K, int E, int S, int pad, int row_capacity) {
    if (pad < 1 || pad > kMaxPad || row_capacity < 0) return false;
    return rows_max(T, K, E, S, pad, 0) < (1ll << 31);   // the padded row count fits an int
}

// A layout filled by a layout call, with every buffer present.
inline bool layout_ok(const ep_layout_t *L) {
    if (!L || !L->row_offsets || !L->row_of || !L->status) return false;
    if (!sizes_ok(L->T, L->K, L->E, L->fused_shared)) return false;
    if (L->P < 1 || L->P > L->E || L->E % L->P != 0) return false;
    if (L->pad_multiple < 0 || L->pad_multiple > kMaxPad || L->row_capacity < 0) return false;
    return rows_max(L->T, L->K, L->E, L->fused_shared, L->pad_multiple, L->row_capacity) < (1ll << 31);
}

// Rows of every dispatched buffer of a layout, and whether it has padding rows.
inline int layout_rows(const ep_layout_t *L) {
    return (int)rows_max(L->T, L->K, L->E, L->fused_shared, L->pad_multiple, L->row_capacity);
}
inline bool layout_padded(const ep_layout_t *L) { return L->pad_multiple > 1; }

inline bool hidden_ok(int H) { return H >= 16 && H <= kMaxH && H % 16 == 0; }

// Map the result of a launch to a return code.
inline int launch_result() { return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA; }
inline int launch_result(cudaError_t e) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return launch_result();
}

// Launch with programmatic stream serialization, so the kernel's launch overlaps the tail of
// the previous kernel in the stream (the kernel itself waits for it; see pdl_begin).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_result(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// SM count of the current device (0 on error), looked up once per device.
inline int device_sm_count() {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev];   // 0: not looked up
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < kMaxDev && cached[dev]) return cached[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDev) cached[dev] = sms;
    return sms;
}

// Whether a grid of `ctas` blocks is no larger than the SM count, so that all of its blocks are
// resident at once (one per SM is enough).
inline int one_wave(int ctas) {
    const int sms = device_sm_count();
    return sms > 0 && ctas <= sms ? 1 : 0;
}

// Blocks of `kernel` that fit on the device at once (SM count x resident blocks per SM),
// for grids that loop over their work.  Cached per (device, kernel, block size, shared memory).
template <typename K>
inline int resident_blocks(K kernel, int threads, size_t smem) {
    struct Entry {
        int dev, threads;
        const void *fn;
        size_t smem;
        int blocks;
    };
    constexpr int kSlots = 32;
    static Entry cache[kSlots];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const void *fn = reinterpret_cast<const void *>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
        if (e.blocks > 0 && e.dev == dev && e.fn == fn && e.threads == threads && e.smem == smem)
            return e.blocks;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
        return 0;
    const int blocks = sms * (per_sm > 0 ? per_sm : 1);
    for (Entry &e : cache)
        if (e.blocks == 0) {
            e = Entry{dev, threads, fn, smem, blocks};
            break;
        }
    return blocks;
}

// Enqueues a dispatch layout (ep_layout.cu) with groups padded to a multiple of `pad` and at
// most `row_capacity` rows (0: the default R_max).  *cluster_ctas_used receives the number of
// SMs the single-cluster layout kernel occupies, or 0 when the two-kernel path ran.  With
// write_rows 0 an unpadded, uncapped layout that takes the single-cluster kernel leaves
// src_info and expert_ids unwritten: the dispatch kernel enqueued right after it writes them.
int launch_layout(const int32_t *topk_ids, int T, int K, int E, int P, int capacity, int S,
                  int pad, int row_capacity, ep_layout_t *L, cudaStream_t st,
                  int *cluster_ctas_used, int write_rows = 1);

// SMs the single-cluster layout kernel would occupy for these sizes, or 0 when the layout
// would take the two-kernel path.
int layout_cluster_plan(int T, int K, int E, int P);

// Enqueues the routing-map -> compact ids conversion (ep_routing.cu); arguments checked.
int launch_map_to_topk(const uint8_t *routing_map, const float *dense_probs, int T, int E, int K,
                       int32_t *topk_ids, float *topk_probs, cudaStream_t st);

}  // namespace ep
