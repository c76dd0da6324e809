// ep_layout.cu -- dispatch layout: per-tile expert histogram, expert-major exclusive scan and
// stable ranks (row_offsets, expert_ids, src_info, row_of, part_tokens, status).
//
// Follows the Mojo EP dispatch page (DistributedEPDispatchBlockScaledNVDynGlobalScales.execute:
// route by top-k ids; row_offsets / expert_ids / src_info; max_token_per_rank;
// atomic_counters coordinating the thread blocks) and the fused_a2a page
// (HybridEPDispatch.forward: the rows come out grouped by expert; an index of -1 routes
// nowhere).
//
// Up to 262,144 (token, slot) ids the whole layout is one launch of ep_layout_cluster_kernel on
// a thread-block cluster (described before that kernel below).  Beyond that, and where the
// cluster's shared-memory plan does not fit, two launches on the caller's stream:
//   1. ep_layout_count_kernel: one CTA per tile of tokens builds the tile's expert histogram
//      and partition token counts in shared memory and writes them to the workspace.  The
//      CTA that finishes last (an atomic ticket, so no CTA ever waits on another) runs the
//      exclusive scan over the [E][nTiles] count table in expert-major, tile-minor order: the
//      scanned value at (e, j) is the first row of tile j's pairs routed to expert e.  It also
//      writes row_offsets, part_tokens and the status word, and re-arms the ticket.
//   2. ep_layout_rank_kernel: one CTA per tile ranks each (t, k) inside its tile and expert,
//      stably in t*K + k order (equal-id lanes found with one ballot per id bit, plus
//      per-warp prefix counters), and
//      writes row_of, src_info and expert_ids; it also writes the shared expert's rows.
#include <cooperative_groups.h>

#include <mutex>

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

// Lanes of the warp whose key equals this lane's (keys in [0, 2^nbits)): the intersection, over
// the key's bits, of the lanes that agree with this lane on that bit -- one ballot per bit.
constexpr int kMaxKeyBits = 11;   // keys id + 1 in [0, kMaxE]

__device__ __forceinline__ unsigned same_key_lanes(unsigned key, int nbits) {
    unsigned peers = kFullMask;
#pragma unroll
    for (int b = 0; b < kMaxKeyBits; ++b) {   // unrolled: the ballots are independent
        if (b < nbits) {
            const unsigned bit = (key >> b) & 1u;
            const unsigned m = __ballot_sync(kFullMask, bit);
            peers &= bit ? m : ~m;
        }
    }
    return peers;
}

// n / d for n < 2^32 / d, from the host-computed magic ceil(2^32 / d): one wide multiply
// instead of an integer division.
__device__ __forceinline__ int div_magic(unsigned n, unsigned long long magic) {
    return (int)(((unsigned long long)n * magic) >> 32);
}
inline unsigned long long magic_of(int d) { return ((1ull << 32) + (unsigned)d - 1) / (unsigned)d; }

// Bits needed to hold the values 0 .. n-1.
inline int key_bits(int n) {
    int b = 0;
    while ((1 << b) < n) ++b;
    return b;
}

// Adds to s_part[p] the number of the ntok staged tokens (ids in s_ids, K per token, -1 for an
// unused slot) that reach partition p; a token counts once per partition.  With at most 32
// partitions each token builds a partition bitmask and each warp adds one ballot count per
// partition; otherwise each token adds its distinct partitions one by one.
__device__ __forceinline__ void count_partition_tokens(const int *s_ids, int ntok, int K,
                                                       unsigned long long per_magic, int P,
                                                       int *s_part) {
    const int lane = threadIdx.x & 31;
    for (int base = 0; base < ntok; base += blockDim.x) {
        const int tl = base + threadIdx.x;
        if (P <= 32) {
            unsigned mask = 0;
            if (tl < ntok)
                for (int k = 0; k < K; ++k) {
                    const int id = s_ids[tl * K + k];
                    if (id >= 0) mask |= 1u << div_magic((unsigned)id, per_magic);
                }
            for (int p = 0; p < P; ++p) {
                const int c = __popc(__ballot_sync(kFullMask, (mask >> p) & 1u));
                if (lane == 0 && c) atomicAdd(&s_part[p], c);
            }
        } else if (tl < ntok) {
            for (int k = 0; k < K; ++k) {
                const int id = s_ids[tl * K + k];
                if (id < 0) continue;
                const int p = div_magic((unsigned)id, per_magic);
                bool first = true;
                for (int k2 = 0; k2 < k && first; ++k2) {
                    const int id2 = s_ids[tl * K + k2];
                    first = !(id2 >= 0 && div_magic((unsigned)id2, per_magic) == p);
                }
                if (first) atomicAdd(&s_part[p], 1);
            }
        }
    }
}

// Stable ranks of one warp's run [w0, w1) of a token range's flat (t, k) indices, the range
// starting at token t0; hist holds the warp's next row per expert and is advanced.  Writes
// row_of, src_info and expert_ids; a row at or past row_limit (the layout's row capacity) is
// not recorded and its pair gets row_of -1.  The (token, slot) of each lane's index is carried
// from chunk to chunk by adding 32 with a carry, so there is one division per lane, not per id.
__device__ __forceinline__ void rank_and_write(const int *s_ids, int w0, int w1, int t0, int K,
                                               int row_limit, int nbits, int *hist, int32_t *row_of,
                                               int32_t *src_info, int32_t *expert_ids,
                                               const int32_t *status) {
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    int tk = (w0 + lane) / K, kk = (w0 + lane) - tk * K;
    const int step_t = 32 / K, step_k = 32 - step_t * K;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const int id = i < w1 ? s_ids[i] : -1;
        const unsigned peers = same_key_lanes((unsigned)(id + 1), nbits);
        int row = -1;
        if (id >= 0) row = hist[id] + __popc(peers & lt_mask);
        __syncwarp();
        if (id >= 0 && lane == __ffs(peers) - 1) hist[id] += __popc(peers);
        __syncwarp();
        if (i < w1) {
            if (kBoundsCheck && id >= 0 && row < 0) bounds_fail(status);
            if (row >= row_limit || row < 0) row = -1;
            row_of[(size_t)t0 * K + i] = row;
            if (row >= 0) {
                reinterpret_cast<int2 *>(src_info)[row] = make_int2(t0 + tk, kk);
                expert_ids[row] = id;
            }
        }
        tk += step_t;
        kk += step_k;
        if (kk >= K) {
            kk -= K;
            ++tk;
        }
    }
}

// Dynamic shared memory of the count kernel: histogram, partition counts and the tile's ids,
// or the last CTA's scan buffer, whichever is larger.
inline size_t count_smem_bytes(int E, int P, int tt, int K) {
    const size_t a = (size_t)E + P + (size_t)tt * K;
    const size_t b = (size_t)kScanChunk + kScanChunk / 32;
    return sizeof(int) * (a > b ? a : b);
}

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
                       int pad, int row_limit, int tile_t, int nTiles, unsigned long long per_magic,
                       int one_wave, Workspace ws, int32_t *__restrict__ row_offsets,
                       int32_t *__restrict__ part_tokens, int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    int *s_hist = smem;          // [E]
    int *s_part = smem + E;      // [P]
    int *s_ids = smem + E + P;   // [tile_t * K], invalid ids replaced by -1
    __shared__ int s_bad;
    __shared__ int s_last;
    __shared__ int s_warp[kLayoutWarps];

    pdl_begin_if(one_wave);
    const int tid = threadIdx.x, lane = tid & 31;
    const int j = blockIdx.x;
    const int t0 = j * tile_t;
    const int t1 = min(T, t0 + tile_t);
    const int n = max(0, t1 - t0) * K;
    const int32_t *tid_ids = ids + (size_t)t0 * K;
    int bad = 0;
#pragma unroll 8
    for (int i = tid; i < n; i += blockDim.x) {   // all of a thread's loads in flight together
        int id = tid_ids[i];
        if (bad_id(id, E)) {
            bad = 1;
            id = -1;
        }
        s_ids[i] = id;
    }
    for (int e = tid; e < E; e += blockDim.x) s_hist[e] = 0;
    for (int p = tid; p < P; p += blockDim.x) s_part[p] = 0;
    bad = __syncthreads_or(bad);
    if (tid == 0) s_bad = bad;

    // Expert histogram (shared-memory atomics) and tokens per partition.
    for (int i = tid; i < n; i += blockDim.x) {
        const int id = s_ids[i];
        if (id >= 0) atomicAdd(&s_hist[id], 1);
    }
    count_partition_tokens(s_ids, max(0, t1 - t0), K, per_magic, P, s_part);
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

    // Padding: each expert's padding rows follow its last tile's rows, so they are added to
    // that tile's count before the scan (the scan is exclusive: the tile's own base is unchanged).
    if (pad > 1) {
        for (int e = tid; e < E; e += blockDim.x) {
            int tot = 0;
#pragma unroll 8
            for (int jj = 0; jj < nTiles; ++jj) tot += __ldcg(ws.cnt + (size_t)e * nTiles + jj);
            const int extra = (tot + pad - 1) / pad * pad - tot;
            if (extra) ws.cnt[(size_t)e * nTiles + nTiles - 1] = __ldcg(ws.cnt + (size_t)e * nTiles + nTiles - 1) + extra;
        }
        __syncthreads();
    }

    // Exclusive scan of cnt in place, kScanChunk entries per pass, through shared memory
    // (padded by one word per 32 so each thread's contiguous segment is conflict-free).  All
    // of a pass's loads are issued before the first is used, so a pass costs about one L2
    // round trip instead of one per entry.
    int *s_chunk = smem;   // reuses the histogram space: kScanChunk + kScanChunk/32 ints
    const long total_n = (long)E * nTiles;
    constexpr int kPer = kScanChunk / kLayoutThreads;
    int carry = 0;
    for (long c0 = 0; c0 < total_n; c0 += kScanChunk) {
        const int len = (int)min((long)kScanChunk, total_n - c0);
        int v[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = q * kLayoutThreads + tid;
            v[q] = i < len ? __ldcg(ws.cnt + c0 + i) : 0;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = q * kLayoutThreads + tid;
            s_chunk[i + (i >> 5)] = v[q];
        }
        __syncthreads();
        int sum = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = tid * kPer + q;
            sum += s_chunk[i + (i >> 5)];
        }
        int tot;
        int run = carry + block_exclusive_scan(sum, s_warp, tot);
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = tid * kPer + q;
            const int c = s_chunk[i + (i >> 5)];
            s_chunk[i + (i >> 5)] = run;
            run += c;
        }
        __syncthreads();
        // row_offsets[e] is the scanned value at (e, tile 0).
        for (int e = tid; e < E; e += blockDim.x) {
            const long f = (long)e * nTiles - c0;
            if (f >= 0 && f < len) row_offsets[e] = s_chunk[f + (f >> 5)];
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = q * kLayoutThreads + tid;
            if (i < len) ws.cnt[c0 + i] = s_chunk[i + (i >> 5)];
        }
        carry += tot;
        __syncthreads();
    }
    const long long rows_needed = (long long)carry + (S ? (long long)(T + pad - 1) / pad * pad : 0);
    if (tid == 0) {
        row_offsets[E] = carry;
        if (S) row_offsets[E + 1] = (int)rows_needed;
    }
    // Partition totals against the capacity (one warp per partition, lanes over the tiles),
    // and the bad-id flags.
    int flags = 0;
    for (int p = tid >> 5; p < P; p += kLayoutWarps) {
        int s = 0;
#pragma unroll 4
        for (int jj = lane; jj < nTiles; jj += 32) s += __ldcg(ws.part + (size_t)p * nTiles + jj);
        s = __reduce_add_sync(kFullMask, s);
        if (lane == 0) {
            part_tokens[p] = s;
            if (s > C) flags |= EP_STATUS_OVERFLOW;
        }
    }
    for (int jj = tid; jj < nTiles; jj += blockDim.x)
        if (__ldcg(ws.tile_flags + jj)) flags |= EP_STATUS_BAD_EXPERT;
    if (rows_needed > row_limit) flags |= EP_STATUS_OVERFLOW;   // the row capacity
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
ep_layout_rank_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int S, int pad,
                      int row_limit, int tile_t, int nTiles, int nbits, int one_wave,
                      const int32_t *__restrict__ cnt,
                      const int32_t *__restrict__ row_offsets, int32_t *__restrict__ row_of,
                      int32_t *__restrict__ src_info, int32_t *__restrict__ expert_ids,
                      const int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    int *s_whist = smem;                       // [kLayoutWarps][E]
    int *s_ids = smem + kLayoutWarps * E;      // [tile_t * K]
    pdl_begin_if(one_wave);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = blockIdx.x;
    const int t0 = j * tile_t;
    const int t1 = min(T, t0 + tile_t);
    const int n = max(0, t1 - t0) * K;

    // The tile's scanned bases (one per expert), loaded before they are needed.
    constexpr int kMaxEPerThread = kMaxE / kLayoutThreads;
    int base_e[kMaxEPerThread];
#pragma unroll
    for (int q = 0; q < kMaxEPerThread; ++q) {
        const int e = tid + q * kLayoutThreads;
        base_e[q] = e < E ? cnt[(size_t)e * nTiles + j] : 0;
    }
#pragma unroll 8
    for (int i = tid; i < n; i += blockDim.x) {
        int id = ids[(size_t)t0 * K + i];
        s_ids[i] = bad_id(id, E) ? -1 : id;
    }
    for (int i = tid; i < kLayoutWarps * E; i += blockDim.x) s_whist[i] = 0;
    __syncthreads();

    // Each warp owns one contiguous run of the tile's flat (t, k) indices.
    const int per_warp = ((n + kLayoutWarps - 1) / kLayoutWarps + 31) / 32 * 32;
    const int w0 = min(n, warp * per_warp), w1 = min(n, w0 + per_warp);
    int *hist = s_whist + warp * E;
    for (int i = w0 + lane; i < w1; i += 32) {
        const int id = s_ids[i];
        if (id >= 0) atomicAdd(&hist[id], 1);
    }
    __syncthreads();
    // First row of each (warp, expert): the tile's scanned base plus earlier warps' counts.
    // The last tile also writes each expert's padding rows: from the end of its routed rows
    // to the next group's first row.
    const bool last_tile = j == nTiles - 1;
#pragma unroll
    for (int q = 0; q < kMaxEPerThread; ++q) {
        const int e = tid + q * kLayoutThreads;
        if (e >= E) break;
        int run = base_e[q];
        for (int w = 0; w < kLayoutWarps; ++w) {
            int c = s_whist[w * E + e];
            s_whist[w * E + e] = run;
            run += c;
        }
        if (pad > 1 && last_tile) {
            const int end = min(row_offsets[e + 1], row_limit);
            for (int r = run; r < end; ++r) {
                reinterpret_cast<int2 *>(src_info)[r] = make_int2(-1, -1);
                expert_ids[r] = e;
            }
        }
    }
    __syncthreads();
    rank_and_write(s_ids, w0, w1, t0, K, row_limit, nbits, hist, row_of, src_info, expert_ids, status);
    if (S) {
        const int rs = row_offsets[E];
        for (int t = t0 + tid; t < t1 && rs + t < row_limit; t += blockDim.x) {
            reinterpret_cast<int2 *>(src_info)[rs + t] = make_int2(t, K);
            expert_ids[rs + t] = E;
        }
        if (pad > 1 && last_tile) {
            const int end = min(row_offsets[E + 1], row_limit);
            for (int r = rs + T + tid; r < end; r += blockDim.x) {
                reinterpret_cast<int2 *>(src_info)[r] = make_int2(-1, -1);
                expert_ids[r] = E;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// Single-cluster layout.  When one thread-block cluster can hold every id, the whole layout is
// one kernel on a cluster of up to 16 CTAs, each on its own SM and each owning a contiguous range
// of tokens.  Per CTA:
//   A. load the range's ids into shared memory (bad ids become -1; with at most 32 partitions a
//      per-token partition bitmask is built on the way), per-warp expert histograms;
//   B. one thread per expert walks the 32 per-warp counts, giving each warp's first local row
//      per expert and the CTA's count per expert; partition token counts from the bitmasks (one
//      reduction per partition);
//   C. each CTA pushes its expert counts into every CTA's shared memory (one warp per
//      destination, 16-byte stores), and its partition counts and bad-id flag into CTA 0's,
//      through distributed shared memory, then arrives at the cluster barrier.  Before waiting
//      it does all its local work: its first local position per expert (a block scan), the
//      stable rank of each routed (t, k) within its expert (equal-id lanes by ballots), and the
//      staging of each routed row in shared memory in expert order;
//   D. after the wait every read is local: cluster totals -> row_offsets (a block scan), counts
//      of the CTAs before this one -> this CTA's first row per expert; then row_of in flat order,
//      and src_info / expert_ids from the staging area as contiguous runs.
// One launch, one cluster barrier after start-up, no global scratch, atomics or fences.  A CTA
// holds up to kClMaxIds ids, so one cluster lays out up to 262,144 (token, slot) pairs.  When
// the NVFP4 dispatch of the same call writes src_info and expert_ids (write_rows 0), the
// staging and its copy-out are skipped and only row_of is written in phase D.
// ---------------------------------------------------------------------------------------
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
static_assert(kClWarps == 32, "the cluster kernel scans per-warp values with one warp");
constexpr int kClMaxCtas = 16;            // largest cluster (non-portable; 8 where 16 is refused)
constexpr int kClMaxIds = 16384;          // ids of one CTA's range held in shared memory
constexpr int kClIdBatch = 8;             // ids a lane requests before using the first
constexpr int kClIdsPerCta = 2048;        // below this many ids per CTA, use fewer CTAs
static_assert(kMaxE <= kClThreads, "the cluster kernel gives one thread to each expert");
constexpr size_t kClMaxSmem = 216 * 1024;   // dynamic; leaves room for the static arrays

// Shared-memory plan of the cluster kernel (ints): per-expert arrays, the pushed counts of every
// CTA, partition counts pushed to CTA 0, per-warp histograms, the ids, the staging area and the
// per-token partition masks.
struct ClusterSmem {
    int hist, first, locoff, all, part_all, bad_all, whist, ids, stage, tokmask, total;
};
__host__ __device__ inline ClusterSmem cluster_smem_plan(int E, int P, int tile_t, int K) {
    ClusterSmem m;
    int o = 0;
    m.hist = o; o += E;
    m.first = o; o += E;
    m.locoff = o; o += E;
    m.all = o; o += kClMaxCtas * E;
    m.part_all = o; o += kClMaxCtas * P;
    m.bad_all = o; o += kClMaxCtas;
    m.whist = o; o += kClWarps * (E + 1);   // rows padded to E + 1: conflict-free scans
    m.ids = o; o += tile_t * K;
    m.stage = o; o += tile_t * K;
    m.tokmask = o; o += tile_t;
    m.total = o;
    return m;
}
inline size_t cluster_smem_bytes(int E, int P, int tile_t, int K) {
    return sizeof(int) * (size_t)cluster_smem_plan(E, P, tile_t, K).total;
}

// CTAs of the single-cluster layout for these sizes (at most max_ctas), or 0 when it cannot
// hold them.
inline int cluster_ctas(int T, int K, int E, int P, int max_ctas) {
    const long n = (long)T * K;
    long c = (n + kClIdsPerCta - 1) / kClIdsPerCta;
    if (c < 1) c = 1;
    if (c > max_ctas) c = max_ctas;
    const long per = (T + c - 1) / c;
    if (per * K > kClMaxIds) return 0;
    if (cluster_smem_bytes(E, P, (int)per, K) > kClMaxSmem) return 0;
    return (int)c;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }

// Exclusive scan of one value per thread over a 1024-thread block, in thread order: shuffles
// within each warp, then one warp over the warp totals.  warp_tot holds 32 ints; every thread
// gets the block total.  Starts and ends with the block in step (two barriers).
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    if (warp == 0) {
        const int w0 = warp_tot[lane];
        int wi = w0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFullMask, wi, o);
            if (lane >= o) wi += u;
        }
        warp_tot[lane] = wi - w0;   // exclusive warp offsets; the total goes in slot 32
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    before = warp_tot[warp];
    total = warp_tot[32];
    return before + incl - v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kClThreads, 1)
ep_layout_cluster_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int P, int C, int S,
                         int pad, int row_limit, int tile_t, int nbits, unsigned long long per_magic,
                         unsigned long long k_magic, int write_rows, int32_t *__restrict__ row_offsets,
                         int32_t *__restrict__ expert_ids, int32_t *__restrict__ src_info,
                         int32_t *__restrict__ row_of, int32_t *__restrict__ part_tokens,
                         int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    const ClusterSmem m = cluster_smem_plan(E, P, tile_t, K);
    int *s_hist = smem + m.hist, *s_first = smem + m.first, *s_locoff = smem + m.locoff;
    int *s_all = smem + m.all, *s_part_all = smem + m.part_all, *s_bad_all = smem + m.bad_all;
    int *s_whist = smem + m.whist, *s_ids = smem + m.ids, *s_stage = smem + m.stage;
    int *s_tokmask = smem + m.tokmask;
    __shared__ int s_warp[kClWarps + 1];    // warp totals of the block scans (+ the block total)
    __shared__ int s_warp2[kClWarps + 1];
    __shared__ int s_bad;
    __shared__ int s_nvalid;
    __shared__ int s_bounds;   // a failed index check of the bounds-checked build

    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int ncta = (int)cluster.num_blocks();
    cluster_arrive_relaxed();   // "this CTA has started"; waited on before the first remote write
    pdl_begin();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = crank * tile_t;
    const int t1 = min(T, t0 + tile_t);
    const int ntok = max(0, t1 - t0);
    const int n = ntok * K;
    const bool masks = P <= 32;

    // A. ids, per-token partition masks, per-warp histograms (row stride E + 1)
    const int EP = E + 1;
    for (int i = tid; i < kClWarps * EP; i += kClThreads) s_whist[i] = 0;
    if (masks)
        for (int i = tid; i < ntok; i += kClThreads) s_tokmask[i] = 0;
    if (tid == 0) {
        s_bad = 0;
        s_bounds = 0;
    }
    __syncthreads();
    const int per_warp = ((n + kClWarps - 1) / kClWarps + 31) / 32 * 32;
    const int w0 = min(n, warp * per_warp), w1 = min(n, w0 + per_warp);
    int *hist = s_whist + warp * EP;
    {
        int bad = 0;
        // the warp's own run, so its histogram needs no second pass over shared memory; a
        // lane's ids are requested kClIdBatch at a time before the first of them is used (one
        // batch covers up to 8192 ids per CTA)
        int tk = (w0 + lane) / K, kk = (w0 + lane) - tk * K;
        const int step_t = 32 / K, step_k = 32 - step_t * K;
        for (int i0 = w0 + lane; i0 < w1; i0 += 32 * kClIdBatch) {
            int idv[kClIdBatch];
#pragma unroll
            for (int j = 0; j < kClIdBatch; ++j) {
                const int i = i0 + 32 * j;
                idv[j] = i < w1 ? ids[(size_t)t0 * K + i] : -1;
            }
#pragma unroll
            for (int j = 0; j < kClIdBatch; ++j) {
                const int i = i0 + 32 * j;
                if (i >= w1) break;
                int id = idv[j];
                if (bad_id(id, E)) {
                    bad = 1;
                    id = -1;
                }
                s_ids[i] = id;
                if (id >= 0) {
                    atomicAdd(&hist[id], 1);
                    if (masks) atomicOr(&s_tokmask[tk], (int)(1u << div_magic((unsigned)id, per_magic)));
                }
                tk += step_t;
                kk += step_k;
                if (kk >= K) {
                    kk -= K;
                    ++tk;
                }
            }
        }
        if (bad) s_bad = 1;
    }
    if (!masks)
        for (int p = tid; p < P; p += kClThreads) s_part_all[crank * P + p] = 0;   // local scratch row
    __syncthreads();

    // B. per-(warp, expert) exclusive prefix over the 32 warps, and the CTA's count per expert:
    //    thread e < E walks expert e's per-warp counts, eight independent shared loads at a time.
    if (tid < E) {
        int run = 0;
#pragma unroll
        for (int h = 0; h < kClWarps; h += 8) {
            int c[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) c[w] = s_whist[(h + w) * EP + tid];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                s_whist[(h + w) * EP + tid] = run;
                run += c[w];
            }
        }
        s_hist[tid] = run;
    }
    //    tokens per partition: warp w counts partitions w, w + 32, ... from the token masks
    if (masks) {
        for (int p = warp; p < P; p += kClWarps) {
            int c = 0;
            for (int tl = lane; tl < ntok; tl += 32) c += (s_tokmask[tl] >> p) & 1;
            c = __reduce_add_sync(kFullMask, c);
            if (lane == 0) s_part_all[crank * P + p] = c;
        }
    } else {
        count_partition_tokens(s_ids, ntok, K, per_magic, P, s_part_all + crank * P);
    }
    __syncthreads();

    // C. push this CTA's counts through distributed shared memory (warp r writes them into CTA
    //    r), its partition counts and bad-id flag into CTA 0's, then arrive at the cluster barrier.
    cluster_wait();   // every CTA of the cluster has started
    for (int r = warp; r < ncta; r += kClWarps) {
        int *dst = cluster.map_shared_rank(s_all, r) + crank * E;
        if ((E & 3) == 0) {   // 16-byte aligned rows (the plan's offsets are multiples of E)
            const int4 *src4 = reinterpret_cast<const int4 *>(s_hist);
            int4 *dst4 = reinterpret_cast<int4 *>(dst);
            for (int e4 = lane; e4 < E / 4; e4 += 32) dst4[e4] = src4[e4];
        } else {
            for (int e = lane; e < E; e += 32) dst[e] = s_hist[e];
        }
    }
    if (crank != 0) {
        int *rp = cluster.map_shared_rank(s_part_all, 0);
        for (int p = tid; p < P; p += kClThreads) rp[crank * P + p] = s_part_all[crank * P + p];
    }
    if (tid == 0) cluster.map_shared_rank(s_bad_all, 0)[crank] = s_bad;
    cluster_arrive();   // release: the pushes are visible to every CTA after its wait

    //    While the other CTAs arrive, everything local: this CTA's first local position per
    //    expert (an exclusive scan of its counts), the stable rank of every routed (t, k) in its
    //    expert's local list (equal-id lanes by ballots), and its staging at that expert-major
    //    local position (flat index in the low bits, expert in the high bits).  s_ids keeps
    //    (local rank << 10 | expert) for the rows written after the wait.
    if (write_rows) {
        int tot_l;
        const int v = tid < E ? s_hist[tid] : 0;
        const int ex = block_exclusive_scan_1024(v, s_warp2, tot_l);
        if (tid < E) s_locoff[tid] = ex;
        if (tid == 0) s_nvalid = tot_l;
        __syncthreads();
    }
    {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = w0; base < w1; base += 32) {
            const int i = base + lane;
            const int id = i < w1 ? s_ids[i] : -1;
            const unsigned peers = same_key_lanes((unsigned)(id + 1), nbits);
            int local = -1;
            if (id >= 0) local = hist[id] + __popc(peers & lt_mask);
            __syncwarp();
            if (id >= 0 && lane == __ffs(peers) - 1) hist[id] += __popc(peers);
            __syncwarp();
            if (id >= 0) {
                if (write_rows) {
                    const int pos = s_locoff[id] + local;
                    if (!kBoundsCheck || (pos >= 0 && pos < n)) s_stage[pos] = (id << 16) | i;
                    else s_bounds = 1;
                }
                s_ids[i] = (local << 10) | id;
            }
        }
    }
    cluster_wait();   // acquire: every CTA's counts are in s_all

    //    cluster totals per expert (thread e owns expert e) and their extents: each total padded
    //    to the next multiple of pad; the counts of the CTAs before this one
    int before = 0, total = 0;
    if (tid < E) {
#pragma unroll
        for (int r = 0; r < kClMaxCtas; ++r) {
            if (r < ncta) {
                const int v = s_all[r * E + tid];
                if (r < crank) before += v;
                total += v;
            }
        }
    }
    const int ext = pad > 1 ? (total + pad - 1) / pad * pad : total;
    //    CTA 0: partition totals against the capacity, and the bad-id flags (status bits kept
    //    above bit 4 of s_bad, whose low bit is this CTA's own bad-id flag)
    if (crank == 0) {
        int f = 0;
        for (int p = tid; p < P; p += kClThreads) {
            int c = 0;
            for (int r = 0; r < ncta; ++r) c += s_part_all[r * P + p];
            part_tokens[p] = c;
            if (c > C) f |= EP_STATUS_OVERFLOW;
        }
        if (tid < ncta && s_bad_all[tid]) f |= EP_STATUS_BAD_EXPERT;
        if (f) atomicOr(&s_bad, f << 4);
    }
    int routed;
    const int excl = block_exclusive_scan_1024(ext, s_warp, routed);   // ends with a barrier
    const int n_valid = write_rows ? s_nvalid : 0;
    const int shared_ext = S ? (pad > 1 ? (T + pad - 1) / pad * pad : T) : 0;
    if (tid < E) {
        if (crank == 0) row_offsets[tid] = excl;
        s_first[tid] = excl + before;
        // padding rows of expert tid, spread over the cluster's CTAs
        for (int r = excl + total + crank; write_rows && r < excl + ext && r < row_limit; r += ncta) {
            reinterpret_cast<int2 *>(src_info)[r] = make_int2(-1, -1);
            expert_ids[r] = tid;
        }
    }
    if (crank == 0 && tid == 0) {
        int flags = s_bad >> 4;
        if ((long long)routed + shared_ext > row_limit) flags |= EP_STATUS_OVERFLOW;   // row capacity
        row_offsets[E] = routed;
        if (S) row_offsets[E + 1] = routed + shared_ext;
        *status = flags;
    }
    __syncthreads();

    // D. rows: row_of in flat order (-1 for an unused slot or a row at or past the row
    //    capacity), then src_info / expert_ids from the staging area in contiguous runs.
    for (int i = tid; i < n; i += kClThreads) {
        const int v = s_ids[i];
        int row = -1;
        if (v >= 0) {
            if (kBoundsCheck && (v & 1023) >= E) {
                s_bounds = 1;
            } else {
                row = s_first[v & 1023] + (v >> 10);
                if (kBoundsCheck && row < 0) s_bounds = 1;
                if (row >= row_limit || row < 0) row = -1;
            }
        }
        row_of[(size_t)t0 * K + i] = row;
    }
    for (int j = tid; write_rows && j < n_valid; j += kClThreads) {
        const int v = s_stage[j];
        const int e = v >> 16, i = v & 0xffff;
        if (e < 0 || e >= E || i >= n) {   // only a layout raced by a writer of ids
            if (kBoundsCheck) s_bounds = 1;
            continue;
        }
        const int row = s_first[e] + (j - s_locoff[e]);
        if (row < 0 || row >= row_limit) {   // at or past the row capacity: not recorded
            if (kBoundsCheck && row < 0) s_bounds = 1;
            continue;
        }
        const int tk = div_magic((unsigned)i, k_magic);
        reinterpret_cast<int2 *>(src_info)[row] = make_int2(t0 + tk, i - tk * K);
        expert_ids[row] = e;
    }
    if (S && write_rows) {
        for (int t = t0 + tid; t < t1 && routed + t < row_limit; t += kClThreads) {
            reinterpret_cast<int2 *>(src_info)[routed + t] = make_int2(t, K);
            expert_ids[routed + t] = E;
        }
        // the shared group's padding rows, spread over the cluster's CTAs
        const int end = min(routed + shared_ext, row_limit);
        for (int r = routed + T + crank * kClThreads + tid; r < end; r += ncta * kClThreads) {
            reinterpret_cast<int2 *>(src_info)[r] = make_int2(-1, -1);
            expert_ids[r] = E;
        }
    }
    if (kBoundsCheck) {   // after CTA 0 has stored the status word, every CTA adds its failures
        __syncthreads();
        cluster_sync_all();
        if (tid == 0 && s_bounds) bounds_fail(status);
    }
}

// Largest cluster the device runs for the layout kernel: 16 CTAs where the non-portable size is
// granted, else 8 (the portable size); 0 when the kernel cannot get its shared memory (the
// layout then takes the two-kernel path).  The kernel's attributes are set and the answer looked
// up once per device, so later calls (and calls inside a stream capture) only launch.
inline int max_cluster_ctas() {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev];   // 0: not looked up; else the answer + 1
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < kMaxDev;
    std::lock_guard<std::mutex> lock(mu);
    if (cacheable && cached[dev]) return cached[dev] - 1;
    int best = 0;
    if (cudaFuncSetAttribute(ep_layout_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kClMaxSmem) == cudaSuccess) {
        best = 8;
        if (cudaFuncSetAttribute(ep_layout_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16);
            cfg.blockDim = dim3(kClThreads);
            cfg.dynamicSmemBytes = kClMaxSmem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 16;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, ep_layout_cluster_kernel, &cfg) == cudaSuccess && n > 0)
                best = 16;
        }
    }
    (void)cudaGetLastError();
    if (cacheable) cached[dev] = best + 1;
    return best;
}

// The whole layout as one cluster of CTAs (see ep_layout_cluster_kernel).  Returns -1 when the
// sizes do not fit one cluster (the caller then uses the two-kernel path).  With write_rows 0
// (unpadded layouts only) the kernel writes row_offsets, row_of, part_tokens and the status but
// leaves src_info and expert_ids to the dispatch kernel that follows it.
inline int launch_cluster_layout(const int32_t *ids, int T, int K, int E, int P, int C, int S,
                                 int pad, int row_limit, ep_layout_t *L, cudaStream_t st,
                                 int *ctas_used, int write_rows = 1) {
    const int max_ctas = max_cluster_ctas();
    if (max_ctas == 0) return -1;   // the two-kernel path needs no shared-memory opt-in
    const int ncta = cluster_ctas(T, K, E, P, max_ctas);
    if (ncta == 0) return -1;
    *ctas_used = ncta;
    const int tile_t = (T + ncta - 1) / ncta;
    const size_t smem = cluster_smem_bytes(E, P, tile_t, K);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return launch_result(cudaLaunchKernelEx(&cfg, ep_layout_cluster_kernel, ids, T, K, E, P, C, S,
                                            pad, row_limit, tile_t, key_bits(E + 1), magic_of(E / P),
                                            magic_of(K), write_rows,
                                            L->row_offsets, L->expert_ids, L->src_info, L->row_of,
                                            L->part_tokens, L->status));
}

}  // namespace
}  // namespace ep

using namespace ep;

namespace ep {
namespace {

// The two-kernel layout (count + scan, then rank) with its scratch at `scratch`, which holds at
// least workspace_bytes(nTiles, E) bytes whose ticket word is zero.
int launch_tiled_layout(const int32_t *topk_ids, int T, int K, int E, int P, int capacity, int S,
                        int pad, int row_limit, void *scratch, ep_layout_t *L, cudaStream_t st) {
    const int tt = tile_tokens(T, K);
    const int nTiles = num_tiles(T, tt);
    const int wave = one_wave(nTiles);
    Workspace ws = carve(scratch, nTiles, E);
    const size_t smem_count = count_smem_bytes(E, P, tt, K);
    int rc = launch_pdl(ep_layout_count_kernel, dim3(nTiles), dim3(kLayoutThreads), smem_count, st,
                        topk_ids, T, K, E, P, capacity, S, pad, row_limit, tt, nTiles,
                        magic_of(E / P), wave, ws, L->row_offsets, L->part_tokens, L->status);
    if (rc != EP_OK) return rc;
    size_t smem_rank = sizeof(int) * ((size_t)kLayoutWarps * E + (size_t)tt * K);
    if (smem_rank > 48 * 1024 &&
        cudaFuncSetAttribute(ep_layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_rank) != cudaSuccess)
        return EP_ERR_CUDA;
    return launch_pdl(ep_layout_rank_kernel, dim3(nTiles), dim3(kLayoutThreads), smem_rank, st,
                      topk_ids, T, K, E, S, pad, row_limit, tt, nTiles, key_bits(E + 1), wave,
                      (const int32_t *)ws.cnt, (const int32_t *)L->row_offsets, L->row_of,
                      L->src_info, L->expert_ids, (const int32_t *)L->status);
}

}  // namespace
}  // namespace ep

extern "C" size_t ep_layout_workspace_bytes(int T, int K, int n_experts, int fused_shared) {
    if (!sizes_ok(T, K, n_experts, fused_shared)) return 0;
    int tt = tile_tokens(T, K);
    return workspace_bytes(num_tiles(T, tt), n_experts);
}

namespace ep {

int layout_cluster_plan(int T, int K, int E, int P) {
    if (!sizes_ok(T, K, E, 0) || P < 1 || P > E || E % P != 0) return 0;
    const int max_ctas = max_cluster_ctas();
    return max_ctas ? cluster_ctas(T, K, E, P, max_ctas) : 0;
}

// Validates the arguments of a layout call and enqueues it.  *cluster_ctas_used receives the
// number of SMs the single-cluster kernel occupies (0 when the two-kernel path ran).
int launch_layout(const int32_t *topk_ids, int T, int K, int E, int P, int capacity, int S,
                  int pad, int row_capacity, ep_layout_t *L, cudaStream_t st,
                  int *cluster_ctas_used, int write_rows) {
    if (cluster_ctas_used) *cluster_ctas_used = 0;
    if (!L || !sizes_ok(T, K, E, S) || !padding_ok(T, K, E, S, pad, row_capacity))
        return EP_ERR_INVALID_ARG;
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
    L->pad_multiple = pad;
    L->row_capacity = row_capacity;
    const int row_limit = layout_rows(L);

    int used = 0;
    const int rc_cl = launch_cluster_layout(topk_ids, T, K, E, P, capacity, S, pad, row_limit, L,
                                            st, &used, pad > 1 || row_capacity > 0 ? 1 : write_rows);
    if (rc_cl != -1) {
        if (cluster_ctas_used) *cluster_ctas_used = used;
        return rc_cl;
    }
    return launch_tiled_layout(topk_ids, T, K, E, P, capacity, S, pad, row_limit, L->workspace, L, st);
}

}  // namespace ep

extern "C" int ep_dispatch_layout(const int32_t *topk_ids, int T, int K, int n_experts,
                                  int n_parts, int capacity, int fused_shared, ep_layout_t *L,
                                  void *stream) {
    EP_NVTX_RANGE("ep_dispatch_layout");
    return launch_layout(topk_ids, T, K, n_experts, n_parts, capacity, fused_shared, 1, 0, L,
                         as_stream(stream), nullptr);
}

extern "C" size_t ep_rows_max(int T, int K, int n_experts, int fused_shared, int pad_multiple,
                              int num_permuted_tokens) {
    if (!sizes_ok(T, K, n_experts, fused_shared) || num_permuted_tokens < 0) return 0;
    const int pad = pad_multiple < 1 ? 1 : pad_multiple;
    if (!padding_ok(T, K, n_experts, fused_shared, pad, num_permuted_tokens)) return 0;
    return (size_t)rows_max(T, K, n_experts, fused_shared, pad, num_permuted_tokens);
}

extern "C" int ep_dispatch_layout_routed(const int32_t *topk_ids, const uint8_t *routing_map,
                                         const float *dense_probs, int T, int K, int n_experts,
                                         int n_parts, int capacity, int fused_shared,
                                         int pad_multiple, int num_permuted_tokens,
                                         int32_t *map_topk_ids, float *map_topk_probs,
                                         ep_layout_t *L, void *stream) {
    EP_NVTX_RANGE("ep_dispatch_layout_routed");
    cudaStream_t st = as_stream(stream);
    const int32_t *ids = topk_ids;
    if (routing_map) {   // the map takes precedence: convert it, then lay out its compact form
        if (!L || !sizes_ok(T, K, n_experts, fused_shared) ||
            !padding_ok(T, K, n_experts, fused_shared, pad_multiple, num_permuted_tokens))
            return EP_ERR_INVALID_ARG;
        const int rc = launch_map_to_topk(routing_map, dense_probs, T, n_experts, K, map_topk_ids,
                                          map_topk_probs, st);
        if (rc != EP_OK) return rc;
        ids = map_topk_ids;
    }
    return launch_layout(ids, T, K, n_experts, n_parts, capacity, fused_shared, pad_multiple,
                         num_permuted_tokens, L, st, nullptr);
}

extern "C" int ep_read_status(const ep_layout_t *L, void *stream, int32_t *host_status) {
    EP_NVTX_RANGE("ep_read_status");
    if (!L || !L->status || !host_status) return EP_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, L->status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return EP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    *host_status = v;
    if (v & EP_STATUS_BOUNDS) return EP_ERR_BOUNDS;
    if (v & EP_STATUS_OVERFLOW) return EP_ERR_OVERFLOW;
    if (v & EP_STATUS_BAD_EXPERT) return EP_ERR_BAD_EXPERT;
    return EP_OK;
}

extern "C" const char *ep_strerror(int code) {
    switch (code) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_OVERFLOW:
            return "a logical partition received more tokens than its capacity, or the rows "
                   "exceeded the layout's row capacity";
        case EP_ERR_BAD_EXPERT: return "an expert id was outside [-1, n_experts)";
        case EP_ERR_CUDA: return "CUDA error";
        case EP_ERR_TOO_LARGE: return "the sizes need more scratch than the fixed no-allocation array holds";
        case EP_ERR_BOUNDS:
            return "an index fell outside its buffer and the access was skipped (bounds-checked build)";
        default: return "unknown error";
    }
}

// ---------------------------------------------------------------------------------------
// ep_dispatch_layout_noalloc: the same layout with its scratch in a fixed device array.
//
// For callers that must not allocate device memory at all: code running under a framework
// whose caching allocator owns the whole device, latency-critical paths where an allocation
// (and the device synchronisation cudaMalloc/cudaFree can imply) is not acceptable, or
// runtimes that hand a library only its inputs and outputs.  Sizes that fit one thread-block
// cluster run the single-cluster kernel, which needs no scratch.  Larger sizes run the two-kernel
// layout with its scratch in a file-scope __device__ array of kNoAllocWorkspaceBytes that every
// GPU which loads this library keeps until the process exits.  Host code cannot use the array's
// name as a device address (on the host it is only a stand-in symbol), so the device address is
// looked up once per device with cudaGetSymbolAddress, with that device current, during the
// first call on that device.  That first call also zeroes the ticket word; every later call leaves it at zero
// when it finishes.  All calls share the one array, so calls whose work overlaps on the GPU
// (other streams, other threads) race on it.
// ---------------------------------------------------------------------------------------

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
    EP_NVTX_RANGE("ep_dispatch_layout_noalloc");
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
    L->pad_multiple = 1;
    L->row_capacity = 0;
    const int row_limit = layout_rows(L);

    cudaStream_t st = as_stream(stream);
    // Sizes that fit one thread-block cluster need no scratch at all: the single-cluster kernel
    // exchanges its counts through distributed shared memory.
    int used = 0;
    rc = launch_cluster_layout(topk_ids, T, K, E, P, capacity, S, 1, row_limit, L, st, &used);
    if (rc != -1) return rc;
    return launch_tiled_layout(topk_ids, T, K, E, P, capacity, S, 1, row_limit, scratch, L, st);
}
