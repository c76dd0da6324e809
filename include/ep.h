/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE token dispatch / combine library (libep_gb300.so).
 *
 * One GPU, one HBM buffer.  Dispatch turns each token's top-k expert ids into an expert-major
 * layout and scatters the token rows into it (BF16, or NVFP4 with a per-token global scale);
 * combine gathers the expert outputs back into token order with the routing probabilities as
 * weights; the two backward passes are the same operations with the roles swapped.
 *
 * Pages this interface follows (cited per entry point by page and section):
 *   fused_a2a        -- NeMo AutoModel v0.4 API, nemo_automodel.components.moe.megatron.fused_a2a
 *   token_dispatcher -- NeMo AutoModel v0.7 API, ...components.moe.megatron.token_dispatcher
 *   Mojo EP dispatch -- Modular MAX API, struct DistributedEPDispatchBlockScaledNVDynGlobalScales
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Pointers.  Every tensor argument is a DEVICE pointer into memory the caller allocated (for
 *   example with PyTorch); the library allocates nothing on these paths and keeps no pointer
 *   after a call returns.  Tensors are dense and row-major.  bf16 tensors are passed as
 *   uint16_t (the IEEE bfloat16 bit pattern).  Every tensor pointer must be 16-byte aligned.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   Every call only enqueues work on it and returns; nothing synchronises the host except
 *   ep_read_status.
 * Return codes.  An ep_status_t: EP_OK when the work was enqueued.  Host-side argument checks
 *   run before any CUDA call and return EP_ERR_INVALID_ARG (nothing enqueued); a failed launch
 *   returns EP_ERR_CUDA.  Conditions only the GPU can see (capacity overflow, expert ids out of
 *   range) are recorded in the layout's device status word instead, see below.
 * Sizes.  T tokens, K top-k slots, E routed experts, S = 1 when a shared expert is fused
 *   (else 0), G = E + S groups, H hidden size, P logical expert partitions, C their capacity.
 *   R = number of (token, slot) pairs with a valid id + S*T = rows in use (plus the padding
 *   rows when groups are padded, see ep_dispatch_layout_routed), and R_max = rows every
 *   dispatched buffer must be sized for, so that no host synchronisation is ever needed to
 *   size an output: T*K + S*T by default, see ep_rows_max.  Rows [R, R_max) are never written.
 * Limits.  0 <= T <= 2^24, 1 <= K <= 32, 1 <= E <= 1024 (K may exceed E: a token may
 *   name an expert in several slots), 1 <= P <= E with E % P == 0,
 *   C >= 0, R_max < 2^31; H % 16 == 0 and 16 <= H <= 32768.
 * Profiling.  With the environment variable EP_GB300_NVTX set to anything but "0" when the
 *   library first checks it, each entry point that enqueues work (and ep_read_status) wraps
 *   itself in an NVTX range named after it, so a profiler can select an op's kernels by range
 *   (for example ncu --nvtx --nvtx-include "ep_combine/").  Off by default; results are the same
 *   either way.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host return codes. */
typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,   /* an argument failed a host-side check; nothing was enqueued  */
    EP_ERR_OVERFLOW = 2,      /* ep_read_status: a partition received more than C tokens,
                                 or the rows exceed the layout's row capacity             */
    EP_ERR_BAD_EXPERT = 3,    /* ep_read_status: an expert id was outside [-1, E)            */
    EP_ERR_CUDA = 5,          /* a CUDA call failed (launch error, or the sync in read_status) */
    EP_ERR_TOO_LARGE = 6,     /* ep_dispatch_layout_noalloc: the sizes need more scratch than
                                 its fixed array holds (EP_NOALLOC_WORKSPACE_BYTES)            */
    EP_ERR_BOUNDS = 7         /* ep_read_status, bounds-checked build only: an index fell
                                 outside its buffer and the access was skipped                */
} ep_status_t;

/* Bits of the device status word written by ep_dispatch_layout. */
#define EP_STATUS_OVERFLOW   1
#define EP_STATUS_BAD_EXPERT 2
/*
 * Set only by the bounds-checked debug build of the library (libep_gb300_checked.so, compiled
 * with EP_BOUNDS_CHECK=1).  That build checks every index that comes from data against the
 * buffer it indexes: a row read from a layout (row_of, row_offsets) against [0, R_max), where
 * -1 marks an unused slot, and a position computed inside the layout kernel against its
 * shared-memory range.  An access that fails is skipped, not performed, and this bit is set.
 * The default build skips rows outside [0, R_max) in the same way but records nothing.
 */
#define EP_STATUS_BOUNDS     8

/*
 * The dispatch layout: caller-allocated device buffers, filled by ep_dispatch_layout and read
 * by every other entry point.  A layout can be reused for any number of dispatch / combine /
 * backward calls with the same routing (for example the recompute pass of activation
 * checkpointing replays a recorded layout without a new layout pass or host read; fused_a2a,
 * DispatchReplayRecorder / HybridEPDispatchReplayRecorder).
 *
 *   row_offsets [G+1]     row_offsets[g] = first row of group g, row_offsets[G] = R
 *                         (Mojo EP dispatch, execute: row_offsets of the received tokens).
 *   expert_ids  [R_max]   group of each row, E for the shared expert's rows
 *                         (Mojo EP dispatch, execute: expert ID of each received token).
 *   src_info    [R_max*2] (token, slot) of each row, slot K for a shared row
 *                         (Mojo EP dispatch, execute: originating rank and token index; one
 *                         GPU, so the rank is always 0 and the slot is kept instead).
 *   row_of      [T*K]     row of each (token, slot), -1 for an unused slot (the saved mapping
 *                         combine and the backward passes read; token_dispatcher,
 *                         _DeepepManager.reversed_mapping_for_combine).
 *   part_tokens [P]       tokens received by each logical partition.
 *   status      [1]       EP_STATUS_* bits (token_dispatcher, _assert_no_hybridep_overflow:
 *                         an overflow flag instead of silent truncation).
 *   workspace             ep_layout_workspace_bytes(T, K, E, S) bytes of scratch.  It must be
 *                         zero-filled once before its first use; every call leaves it ready
 *                         for the next one.  Calls that share a workspace must not overlap on
 *                         the GPU (use one stream, or one workspace per stream).
 * The remaining fields are recorded by the layout call and checked by the other calls;
 * pad_multiple and row_capacity are 1 and 0 (no padding, default R_max) unless the layout was
 * made by ep_dispatch_layout_routed.
 */
typedef struct {
    int32_t *row_offsets;
    int32_t *expert_ids;
    int32_t *src_info;
    int32_t *row_of;
    int32_t *part_tokens;
    int32_t *status;
    void *workspace;
    size_t workspace_bytes;
    int T, K, E, P, capacity, fused_shared;
    int pad_multiple, row_capacity;
} ep_layout_t;

/*
 * Rows every dispatched buffer (and expert_ids / src_info) must hold for a layout of these
 * sizes: num_permuted_tokens when it is > 0 (a static row capacity), else
 * T*K + S*T + (E+S)*(pad_multiple-1), the most rows any routing can need.  pad_multiple <= 1
 * means no padding.  Returns 0 on invalid sizes.
 */
size_t ep_rows_max(int T, int K, int n_experts, int fused_shared, int pad_multiple,
                   int num_permuted_tokens);

/* Scratch bytes ep_dispatch_layout needs for these sizes (0 on invalid sizes). */
size_t ep_layout_workspace_bytes(int T, int K, int n_experts, int fused_shared);

/*
 * ep_dispatch_layout -- the routing metadata of a dispatch.
 * Defined by: Mojo EP dispatch, execute (route tokens by their top-k ids; row_offsets,
 * expert_ids, src_info; max_token_per_rank; fused_shared_expert) and fused_a2a,
 * HybridEPDispatch.forward (compact per-token expert indices, a slot holding -1 carries no
 * token; the dispatched rows come out grouped by expert).
 *
 *   topk_ids  [T*K] int32 device: expert id of each (token, slot) in [-1, E); -1 = unused.
 *   n_parts   P logical expert partitions: partition p owns experts [p*E/P, (p+1)*E/P).
 *   capacity  C: most tokens a partition may receive (a token counts once per partition it
 *             reaches; the shared expert does not count).
 *   fused_shared  1: add a group E holding one row per token (slot K), after every routed row.
 *   L         caller-filled buffer pointers and workspace; the size fields are written here.
 *
 * Order: group-major (experts ascending, then the shared group), and inside a group the
 * (token, slot) pairs in ascending t*K + k order, so the result is deterministic and does not
 * depend on the launch configuration.
 * Device-side errors: an id outside [-1, E) sets EP_STATUS_BAD_EXPERT and is treated as unused;
 * a partition over capacity sets EP_STATUS_OVERFLOW.  The metadata is written in full in both
 * cases; the status word is rewritten (not OR-ed) by every call.  Every later call that reads
 * this layout writes none of its outputs while the status word is non-zero: nothing is
 * silently truncated.
 */
int ep_dispatch_layout(const int32_t *topk_ids, int T, int K, int n_experts, int n_parts,
                       int capacity, int fused_shared, ep_layout_t *L, void *stream);

/*
 * ep_dispatch_layout_routed -- the layout from either routing representation, with optional
 * per-group padding and a static row capacity.
 * Defined by: fused_a2a, HybridEPDispatch.forward (a dense Boolean routing map [tokens,
 * experts] or compact top-k indices, the map taking precedence when both are given;
 * pad_multiple; num_permuted_tokens, the optional static dispatched-token capacity);
 * token_dispatcher, TokenDispatcherConfig.moe_router_expert_pad_multiple and _align_up (each
 * expert's token count rounded up to a multiple), TokenDispatcherConfig.
 * moe_benchmark_static_routing (a persisted row count keeps the dispatch free of host reads),
 * and _assert_no_hybridep_overflow (an overflow flag, never a silent truncation).
 *
 *   topk_ids       [T*K] int32 device, as for ep_dispatch_layout; read only when routing_map
 *                  is NULL.
 *   routing_map    [T*E] uint8 device or NULL: non-zero where token t goes to expert e.  When
 *                  given it is converted first (exactly as ep_routing_map_to_topk does) into
 *                  map_topk_ids / map_topk_probs, and the layout is made from map_topk_ids.
 *   dense_probs    [T*E] fp32 device or NULL: probabilities of the map's entries.
 *   map_topk_ids   [T*K] int32 device: required when routing_map is given (ignored otherwise).
 *   map_topk_probs [T*K] fp32 device or NULL: written when routing_map and dense_probs are
 *                  given; these are the probabilities ep_combine then takes.
 *   pad_multiple   >= 1 (1: no padding), at most 65536.  Every group's rows (the shared
 *                  group's too) are followed by padding rows up to a multiple of it:
 *                  row_offsets[g+1] - row_offsets[g] is a multiple of pad_multiple.  A padding
 *                  row has expert_ids = its group and src_info = (-1, -1).
 *   num_permuted_tokens  > 0: the rows the caller's buffers hold (R_max, see ep_rows_max);
 *                  0: the default R_max.  When the rows needed, row_offsets[G], exceed R_max,
 *                  EP_STATUS_OVERFLOW is set; rows at or past R_max are not recorded
 *                  (row_of of their pairs is -1) and no payload is written by later calls.
 * Everything else (order, partitions, capacity, status) is as for ep_dispatch_layout, which
 * is this call with routing_map = NULL, pad_multiple = 1, num_permuted_tokens = 0.  Every
 * dispatch call writes the padding rows of its outputs as the dispatch of an all-zero token,
 * and ep_combine_bwd writes zero gradients there, so a grouped GEMM over the padded extents
 * sees zeros; ep_combine and ep_dispatch_bwd never read them.
 */
int ep_dispatch_layout_routed(const int32_t *topk_ids, const uint8_t *routing_map,
                              const float *dense_probs, int T, int K, int n_experts, int n_parts,
                              int capacity, int fused_shared, int pad_multiple,
                              int num_permuted_tokens, int32_t *map_topk_ids,
                              float *map_topk_probs, ep_layout_t *L, void *stream);

/*
 * ep_routing_map_to_topk -- dense routing map to compact top-k ids.
 * Defined by: fused_a2a, HybridEPDispatch.forward (routing_map [tokens, experts] Boolean,
 * probs [tokens, experts] dense; topk_idx [tokens, top_k] with -1 for an unused slot).
 *   routing_map [T*E] uint8, dense_probs [T*E] fp32 or NULL
 *   -> topk_ids [T*K] int32: slot j of token t = the j-th expert (ascending id) whose map entry
 *      is non-zero, -1 after the last one; topk_probs [T*K] fp32 or NULL: the dense
 *      probability of that entry, 0 for a -1 slot.
 * A token with more than K experts in the map cannot be written in K slots: every slot of it
 * gets the id E (and probability 0), which a later layout reports as EP_STATUS_BAD_EXPERT.
 */
int ep_routing_map_to_topk(const uint8_t *routing_map, const float *dense_probs, int T,
                           int n_experts, int K, int32_t *topk_ids, float *topk_probs,
                           void *stream);

/*
 * ep_indices_to_multihot -- compact top-k ids to a dense routing map.
 * Defined by: token_dispatcher, _DeepepManager._indices_to_multihot /
 * _HybridEPManager._indices_to_multihot ([num_tokens, topk] indices with -1 masked out, and
 * their probabilities, to a multihot routing map and multihot probabilities).
 *   topk_ids [T*K] int32, topk_probs [T*K] fp32 or NULL
 *   -> routing_map [T*E] uint8: 1 where some slot of t names e, else 0;
 *   -> dense_probs [T*E] fp32 or NULL: the fp32 sum over those slots in ascending k (from +0),
 *      0 elsewhere (a token naming an expert twice sends it the sum).
 * Ids outside [0, E) are skipped (the layout is what reports ids outside [-1, E)).  With
 * topk_probs = grad_probs of ep_combine_bwd this gives the gradient in the dense layout.
 */
int ep_indices_to_multihot(const int32_t *topk_ids, const float *topk_probs, int T, int K,
                           int n_experts, uint8_t *routing_map, float *dense_probs, void *stream);

/*
 * ep_dispatch_nvfp4 -- scatter every token into its rows as NVFP4.
 * Defined by: Mojo EP dispatch, execute (a token is sent to its experts as NVFP4, scaled by a
 * per-token factor 2688 divided by the token's largest magnitude; the side that receives it
 * stores that factor's reciprocal as BF16 per row in output_rowwise_scales; output_scales
 * holds the per-block scales and scales_offsets tells where each group's scales begin).
 *
 *   input_tokens           [T*H] bf16.
 *   out_fp4                [R_max * H/2] uint8: E2M1 codes, element 2j in the low nibble of
 *                          byte j of the row.
 *   out_scales             [R_max * H/16] uint8: E4M3 block scale of each 16-element block,
 *                          row-major, unswizzled.
 *   out_rowwise_inv_scale  [R_max] bf16: bf16(1/g) per row.
 *   scales_offsets         [G+1] int32: first scale row of each group (= row_offsets).
 * Per token, in fp32 with every operation rounded to nearest even: a = max|x|,
 * g = (a == 0 ? 1 : 2688/a, clamped to FLT_MAX), block scale s = E4M3((blockmax*g)/6),
 * code = E2M1(x * (g/s)) (0 when s decodes to 0; g/s clamped to FLT_MAX), E4M3 and E2M1
 * saturating to their largest finite values.  All rows of a token receive identical bytes.
 */
int ep_dispatch_nvfp4(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                      uint8_t *out_fp4, uint8_t *out_scales, uint16_t *out_rowwise_inv_scale,
                      int32_t *scales_offsets, void *stream);

/*
 * ep_dispatch_layout_nvfp4 -- ep_dispatch_layout followed by ep_dispatch_nvfp4, in one call.
 * Defined by: fused_a2a, HybridEPDispatch.forward (routing metadata and the permuted copy of
 * the tokens produced by one dispatch; fuse_permute) and Mojo EP dispatch, execute (routing by
 * top-k ids and NVFP4 quantisation in one operation).
 *
 * Arguments are those of ep_dispatch_layout followed by those of ep_dispatch_nvfp4, and the
 * results are identical to calling the two in sequence.  Doing both in one call lets the
 * quantisation of input_tokens overlap the layout computation: the dispatch kernel launches
 * on the SMs the layout leaves free and its CTAs read and quantise their tokens before the
 * layout has finished (safe because input_tokens, like every argument, must be complete in
 * stream order when the call is made); they wait for the layout only before storing.  Errors
 * are those of the two calls.
 */
int ep_dispatch_layout_nvfp4(const int32_t *topk_ids, int T, int K, int n_experts, int n_parts,
                             int capacity, int fused_shared, const uint16_t *input_tokens,
                             int hidden_size, ep_layout_t *L, uint8_t *out_fp4,
                             uint8_t *out_scales, uint16_t *out_rowwise_inv_scale,
                             int32_t *scales_offsets, void *stream);

/*
 * ep_dispatch_layout_padded_nvfp4 -- ep_dispatch_layout_routed from compact ids (routing_map
 * NULL), with groups padded to pad_multiple rows and an optional static row capacity, followed
 * by ep_dispatch_nvfp4, in one call.
 * Defined by: token_dispatcher, TokenDispatcherConfig.moe_router_expert_pad_multiple and
 * moe_benchmark_static_routing (padded groups, a persisted row count); fused_a2a,
 * HybridEPDispatch.forward (pad_multiple, num_permuted_tokens; fuse_permute); Mojo EP dispatch,
 * execute (NVFP4 quantisation in the dispatch).
 *
 * Arguments are those of ep_dispatch_layout_routed (without the routing map and its outputs)
 * followed by those of ep_dispatch_nvfp4, and the results are identical to calling the two in
 * sequence: every padding row receives the dispatch of an all-zero token (codes 0, block scales
 * 0, inverse scale bf16(1)), rows at or past row_offsets[G] are untouched, and nothing but the
 * layout is written when the status word is set.  As in ep_dispatch_layout_nvfp4, the
 * quantisation of input_tokens overlaps the layout.  The buffers hold R_max rows, as
 * ep_rows_max(T, K, E, S, pad_multiple, num_permuted_tokens) gives.  Errors are those of the
 * two calls.
 */
int ep_dispatch_layout_padded_nvfp4(const int32_t *topk_ids, int T, int K, int n_experts,
                                    int n_parts, int capacity, int fused_shared, int pad_multiple,
                                    int num_permuted_tokens, const uint16_t *input_tokens,
                                    int hidden_size, ep_layout_t *L, uint8_t *out_fp4,
                                    uint8_t *out_scales, uint16_t *out_rowwise_inv_scale,
                                    int32_t *scales_offsets, void *stream);

/*
 * ep_dispatch_bf16 -- scatter every token into its rows unchanged.
 * Defined by: fused_a2a, HybridEPDispatch.forward / hybrid_ep_dispatch (dispatched hidden
 * states [dispatched_tokens, hidden] grouped by expert).
 *   input_tokens [T*H] bf16  ->  out [R_max*H] bf16.
 */
int ep_dispatch_bf16(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                     uint16_t *out, void *stream);

/*
 * ep_dispatch_fp8 -- scatter every token into its rows as FP8 (E4M3) with one scale per block
 * of 128 elements.
 * Defined by: fused_a2a, init_hybrid_ep_buffer, fp8_dispatch (the dispatch may carry FP8
 * instead of BF16; the pages fix no block size or scale format: this library's reading).
 *   input_tokens [T*H] bf16, H % 128 == 0
 *   -> out_fp8    [R_max * H] uint8: E4M3 codes (round to nearest even, saturating to +-448);
 *   -> out_scales [R_max * H/128] fp32: the factor a consumer multiplies the codes by.
 * Per block of 128, in fp32 with every operation rounded once: m = max|x|,
 * s = (m == 0 ? 1 : 448/m, clamped to FLT_MAX), code = E4M3(x * s), scale = 1/s.
 * All rows of a token receive identical bytes.
 */
int ep_dispatch_fp8(const uint16_t *input_tokens, int hidden_size, const ep_layout_t *L,
                    uint8_t *out_fp8, float *out_scales, void *stream);

/*
 * ep_combine -- probability-weighted gather-reduce of the expert outputs into token order.
 * Defined by: fused_a2a, hybrid_ep_combine / HybridEPCombine.forward (the expert outputs,
 * one row per dispatched token, are brought back to one row per input token, in input order);
 * token_dispatcher, TokenDispatcherConfig.moe_router_dtype (the router's fp32 probabilities
 * are the weights).
 *   expert_out [R_max*H] bf16, probs [T*K] fp32  ->  out [T*H] bf16:
 *   out[t] = bf16( sum over k ascending with row_of[t,k] >= 0 of probs[t,k] * expert_out[row]
 *                  + (S ? expert_out[row_offsets[E] + t] : 0) ), accumulated in fp32.
 */
int ep_combine(const uint16_t *expert_out, const float *probs, int hidden_size,
               const ep_layout_t *L, uint16_t *out, void *stream);

/*
 * ep_combine_bwd -- backward of ep_combine.
 * Defined by: fused_a2a, HybridEPCombine.backward (the combined-output gradient [tokens,
 * hidden] is dispatched again through the saved layout).
 *   grad_out [T*H] bf16, expert_out [R_max*H] bf16, probs [T*K] fp32
 *   -> grad_expert_out [R_max*H] bf16: row of (t,k) = bf16(probs[t,k] * grad_out[t]),
 *                                      shared row of t = grad_out[t];
 *   -> grad_probs [T*K] fp32: sum_i grad_out[t,i] * expert_out[row_of[t,k], i] (fp32
 *      accumulation), 0 for an unused slot.
 */
int ep_combine_bwd(const uint16_t *grad_out, const uint16_t *expert_out, const float *probs,
                   int hidden_size, const ep_layout_t *L, uint16_t *grad_expert_out,
                   float *grad_probs, void *stream);

/*
 * ep_dispatch_bwd -- backward of ep_dispatch_bf16 / ep_dispatch_nvfp4 (straight through the
 * quantiser).
 * Defined by: fused_a2a, HybridEPDispatch.backward (the dispatched rows' gradients
 * [dispatched_tokens, hidden] are combined back per token).
 *   grad_rows [R_max*H] bf16  ->  grad_input [T*H] bf16:
 *   grad_input[t] = bf16( sum over valid k ascending of grad_rows[row_of[t,k]]
 *                         + (S ? grad_rows[row_offsets[E] + t] : 0) ), fp32 accumulation.
 */
int ep_dispatch_bwd(const uint16_t *grad_rows, int hidden_size, const ep_layout_t *L,
                    uint16_t *grad_input, void *stream);

/*
 * ep_read_status -- synchronise `stream` and copy the layout's status word to *host_status.
 * Returns EP_OK, EP_ERR_BOUNDS (bounds-checked build only; reported first), EP_ERR_OVERFLOW or
 * EP_ERR_BAD_EXPERT (overflow reported before a bad expert id when both bits are set), or
 * EP_ERR_CUDA.  The one call of this library that blocks the host.
 */
int ep_read_status(const ep_layout_t *L, void *stream, int32_t *host_status);

/*
 * ep_dispatch_layout_noalloc -- ep_dispatch_layout for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point.
 *
 * Some callers cannot call cudaMalloc: code that runs inside a framework whose allocator owns
 * all device memory, latency-critical paths that must not pay for (or synchronise on) an
 * allocation, and runtimes that give a library its inputs and outputs and nothing else.  This
 * entry point computes exactly what ep_dispatch_layout computes, from the same arguments, but
 * never touches L->workspace (L->workspace and L->workspace_bytes are ignored and may be
 * NULL / 0).  Sizes whose ids fit one thread-block cluster (the single-cluster layout kernel
 * ep_dispatch_layout also uses) need no scratch at all; larger sizes run the two-kernel layout
 * with its scratch in a fixed array inside the library.  The caller still passes every input
 * and output buffer.
 *
 *   Limit: the sizes must satisfy ep_layout_workspace_bytes(T, K, E, S) <=
 *   EP_NOALLOC_WORKSPACE_BYTES (1 MiB; T = 32768, K = 8, E = 256 needs 128.5 KiB (131,584
 *   bytes), and at K = 8, E = 256 every T up to 522240 fits); larger sizes return
 *   EP_ERR_TOO_LARGE and enqueue nothing.  Every GPU that loads the library holds that 1 MiB
 *   until the process exits.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and zeroes its first 256 bytes with a
 *   synchronous cudaMemset; make that first call before any stream capture.  Later calls only
 *   enqueue the layout kernels.
 *   Sharing: every call on a device uses the same array, and each call leaves it ready for the
 *   next.  Calls whose work overlaps on the GPU (two streams, or two host threads) race on the
 *   array and give undefined results; serialise them.
 *   No call allocates or frees device memory (no cudaMalloc, cudaFree or allocating library
 *   routine).  Other errors are those of ep_dispatch_layout.
 */
#define EP_NOALLOC_WORKSPACE_BYTES (1u << 20)
int ep_dispatch_layout_noalloc(const int32_t *topk_ids, int T, int K, int n_experts,
                               int n_parts, int capacity, int fused_shared, ep_layout_t *L,
                               void *stream);

/* Human-readable name of a return code. */
const char *ep_strerror(int code);

/*
 * Conversion primitives used by ep_dispatch_nvfp4, exposed so the conversions can be checked
 * on their own (NVFP4's element and scale formats, Mojo EP dispatch, execute).
 *   ep_cvt_e2m1: codes[i] = E2M1 code of in[i] (round to nearest even, saturating to +-6,
 *                sign bit = sign of in[i]), one code per byte in the low nibble.
 *   ep_cvt_e4m3: codes[i] = E4M3 code of in[i] (round to nearest even, saturating to +-448).
 *   in [n] fp32 device, codes [n] uint8 device, n >= 0.
 */
int ep_cvt_e2m1(const float *in, uint8_t *codes, long n, void *stream);
int ep_cvt_e4m3(const float *in, uint8_t *codes, long n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
