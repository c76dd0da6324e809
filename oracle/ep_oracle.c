/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle of the MoE dispatch / combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, calls or imports this file.
 * Only tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources, cited below by page and section:
 *   "fused_a2a"        NeMo AutoModel v0.4 API page nemo_automodel...moe.megatron.fused_a2a
 *   "token_dispatcher" NeMo AutoModel v0.7 API page nemo_automodel...moe.megatron.token_dispatcher
 *   "Mojo EP dispatch" Modular MAX API page, struct DistributedEPDispatchBlockScaledNVDynGlobalScales
 *
 * Floating point: IEEE binary32 for every step whose result is a quantised code (the kernel's
 * precision; the pages fix none), binary64 for every accumulation (combine and its backward).
 * Build with -O2 -ffp-contract=off and no fast-math, so no multiply-add is fused.
 *
 * Pins (tests/test_oracle_*.py): brute-force layout invariants, the E2M1 / E4M3 value tables
 * from the format definitions, the 2688 = 6 * 448 closed form, the zero row, the dequantisation
 * error bound, round trips with identity experts, and adjoint identities for both backward
 * passes; the padded layout against a row list built by concatenation and hand-worked
 * examples; FP8 blocks worked by hand, exact power-of-two scaling and the E4M3 error bound;
 * both routing conversions by brute force over every small map and by round trips.  No
 * function here is "parity unpinned".
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OVERFLOW   1
#define ORC_BAD_EXPERT 2

/* ------------------------------------------------------------------------------------------
 * bf16 <-> binary64.  bf16 is the upper half of an IEEE binary32.
 * ---------------------------------------------------------------------------------------- */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a finite binary64 value to bf16 (8 significant bits), nearest with ties to even.
 * Values past the largest finite bf16 by half a quantum or more become infinity. */
uint16_t oracle_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);              /* a = m * 2^e2, m in [0.5, 1): floor(log2 a) = e2 - 1 */
    int ex = e2 - 1;
    if (ex < -126)
        ex = -126;              /* bf16 subnormals share the quantum of the lowest normal binade */
    double q = ldexp(1.0, ex - 7);
    double r = nearbyint(a / q) * q;   /* default rounding mode: nearest, ties to even */
    double maxb = ldexp(255.0 / 128.0, 127);
    float f = (r > maxb) ? INFINITY : (float)r;   /* r has <= 8 significant bits: exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16) | sign;
}

/* ------------------------------------------------------------------------------------------
 * E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf / NaN.
 * Magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * E4M3 (FP8, the "FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities,
 * code 0x7F is NaN, largest finite 448 (0x7E), smallest subnormal 2^-9.
 * Encoding: round to nearest, ties to the even code, saturating to the largest finite value;
 * the sign bit is the sign of the input (so -0 and tiny negatives give a negative zero code).
 * ---------------------------------------------------------------------------------------- */
static double e2m1_mag(int c)
{
    int ex = (c >> 1) & 3, m = c & 1;
    return ex == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
}

static double e4m3_mag(int c)
{
    int ex = (c >> 3) & 15, m = c & 7;
    return ex == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, ex - 7);
}

/* Nearest-even rounding of a >= 0 onto the ascending grid mag(0..top), saturating at top. */
static int round_to_grid(double a, double (*mag)(int), int top)
{
    if (!(a < mag(top)))   /* saturate; a NaN (outside the method's domain) also stops here */
        return top;
    int c = 0;
    while (!(a < mag(c + 1)))
        c++;                                  /* mag(c) <= a < mag(c+1) */
    double mid = 0.5 * (mag(c) + mag(c + 1)); /* exact: both have few significant bits */
    if (a < mid)
        return c;
    if (a > mid)
        return c + 1;
    return (c % 2 == 0) ? c : c + 1;          /* tie: the even code */
}

uint8_t oracle_e2m1_encode(float v)
{
    uint8_t s = signbit(v) ? 0x8 : 0x0;
    return (uint8_t)(s | round_to_grid(fabs((double)v), e2m1_mag, 7));
}

float oracle_e2m1_decode(uint8_t code)
{
    double m = e2m1_mag(code & 7);
    return (float)((code & 8) ? -m : m);
}

uint8_t oracle_e4m3_encode(float v)
{
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    return (uint8_t)(s | round_to_grid(fabs((double)v), e4m3_mag, 0x7E));
}

float oracle_e4m3_decode(uint8_t code)
{
    double m = e4m3_mag(code & 0x7F);
    return (float)((code & 0x80) ? -m : m);
}

/* ------------------------------------------------------------------------------------------
 * Layout [Mojo EP dispatch, execute: row_offsets, expert_ids, src_info;
 * fused_a2a, HybridEPDispatch.forward: the rows come out grouped by expert, an index of -1
 * routes nowhere, pad_multiple and num_permuted_tokens; token_dispatcher,
 * TokenDispatcherConfig.moe_router_expert_pad_multiple and _align_up: each expert's token count
 * is rounded up to a multiple; _assert_no_hybridep_overflow: an overflow flag instead of
 * silent truncation].
 *
 * 1. An id outside [-1, E) sets BAD_EXPERT and is then treated as an unused slot.
 * 2. counts[e] = #{(t,k): id = e}; with a fused shared expert, group E holds one row per token.
 * 3. extent[g] = the smallest multiple of pad that is >= counts[g] (pad = 1: no padding);
 *    row_offsets = exclusive scan of the extents over the G = E + S groups.
 * 4. Rows of group e are its (t,k) pairs in ascending flat index t*K+k: a stable sort of the
 *    flat indices keyed by expert id; the i-th pair of group e is row row_offsets[e] + i.
 * 5. row_of[t*K+k] = row (or -1), src_info[row] = (t, k), expert_ids[row] = e.
 * 6. Shared rows: row_offsets[E] + t, src_info (t, K), expert_ids E.
 * 7. Padding rows row_offsets[g] + counts[g] .. row_offsets[g+1] - 1: expert_ids g,
 *    src_info (-1, -1).
 * 8. part_tokens[p] = #{t : some id of t lies in partition p = id / (E/P)}; OVERFLOW when any
 *    partition receives more tokens than the capacity C (Mojo EP dispatch, parameter
 *    max_token_per_rank).
 * 9. Row capacity R_max = row_cap when row_cap > 0 (the static dispatched-token capacity),
 *    else T*K + S*T + G*(pad-1) (the most rows any routing can need).  OVERFLOW when
 *    row_offsets[G] > R_max; a row at or past R_max is not recorded: its src_info and
 *    expert_ids are not written and row_of of its pair is -1.
 * Returns the status bitmask.  Apart from step 9 the metadata is written in full in every case.
 * ---------------------------------------------------------------------------------------- */
typedef struct { int32_t e; int32_t i; } sort_key;

static int cmp_key(const void *pa, const void *pb)
{
    const sort_key *a = pa, *b = pb;
    if (a->e != b->e)
        return a->e < b->e ? -1 : 1;
    return a->i < b->i ? -1 : (a->i > b->i);
}

long oracle_rows_max(int T, int K, int E, int S, int pad, long row_cap)
{
    if (row_cap > 0)
        return row_cap;
    return (long)T * K + (long)S * T + (long)(E + S) * (pad - 1);
}

int oracle_layout_padded(const int32_t *topk_ids, int T, int K, int E, int P, int C, int S,
                         int pad, long row_cap, int32_t *row_offsets, int32_t *expert_ids,
                         int32_t *src_info, int32_t *row_of, int32_t *part_tokens)
{
    int status = 0;
    long n = (long)T * K;
    int G = E + S;
    long R_max = oracle_rows_max(T, K, E, S, pad, row_cap);
    int32_t *id = malloc(sizeof(int32_t) * (n ? n : 1));
    for (long i = 0; i < n; i++) {
        int32_t v = topk_ids[i];
        if (v < -1 || v >= E) {
            status |= ORC_BAD_EXPERT;
            v = -1;
        }
        id[i] = v;
    }

    long *counts = calloc((size_t)G, sizeof(long));
    for (long i = 0; i < n; i++)
        if (id[i] >= 0)
            counts[id[i]]++;
    if (S)
        counts[E] = T;

    long acc = 0;
    for (int g = 0; g < G; g++) {
        row_offsets[g] = (int32_t)acc;
        acc += (counts[g] + pad - 1) / pad * pad;
    }
    row_offsets[G] = (int32_t)acc;
    if (acc > R_max)
        status |= ORC_OVERFLOW;

    sort_key *keys = malloc(sizeof(sort_key) * (n ? n : 1));
    long nv = 0;
    for (long i = 0; i < n; i++) {
        row_of[i] = -1;
        if (id[i] >= 0) {
            keys[nv].e = id[i];
            keys[nv].i = (int32_t)i;
            nv++;
        }
    }
    qsort(keys, (size_t)nv, sizeof(sort_key), cmp_key);   /* (e, i) keys are distinct: stable */
    long j = 0;
    while (j < nv) {   /* one run of equal experts at a time */
        int e = keys[j].e;
        long first = j;
        for (; j < nv && keys[j].e == e; j++) {
            long r = row_offsets[e] + (j - first);
            if (r >= R_max)
                continue;
            int32_t i = keys[j].i;
            row_of[i] = (int32_t)r;
            src_info[2 * r] = i / K;
            src_info[2 * r + 1] = i % K;
            expert_ids[r] = e;
        }
    }
    if (S) {
        for (int t = 0; t < T; t++) {
            long r = row_offsets[E] + t;
            if (r >= R_max)
                continue;
            src_info[2 * r] = t;
            src_info[2 * r + 1] = K;
            expert_ids[r] = E;
        }
    }
    for (int g = 0; g < G; g++) {
        for (long r = row_offsets[g] + counts[g]; r < row_offsets[g + 1]; r++) {
            if (r >= R_max)
                continue;
            src_info[2 * r] = -1;
            src_info[2 * r + 1] = -1;
            expert_ids[r] = g;
        }
    }

    int per = E / P;
    for (int p = 0; p < P; p++) {
        long cnt = 0;
        for (int t = 0; t < T; t++) {
            int hit = 0;
            for (int k = 0; k < K; k++) {
                int32_t v = id[(long)t * K + k];
                if (v >= 0 && v / per == p)
                    hit = 1;
            }
            cnt += hit;
        }
        part_tokens[p] = (int32_t)cnt;
        if (cnt > C)
            status |= ORC_OVERFLOW;
    }
    free(keys);
    free(counts);
    free(id);
    return status;
}

/* The layout without padding or a row capacity (pad = 1, R_max = T*K + S*T). */
int oracle_layout(const int32_t *topk_ids, int T, int K, int E, int P, int C, int S,
                  int32_t *row_offsets, int32_t *expert_ids, int32_t *src_info,
                  int32_t *row_of, int32_t *part_tokens)
{
    return oracle_layout_padded(topk_ids, T, K, E, P, C, S, 1, 0, row_offsets, expert_ids,
                                src_info, row_of, part_tokens);
}

/* ------------------------------------------------------------------------------------------
 * NVFP4 quantisation of one token [Mojo EP dispatch, execute: each token is quantised to NVFP4
 * against a global scale of its own, 2688 / rowmax, and the receiving side keeps the BF16
 * inverse of that scale per row in output_rowwise_scales].  All arithmetic in binary32, each operation rounded once:
 *   a  = max_i |x_i|
 *   g  = 1 if a == 0, else 2688 / a (clamped to FLT_MAX if that overflows)
 *   inv = bf16(1 / g)
 *   per 16-element block b:  ab = max |x| over b,  sf = (ab * g) / 6,  s = E4M3(sf),  sd = s
 *   per element:  code = 0 if sd == 0, else E2M1(x * r) with r = g / sd (clamped to FLT_MAX)
 *   packing: element 2j in the low nibble of byte j, element 2j+1 in the high nibble.
 * ---------------------------------------------------------------------------------------- */
void oracle_nvfp4_quantize_row(const uint16_t *x, int H, uint8_t *codes, uint8_t *scales,
                               uint16_t *inv)
{
    float a = 0.0f;
    for (int i = 0; i < H; i++) {
        float v = fabsf((float)oracle_bf16_to_double(x[i]));
        if (v > a)
            a = v;
    }
    float g = 1.0f;
    if (a != 0.0f) {
        g = 2688.0f / a;
        if (isinf(g))
            g = FLT_MAX;
    }
    float ginv = 1.0f / g;
    *inv = oracle_bf16_from_double((double)ginv);

    memset(codes, 0, (size_t)H / 2);
    for (int b = 0; b < H / 16; b++) {
        const uint16_t *xb = x + 16 * b;
        float ab = 0.0f;
        for (int i = 0; i < 16; i++) {
            float v = fabsf((float)oracle_bf16_to_double(xb[i]));
            if (v > ab)
                ab = v;
        }
        float prod = ab * g;
        float sf = prod / 6.0f;
        uint8_t s = oracle_e4m3_encode(sf);
        float sd = oracle_e4m3_decode(s);
        scales[b] = s;
        for (int i = 0; i < 16; i++) {
            uint8_t q = 0;
            if (sd != 0.0f) {
                float r = g / sd;
                if (isinf(r))
                    r = FLT_MAX;
                float y = (float)oracle_bf16_to_double(xb[i]) * r;
                q = oracle_e2m1_encode(y);
            }
            int e = 16 * b + i;
            codes[e / 2] |= (uint8_t)((e % 2 == 0) ? q : (q << 4));
        }
    }
}

/* NVFP4 dispatch [Mojo EP dispatch, execute]: every row of token t (its K routed copies and the shared copy)
 * receives the same codes, block scales and inverse scale.  scales_offsets = row_offsets (the
 * scales are stored row-major, H/16 per row).  Writes nothing when status != 0. */
void oracle_dispatch_nvfp4(const uint16_t *x, int T, int H, int K, int E, int S,
                           const int32_t *row_offsets, const int32_t *row_of, int status,
                           uint8_t *out_fp4, uint8_t *out_scales, uint16_t *out_inv,
                           int32_t *scales_offsets)
{
    if (status)
        return;
    int G = E + S;
    for (int g = 0; g <= G; g++)
        scales_offsets[g] = row_offsets[g];
    uint8_t *codes = malloc((size_t)H / 2);
    uint8_t *sc = malloc((size_t)H / 16);
    for (int t = 0; t < T; t++) {
        uint16_t inv;
        oracle_nvfp4_quantize_row(x + (size_t)t * H, H, codes, sc, &inv);
        for (int k = 0; k <= K; k++) {
            long r;
            if (k < K)
                r = row_of[(long)t * K + k];
            else
                r = S ? (long)row_offsets[E] + t : -1;
            if (r < 0)
                continue;
            memcpy(out_fp4 + (size_t)r * (H / 2), codes, (size_t)H / 2);
            memcpy(out_scales + (size_t)r * (H / 16), sc, (size_t)H / 16);
            out_inv[r] = inv;
        }
    }
    free(sc);
    free(codes);
}

/* BF16 dispatch [fused_a2a, HybridEPDispatch.forward: dispatched hidden states
 * grouped by expert]:
 * every row of token t receives a copy of x[t].  Writes nothing when status != 0. */
void oracle_dispatch_bf16(const uint16_t *x, int T, int H, int K, int E, int S,
                          const int32_t *row_offsets, const int32_t *row_of, int status,
                          uint16_t *out)
{
    if (status)
        return;
    for (int t = 0; t < T; t++) {
        for (int k = 0; k <= K; k++) {
            long r;
            if (k < K)
                r = row_of[(long)t * K + k];
            else
                r = S ? (long)row_offsets[E] + t : -1;
            if (r < 0)
                continue;
            memcpy(out + (size_t)r * H, x + (size_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
    }
}

/* Combine [fused_a2a, hybrid_ep_combine: expert outputs brought back to one row per input token,
 * shape [tokens, hidden]; token_dispatcher, TokenDispatcherConfig.moe_router_dtype: the
 * probabilities weight the expert outputs] and, with probs == NULL, the dispatch backward
 * pass [fused_a2a, HybridEPDispatch.backward: the dispatched rows' gradients are combined
 * back per token]:
 *   out[t] = bf16( sum_{k ascending, row_of >= 0} w[t,k] * y[row_of[t,k]]  +  S * y[shared t] )
 * with w = probs (combine) or 1 (dispatch backward), accumulated in binary64.
 * out64, when given, receives the unrounded sums.  Writes nothing when status != 0. */
void oracle_combine(const uint16_t *y, const float *probs, int T, int H, int K, int E, int S,
                    const int32_t *row_offsets, const int32_t *row_of, int status,
                    uint16_t *out, double *out64)
{
    if (status)
        return;
    double *acc = malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; t++) {
        for (int i = 0; i < H; i++)
            acc[i] = 0.0;
        for (int k = 0; k < K; k++) {
            long r = row_of[(long)t * K + k];
            if (r < 0)
                continue;
            double w = probs ? (double)probs[(long)t * K + k] : 1.0;
            for (int i = 0; i < H; i++)
                acc[i] += w * oracle_bf16_to_double(y[(size_t)r * H + i]);
        }
        if (S) {
            long r = (long)row_offsets[E] + t;
            for (int i = 0; i < H; i++)
                acc[i] += oracle_bf16_to_double(y[(size_t)r * H + i]);
        }
        for (int i = 0; i < H; i++) {
            out[(size_t)t * H + i] = oracle_bf16_from_double(acc[i]);
            if (out64)
                out64[(size_t)t * H + i] = acc[i];
        }
    }
    free(acc);
}

/* Combine backward [fused_a2a, HybridEPCombine.backward: the combined-output gradient is
 * dispatched again through the saved layout], the gradient of out = sum_k p_k y_k + S y_sh:
 *   grad_y[row_of[t,k]] = bf16(p[t,k] * g[t]),  grad_y[shared t] = g[t],
 *   grad_p[t,k] = sum_i g[t,i] * y[row_of[t,k], i]   (binary64; 0 for an unused slot).
 * grad_y64, when given, receives the unrounded row values.  Writes nothing when status != 0. */
void oracle_combine_bwd(const uint16_t *g, const uint16_t *y, const float *probs, int T, int H,
                        int K, int E, int S, const int32_t *row_offsets, const int32_t *row_of,
                        int status, uint16_t *grad_y, double *grad_p, double *grad_y64)
{
    if (status)
        return;
    for (int t = 0; t < T; t++) {
        const uint16_t *gt = g + (size_t)t * H;
        for (int k = 0; k < K; k++) {
            long r = row_of[(long)t * K + k];
            if (r < 0) {
                grad_p[(long)t * K + k] = 0.0;
                continue;
            }
            double p = (double)probs[(long)t * K + k];
            double dot = 0.0;
            for (int i = 0; i < H; i++) {
                double gi = oracle_bf16_to_double(gt[i]);
                double v = p * gi;
                grad_y[(size_t)r * H + i] = oracle_bf16_from_double(v);
                if (grad_y64)
                    grad_y64[(size_t)r * H + i] = v;
                dot += gi * oracle_bf16_to_double(y[(size_t)r * H + i]);
            }
            grad_p[(long)t * K + k] = dot;
        }
        if (S) {
            long r = (long)row_offsets[E] + t;
            for (int i = 0; i < H; i++) {
                grad_y[(size_t)r * H + i] = gt[i];
                if (grad_y64)
                    grad_y64[(size_t)r * H + i] = oracle_bf16_to_double(gt[i]);
            }
        }
    }
}

/* Expert outputs of the Tiny workload: each dispatched row dequantised (code value x block
 * scale x the stored bf16 inverse global scale, as a consumer of the NVFP4 rows sees it) and
 * multiplied by (1 + expert/8), then rounded to bf16.  Rows past R are left untouched. */
void oracle_tiny_expert_outputs(const uint8_t *fp4, const uint8_t *scales, const uint16_t *inv,
                                const int32_t *expert_ids, long R, int H, uint16_t *y)
{
    for (long r = 0; r < R; r++) {
        double gi = oracle_bf16_to_double(inv[r]);
        double f = 1.0 + expert_ids[r] / 8.0;
        for (int i = 0; i < H; i++) {
            uint8_t byte = fp4[(size_t)r * (H / 2) + i / 2];
            uint8_t q = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            double sd = oracle_e4m3_decode(scales[(size_t)r * (H / 16) + i / 16]);
            double v = (double)oracle_e2m1_decode(q) * sd * gi * f;
            y[(size_t)r * H + i] = oracle_bf16_from_double(v);
        }
    }
}

/* Array forms of the two encoders (one code per byte), for comparing many values at once. */
void oracle_e2m1_encode_n(const float *v, uint8_t *codes, long n)
{
    for (long i = 0; i < n; i++)
        codes[i] = oracle_e2m1_encode(v[i]);
}

void oracle_e4m3_encode_n(const float *v, uint8_t *codes, long n)
{
    for (long i = 0; i < n; i++)
        codes[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------------------------
 * Padding rows of a dispatched buffer [token_dispatcher,
 * TokenDispatcherConfig.moe_router_expert_pad_multiple: the tokens an expert's count is padded
 * with; fused_a2a, HybridEPDispatch.forward pad_multiple].  A padding token is an all-zero
 * token: every padding row (src_info token -1) below min(row_offsets[G], R_max) receives
 * `row`, the row_bytes bytes that the dispatch writes for an all-zero token.  Writes nothing
 * when status != 0.
 * ---------------------------------------------------------------------------------------- */
void oracle_fill_padding_rows(const int32_t *src_info, long R_pad, long R_max, int status,
                              uint8_t *buf, long row_bytes, const uint8_t *row)
{
    if (status)
        return;
    long end = R_pad < R_max ? R_pad : R_max;
    for (long r = 0; r < end; r++)
        if (src_info[2 * r] < 0)
            memcpy(buf + (size_t)r * (size_t)row_bytes, row, (size_t)row_bytes);
}

/* ------------------------------------------------------------------------------------------
 * FP8 quantisation of one token [fused_a2a, init_hybrid_ep_buffer, fp8_dispatch: the
 * dispatch may carry FP8 instead of BF16; the pages fix no block size or scale format].  E4M3 codes with one binary32 scale per block of
 * 128 consecutive elements; every operation in binary32, rounded once:
 *   ab = max |x| over the block
 *   s  = 1 if ab == 0, else 448 / ab (clamped to FLT_MAX if that overflows)
 *   code = E4M3(x * s)                    (round to nearest even, saturating to +-448)
 *   scale = 1 / s                         (what a consumer multiplies the codes by)
 * so the block's largest magnitude lands on E4M3's largest finite value.
 * ---------------------------------------------------------------------------------------- */
#define ORC_FP8_BLOCK 128

void oracle_fp8_quantize_row(const uint16_t *x, int H, uint8_t *codes, float *scales)
{
    for (int b = 0; b < H / ORC_FP8_BLOCK; b++) {
        const uint16_t *xb = x + ORC_FP8_BLOCK * b;
        float ab = 0.0f;
        for (int i = 0; i < ORC_FP8_BLOCK; i++) {
            float v = fabsf((float)oracle_bf16_to_double(xb[i]));
            if (v > ab)
                ab = v;
        }
        float s = 1.0f;
        if (ab != 0.0f) {
            s = 448.0f / ab;
            if (isinf(s))
                s = FLT_MAX;
        }
        scales[b] = 1.0f / s;
        for (int i = 0; i < ORC_FP8_BLOCK; i++) {
            float y = (float)oracle_bf16_to_double(xb[i]) * s;
            codes[ORC_FP8_BLOCK * b + i] = oracle_e4m3_encode(y);
        }
    }
}

/* FP8 dispatch: every row of token t (its K routed copies and the shared copy) receives the
 * same codes and block scales.  Writes nothing when status != 0. */
void oracle_dispatch_fp8(const uint16_t *x, int T, int H, int K, int E, int S,
                         const int32_t *row_offsets, const int32_t *row_of, int status,
                         uint8_t *out_codes, float *out_scales)
{
    if (status)
        return;
    int nb = H / ORC_FP8_BLOCK;
    uint8_t *codes = malloc((size_t)H);
    float *sc = malloc(sizeof(float) * (size_t)nb);
    for (int t = 0; t < T; t++) {
        oracle_fp8_quantize_row(x + (size_t)t * H, H, codes, sc);
        for (int k = 0; k <= K; k++) {
            long r;
            if (k < K)
                r = row_of[(long)t * K + k];
            else
                r = S ? (long)row_offsets[E] + t : -1;
            if (r < 0)
                continue;
            memcpy(out_codes + (size_t)r * H, codes, (size_t)H);
            memcpy(out_scales + (size_t)r * nb, sc, sizeof(float) * (size_t)nb);
        }
    }
    free(sc);
    free(codes);
}

/* ------------------------------------------------------------------------------------------
 * Routing representations [fused_a2a, HybridEPDispatch.forward: a dense Boolean routing map
 * [tokens, experts] or compact top-k indices [tokens, top_k] with -1 for an unused slot, the
 * map taking precedence, the probabilities staying dense; token_dispatcher,
 * _DeepepManager._indices_to_multihot / _HybridEPManager._indices_to_multihot].
 *
 * Map -> compact: slot j of token t holds the j-th expert (ascending id) whose map entry is
 * non-zero, and its dense probability; the slots after the last one hold -1 and probability 0.
 * A token with more than K experts in its map cannot be written in K slots: all its slots get
 * the id E (outside [-1, E), so the layout that reads them reports BAD_EXPERT) and
 * probability 0.  dense_probs / topk_probs may be NULL (no probabilities).
 * ---------------------------------------------------------------------------------------- */
void oracle_routing_map_to_topk(const uint8_t *routing_map, const float *dense_probs, int T,
                                int E, int K, int32_t *topk_ids, float *topk_probs)
{
    for (int t = 0; t < T; t++) {
        int n = 0;
        for (int e = 0; e < E; e++)
            if (routing_map[(long)t * E + e])
                n++;
        int j = 0;
        for (int e = 0; e < E && n <= K; e++) {
            if (!routing_map[(long)t * E + e])
                continue;
            topk_ids[(long)t * K + j] = e;
            if (topk_probs)
                topk_probs[(long)t * K + j] = dense_probs ? dense_probs[(long)t * E + e] : 0.0f;
            j++;
        }
        for (int k = (n <= K ? n : 0); k < K; k++) {
            topk_ids[(long)t * K + k] = n <= K ? -1 : E;
            if (topk_probs)
                topk_probs[(long)t * K + k] = 0.0f;
        }
    }
}

/* Compact -> map: routing_map[t,e] = 1 when some slot of t holds e, else 0; dense[t,e] = the
 * binary32 sum, over those slots in ascending k and starting from +0, of their probabilities
 * (a token naming an expert twice sends it the sum).  Ids outside [0, E) are skipped: they
 * route nowhere here (the layout is what reports ids outside [-1, E)).  topk_probs /
 * dense_probs may be NULL. */
void oracle_indices_to_multihot(const int32_t *topk_ids, const float *topk_probs, int T, int K,
                                int E, uint8_t *routing_map, float *dense_probs)
{
    for (int t = 0; t < T; t++) {
        for (int e = 0; e < E; e++) {
            uint8_t hit = 0;
            float acc = 0.0f;
            for (int k = 0; k < K; k++) {
                if (topk_ids[(long)t * K + k] != e)
                    continue;
                hit = 1;
                if (topk_probs)
                    acc = acc + topk_probs[(long)t * K + k];
            }
            routing_map[(long)t * E + e] = hit;
            if (dense_probs)
                dense_probs[(long)t * E + e] = acc;
        }
    }
}
