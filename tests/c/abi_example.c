/*
 * A C caller of libep_gb300.so: no Python, no torch, only include/ep.h and the CUDA runtime.
 *
 * On the hand-worked routing of tests/golden/layout_example.txt (T=4 tokens, top-2 of E=3
 * experts, a fused shared expert, 3 partitions) it runs the layout, the BF16 dispatch, the
 * combine, the fused layout + NVFP4 call, both backward passes and the no-allocation layout,
 * and checks every value against numbers derived by hand.  Token t's row is all t+1.
 *   - the layout: row_offsets, row_of, expert_ids, src_info of the golden file;
 *   - the dispatch: every row holds its source token's row;
 *   - the combine with identity experts and probabilities 0.25: token t gets
 *     (t+1) * (0.25 * valid slots + 1), exact in bf16 (1.5, 2.5, 4.5, 6);
 *   - NVFP4: a constant row has block maximum = row maximum a = t+1, so the global scale is
 *     g = 2688/a, every block scale is (a g)/6 = 448 (E4M3 0x7E), every element encodes
 *     a * g / 448 = 6 (E2M1 0x7, two per byte: 0x77), and the row's inverse scale is
 *     bf16(1/g): 0x39C3, 0x3A43, 0x3A92, 0x3AC3 for g = 2688, 1344, 896, 672;
 *   - combine_bwd with grad_out = x and the dispatched rows as expert outputs: a routed row of
 *     token t gets bf16(0.25 (t+1)), its shared row t+1, and grad_p = sum over the 16 columns
 *     of (t+1)(t+1) = 16 (t+1)^2 for a routed slot, 0 for the unused one;
 *   - dispatch_bwd of the dispatched rows: token t gets (t+1)(valid slots + 1): 3, 4, 9, 12;
 *   - the status: 0 at capacity 3, the overflow code at capacity 2; an invalid argument is
 *     refused before any work.
 * Exits 0 when everything matches.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep.h"

#define T 4
#define K 2
#define E 3
#define S 1
#define P 3
#define H 16
#define G (E + S)
#define RMAX (T * K + S * T)

static int failures = 0;

static void expect_eq(const char *what, long got, long want)
{
    if (got != want) {
        fprintf(stderr, "%s: got %ld, want %ld\n", what, got, want);
        ++failures;
    }
}

static uint16_t bf16_of_small(float v)   /* exact for the small values used here */
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return (uint16_t)(u >> 16);
}

static void *dev_alloc(size_t bytes)
{
    void *p = NULL;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return NULL;
    }
    cudaMemset(p, 0, bytes);
    return p;
}

int main(void)
{
    const int32_t ids[T * K] = {2, 0, 1, -1, 0, 2, 2, 1};
    const int32_t want_offsets[G + 1] = {0, 2, 4, 7, 11};
    const int32_t want_row_of[T * K] = {4, 0, 2, -1, 1, 5, 6, 3};
    const int32_t want_expert[11] = {0, 0, 1, 1, 2, 2, 2, 3, 3, 3, 3};
    const int32_t want_src[22] = {0, 1, 2, 0, 1, 0, 3, 1, 0, 0, 2, 1, 3, 0, 0, 2, 1, 2, 2, 2, 3, 2};
    const float want_out[T] = {1.5f, 2.5f, 4.5f, 6.0f};

    uint16_t x[T * H];
    float probs[T * K];
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < H; ++i)
            x[t * H + i] = bf16_of_small((float)(t + 1));
    for (int i = 0; i < T * K; ++i)
        probs[i] = 0.25f;

    ep_layout_t L;
    memset(&L, 0, sizeof L);
    L.row_offsets = dev_alloc(sizeof(int32_t) * (G + 1));
    L.expert_ids = dev_alloc(sizeof(int32_t) * RMAX);
    L.src_info = dev_alloc(sizeof(int32_t) * 2 * RMAX);
    L.row_of = dev_alloc(sizeof(int32_t) * T * K);
    L.part_tokens = dev_alloc(sizeof(int32_t) * P);
    L.status = dev_alloc(16);
    L.workspace_bytes = ep_layout_workspace_bytes(T, K, E, S);
    L.workspace = dev_alloc(L.workspace_bytes);
    int32_t *d_ids = dev_alloc(sizeof ids);
    uint16_t *d_x = dev_alloc(sizeof x);
    float *d_probs = dev_alloc(sizeof probs);
    uint16_t *d_rows = dev_alloc(sizeof(uint16_t) * RMAX * H);
    uint16_t *d_out = dev_alloc(sizeof(uint16_t) * T * H);
    if (!L.workspace || !d_rows || !d_out)
        return 1;
    cudaMemcpy(d_ids, ids, sizeof ids, cudaMemcpyHostToDevice);
    cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice);
    cudaMemcpy(d_probs, probs, sizeof probs, cudaMemcpyHostToDevice);

    /* an invalid argument is refused before any work: partitions that do not divide E */
    expect_eq("invalid P", ep_dispatch_layout(d_ids, T, K, E, 2, 3, S, &L, NULL), EP_ERR_INVALID_ARG);

    expect_eq("layout", ep_dispatch_layout(d_ids, T, K, E, P, 3, S, &L, NULL), EP_OK);
    expect_eq("bf16 dispatch", ep_dispatch_bf16(d_x, H, &L, d_rows, NULL), EP_OK);
    /* identity experts: the dispatched rows are the expert outputs */
    expect_eq("combine", ep_combine(d_rows, d_probs, H, &L, d_out, NULL), EP_OK);
    int32_t status = -1;
    expect_eq("read_status", ep_read_status(&L, NULL, &status), EP_OK);
    expect_eq("status word", status, 0);

    int32_t offsets[G + 1], row_of[T * K], expert[RMAX], src[2 * RMAX];
    uint16_t rows[RMAX * H], out[T * H];
    cudaMemcpy(offsets, L.row_offsets, sizeof offsets, cudaMemcpyDeviceToHost);
    cudaMemcpy(row_of, L.row_of, sizeof row_of, cudaMemcpyDeviceToHost);
    cudaMemcpy(expert, L.expert_ids, sizeof expert, cudaMemcpyDeviceToHost);
    cudaMemcpy(src, L.src_info, sizeof src, cudaMemcpyDeviceToHost);
    cudaMemcpy(rows, d_rows, sizeof rows, cudaMemcpyDeviceToHost);
    cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost);
    for (int g = 0; g <= G; ++g)
        expect_eq("row_offsets", offsets[g], want_offsets[g]);
    for (int i = 0; i < T * K; ++i)
        expect_eq("row_of", row_of[i], want_row_of[i]);
    for (int r = 0; r < 11; ++r) {
        expect_eq("expert_ids", expert[r], want_expert[r]);
        expect_eq("src_info token", src[2 * r], want_src[2 * r]);
        expect_eq("src_info slot", src[2 * r + 1], want_src[2 * r + 1]);
        for (int i = 0; i < H; ++i)
            expect_eq("dispatched row", rows[r * H + i], bf16_of_small((float)(want_src[2 * r] + 1)));
    }
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < H; ++i)
            expect_eq("combined", out[t * H + i], bf16_of_small(want_out[t]));

    /* the fused layout + NVFP4 call */
    const uint16_t want_inv[T] = {0x39C3, 0x3A43, 0x3A92, 0x3AC3};
    uint8_t *d_fp4 = dev_alloc(RMAX * H / 2);
    uint8_t *d_sc = dev_alloc(RMAX * H / 16);
    uint16_t *d_inv = dev_alloc(sizeof(uint16_t) * RMAX);
    int32_t *d_so = dev_alloc(sizeof(int32_t) * (G + 1));
    if (!d_fp4 || !d_sc || !d_inv || !d_so)
        return 1;
    expect_eq("layout + nvfp4", ep_dispatch_layout_nvfp4(d_ids, T, K, E, P, 3, S, d_x, H, &L, d_fp4, d_sc,
                                                          d_inv, d_so, NULL), EP_OK);
    uint8_t fp4[RMAX * H / 2], sc[RMAX * H / 16];
    uint16_t inv[RMAX];
    int32_t so[G + 1];
    cudaMemcpy(fp4, d_fp4, sizeof fp4, cudaMemcpyDeviceToHost);
    cudaMemcpy(sc, d_sc, sizeof sc, cudaMemcpyDeviceToHost);
    cudaMemcpy(inv, d_inv, sizeof inv, cudaMemcpyDeviceToHost);
    cudaMemcpy(so, d_so, sizeof so, cudaMemcpyDeviceToHost);
    cudaMemcpy(row_of, L.row_of, sizeof row_of, cudaMemcpyDeviceToHost);
    for (int i = 0; i < T * K; ++i)
        expect_eq("fused call row_of", row_of[i], want_row_of[i]);
    for (int g = 0; g <= G; ++g)
        expect_eq("scales_offsets", so[g], want_offsets[g]);
    for (int r = 0; r < 11; ++r) {
        for (int b = 0; b < H / 2; ++b)
            expect_eq("E2M1 codes", fp4[r * H / 2 + b], 0x77);
        for (int b = 0; b < H / 16; ++b)
            expect_eq("E4M3 block scale", sc[r * H / 16 + b], 0x7E);
        expect_eq("inverse global scale", inv[r], want_inv[want_src[2 * r]]);
    }

    /* the backward passes, on the layout of the fused call (the same routing) */
    uint16_t *d_gy = dev_alloc(sizeof(uint16_t) * RMAX * H);
    float *d_gp = dev_alloc(sizeof(float) * T * K);
    uint16_t *d_gx = dev_alloc(sizeof(uint16_t) * T * H);
    if (!d_gy || !d_gp || !d_gx)
        return 1;
    expect_eq("combine_bwd", ep_combine_bwd(d_x, d_rows, d_probs, H, &L, d_gy, d_gp, NULL), EP_OK);
    expect_eq("dispatch_bwd", ep_dispatch_bwd(d_rows, H, &L, d_gx, NULL), EP_OK);
    uint16_t gy[RMAX * H], gx[T * H];
    float gp[T * K];
    cudaMemcpy(gy, d_gy, sizeof gy, cudaMemcpyDeviceToHost);
    cudaMemcpy(gp, d_gp, sizeof gp, cudaMemcpyDeviceToHost);
    cudaMemcpy(gx, d_gx, sizeof gx, cudaMemcpyDeviceToHost);
    for (int r = 0; r < 11; ++r) {
        const int t = want_src[2 * r], shared = want_src[2 * r + 1] == K;
        for (int i = 0; i < H; ++i)
            expect_eq("grad_y", gy[r * H + i], bf16_of_small(shared ? (float)(t + 1) : 0.25f * (float)(t + 1)));
    }
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            expect_eq("grad_p", (long)gp[t * K + k], ids[t * K + k] < 0 ? 0 : 16L * (t + 1) * (t + 1));
    const float want_gx[T] = {3.0f, 4.0f, 9.0f, 12.0f};
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < H; ++i)
            expect_eq("grad_x", gx[t * H + i], bf16_of_small(want_gx[t]));

    /* the no-allocation layout: no workspace, the same layout */
    ep_layout_t N = L;
    N.workspace = NULL;
    N.workspace_bytes = 0;
    cudaMemset(N.row_of, 0, sizeof(int32_t) * T * K);
    cudaMemset(N.expert_ids, 0, sizeof(int32_t) * RMAX);
    cudaMemset(N.src_info, 0, sizeof(int32_t) * 2 * RMAX);
    expect_eq("noalloc layout", ep_dispatch_layout_noalloc(d_ids, T, K, E, P, 3, S, &N, NULL), EP_OK);
    expect_eq("noalloc read_status", ep_read_status(&N, NULL, &status), EP_OK);
    cudaMemcpy(row_of, N.row_of, sizeof row_of, cudaMemcpyDeviceToHost);
    cudaMemcpy(expert, N.expert_ids, sizeof expert, cudaMemcpyDeviceToHost);
    cudaMemcpy(src, N.src_info, sizeof src, cudaMemcpyDeviceToHost);
    for (int i = 0; i < T * K; ++i)
        expect_eq("noalloc row_of", row_of[i], want_row_of[i]);
    for (int r = 0; r < 11; ++r) {
        expect_eq("noalloc expert_ids", expert[r], want_expert[r]);
        expect_eq("noalloc src_info token", src[2 * r], want_src[2 * r]);
        expect_eq("noalloc src_info slot", src[2 * r + 1], want_src[2 * r + 1]);
    }

    /* capacity 2: partition 2 receives 3 tokens, so the overflow is reported */
    expect_eq("layout C=2", ep_dispatch_layout(d_ids, T, K, E, P, 2, S, &L, NULL), EP_OK);
    expect_eq("read_status C=2", ep_read_status(&L, NULL, &status), EP_ERR_OVERFLOW);
    expect_eq("status word C=2", status, EP_STATUS_OVERFLOW);
    if (ep_strerror(EP_ERR_OVERFLOW) == NULL)
        ++failures;

    if (failures)
        fprintf(stderr, "%d mismatches\n", failures);
    else
        printf("C ABI example ok\n");
    return failures ? 1 : 0;
}
