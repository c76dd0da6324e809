/*
 * A C caller of libep_gb300.so: no Python, no torch, only include/ep.h and the CUDA runtime.
 *
 * On the hand-worked routing of tests/golden/layout_example.txt (T=4 tokens, top-2 of E=3
 * experts, a fused shared expert, 3 partitions) it runs the layout, the BF16 dispatch and the
 * combine, and checks every value against numbers derived by hand:
 *   - the layout: row_offsets, row_of, expert_ids, src_info of the golden file;
 *   - the dispatch: every row holds its source token's row (token t's row is all t+1);
 *   - the combine with identity experts and probabilities 0.25: token t gets
 *     (t+1) * (0.25 * valid slots + 1), exact in bf16 (1.5, 2.5, 4.5, 6);
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
