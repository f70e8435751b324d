/*
 * abi_smoke.c -- libc3.so used from plain C99 through include/c3_api.h only.
 *
 * Built by tests/test_c_abi.py: on any machine it must compile as C99 with
 * warnings as errors and link against libc3.so with every declared entry point
 * resolved (the table below takes each one's address).  With --run, on a GPU,
 * it drives the library through the C ABI alone and checks the results:
 *   - a GEMM whose A is the identity, so C = B^T exactly (small integers are
 *     exact in bf16 and in fp32), for a product C[m][n] = sum_k A[m][k] B[n][k];
 *   - an all-gather of 8 tagged shards, which must equal their rank-order
 *     concatenation ("Optimizing ML Concurrent Computation and Communication
 *     with GPU DMA Engines", review pages: the skeptic's "concrete_test");
 *   - one concurrent baseline run of the pair through c3_run.
 * Exit status 0 and the line "c abi smoke ok" mean success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "c3_api.h"

typedef void (*any_fn)(void);

/* Every entry point of the header: a missing export fails the link. */
static const any_fn k_entry_points[] = {
    (any_fn)c3_get_device_info, (any_fn)c3_strerror,     (any_fn)c3_last_error,    (any_fn)c3_status_check,
    (any_fn)c3_shutdown,        (any_fn)c3_kernel_launches, (any_fn)c3_gemm,       (any_fn)c3_gemm_plan,
    (any_fn)c3_allgather,       (any_fn)c3_alltoall,     (any_fn)c3_allreduce,     (any_fn)c3_run,
    (any_fn)c3_time,            (any_fn)c3_gemm_noalloc, (any_fn)c3_selftest_wait, (any_fn)c3_inject_fault,
    (any_fn)c3_sp_predict,      (any_fn)c3_rp_predict,   (any_fn)c3_l2_flush,      (any_fn)c3_cta_windows,
    (any_fn)c3_rp_predict_elastic,
};

#define N_RANKS 8
#define DIM 128
#define SHARD 4096

static int fail(const char *what, int rc) {
    fprintf(stderr, "%s: %d (%s; %s)\n", what, rc, c3_strerror(rc), c3_last_error());
    return 1;
}

static int cuda_fail(const char *what, cudaError_t e) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
}

/* bf16 of a small integer: the top half of its fp32 bits (exact). */
static uint16_t bf16_of_int(int v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static int run(void) {
    c3_device_info info;
    int rc = c3_get_device_info(&info);
    if (rc) return fail("c3_get_device_info", rc);
    if (info.sm_count <= 0) return fail("sm_count", info.sm_count);

    uint16_t *hA = (uint16_t *)calloc(DIM * DIM, 2), *hB = (uint16_t *)malloc(DIM * DIM * 2);
    float *hC = (float *)malloc(DIM * DIM * 4);
    unsigned char *hs = (unsigned char *)malloc(N_RANKS * SHARD), *ho = (unsigned char *)malloc(N_RANKS * SHARD);
    if (!hA || !hB || !hC || !hs || !ho) return fail("host allocation", -1);
    for (int i = 0; i < DIM; ++i) hA[i * DIM + i] = bf16_of_int(1);
    for (int n = 0; n < DIM; ++n)
        for (int k = 0; k < DIM; ++k) hB[n * DIM + k] = bf16_of_int((n * 7 + k * 3) % 17 - 8);
    for (int r = 0; r < N_RANKS; ++r)
        for (int i = 0; i < SHARD; ++i) hs[r * SHARD + i] = (unsigned char)((r * 31 + i * 7) & 0xff);

    void *dA = NULL, *dB = NULL, *dC = NULL, *dout = NULL, *dsh[N_RANKS];
    cudaError_t e;
    if ((e = cudaMalloc(&dA, DIM * DIM * 2)) || (e = cudaMalloc(&dB, DIM * DIM * 2)) ||
        (e = cudaMalloc(&dC, DIM * DIM * 4)) || (e = cudaMalloc(&dout, N_RANKS * SHARD)))
        return cuda_fail("cudaMalloc", e);
    for (int r = 0; r < N_RANKS; ++r) {
        if ((e = cudaMalloc(&dsh[r], SHARD))) return cuda_fail("cudaMalloc", e);
        if ((e = cudaMemcpy(dsh[r], hs + r * SHARD, SHARD, cudaMemcpyHostToDevice))) return cuda_fail("H2D", e);
    }
    if ((e = cudaMemcpy(dA, hA, DIM * DIM * 2, cudaMemcpyHostToDevice)) ||
        (e = cudaMemcpy(dB, hB, DIM * DIM * 2, cudaMemcpyHostToDevice)))
        return cuda_fail("H2D", e);

    /* the two halves, one call each, on the default stream */
    if ((rc = c3_gemm(dA, dB, (float *)dC, DIM, DIM, DIM, 0, NULL))) return fail("c3_gemm", rc);
    if ((rc = c3_allgather((const void *const *)dsh, dout, SHARD, N_RANKS, C3_ENGINE_SM, 0, NULL)))
        return fail("c3_allgather", rc);
    if ((rc = c3_status_check(NULL))) return fail("c3_status_check", rc);
    if ((e = cudaMemcpy(hC, dC, DIM * DIM * 4, cudaMemcpyDeviceToHost)) ||
        (e = cudaMemcpy(ho, dout, N_RANKS * SHARD, cudaMemcpyDeviceToHost)))
        return cuda_fail("D2H", e);
    for (int m = 0; m < DIM; ++m)
        for (int n = 0; n < DIM; ++n)
            if (hC[m * DIM + n] != (float)((n * 7 + m * 3) % 17 - 8)) return fail("GEMM entry", m * DIM + n);
    if (memcmp(ho, hs, N_RANKS * SHARD) != 0) return fail("all-gather output", -1);

    /* the pair, concurrently, in the baseline mode */
    if ((e = cudaMemset(dC, 0xff, DIM * DIM * 4)) || (e = cudaMemset(dout, 0, N_RANKS * SHARD)))
        return cuda_fail("cudaMemset", e);
    c3_problem p;
    memset(&p, 0, sizeof p);
    p.A = dA;
    p.B = dB;
    p.C = (float *)dC;
    p.M = p.N = p.K = DIM;
    p.coll = C3_COLL_ALLGATHER;
    p.shards = (const void *const *)dsh;
    p.recv = dout;
    p.unit_bytes = SHARD;
    p.nranks = N_RANKS;
    c3_timing t;
    if ((rc = c3_run(&p, C3_MODE_CONCURRENT_SM, 0, 0, &t))) return fail("c3_run", rc);
    if (!(t.t_conc > 0.0) || t.status != 0) return fail("c3_run timing", t.status);
    if ((e = cudaMemcpy(hC, dC, DIM * DIM * 4, cudaMemcpyDeviceToHost)) ||
        (e = cudaMemcpy(ho, dout, N_RANKS * SHARD, cudaMemcpyDeviceToHost)))
        return cuda_fail("D2H", e);
    for (int i = 0; i < DIM * DIM; ++i)
        if (hC[i] != (float)(((i % DIM) * 7 + (i / DIM) * 3) % 17 - 8)) return fail("concurrent GEMM entry", i);
    if (memcmp(ho, hs, N_RANKS * SHARD) != 0) return fail("concurrent all-gather output", -1);

    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dC);
    cudaFree(dout);
    for (int r = 0; r < N_RANKS; ++r) cudaFree(dsh[r]);
    free(hA);
    free(hB);
    free(hC);
    free(hs);
    free(ho);
    if ((rc = c3_shutdown())) return fail("c3_shutdown", rc);
    printf("c abi smoke ok: t_conc %.1f us, %d GEMM CTAs, %d collective CTAs\n", 1e6 * t.t_conc, t.gemm_ctas,
           t.comm_ctas);
    return 0;
}

int main(int argc, char **argv) {
    printf("%d entry points\n", (int)(sizeof k_entry_points / sizeof k_entry_points[0]));
    if (argc > 1 && strcmp(argv[1], "--run") == 0) return run();
    return 0;
}
