/* A plain C caller of libbsmooth.
 *
 * Without arguments: host-side checks only, for hosts without a GPU -- the
 * header compiles as C without any CUDA header, argument errors come back as
 * the documented codes (the fake pointers are never dereferenced), and every
 * status has a text.
 *
 * With "gpu" (built with WITH_CUDA): smooths worked example A (4 atoms;
 * tests/golden) on the device through cudaMalloc'd buffers and checks every
 * value. */
#include <stdio.h>
#include <string.h>

#include "bsmooth.h"

#ifdef WITH_CUDA
#include <cuda_runtime_api.h>
#endif

static int fails = 0;
#define CHECK(cond) do { if (!(cond)) { printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond); ++fails; } } while (0)

static int host_checks(void) {
    void *u = (void *)(1 << 20), *l = (void *)(2 << 20);   /* never dereferenced */
    long long cnt = -1;
    CHECK(bs_smooth_bounds(u, l, -1, 4, NULL, BS_FP32) == BS_ERR_ARG);
    CHECK(bs_smooth_bounds(u, l, 8, 7, NULL, BS_FP32) == BS_ERR_ARG);
    CHECK(bs_smooth_bounds(u, u, 8, 8, NULL, BS_FP32) == BS_ERR_ARG);
    CHECK(bs_smooth_bounds(u, l, 8, 8, NULL, BS_RULE_LITERAL) == BS_ERR_ARG);
    CHECK(bs_smooth_bounds(u, l, 0, 0, NULL, BS_FP32) == BS_OK);
    CHECK(bs_smooth_upper(NULL, 3, 3, NULL, BS_INT32_Q10) == BS_ERR_ARG);
    CHECK(bs_smooth_bounds_batched(u, l, 8, 8, 63, 2, NULL, BS_FP32) == BS_ERR_ARG);
    CHECK(bs_check_feasible(u, l, 8, 8, NULL, BS_FP32, NULL, NULL) == BS_ERR_ARG);
    CHECK(bs_check_feasible(u, l, 0, 0, NULL, BS_FP32, &cnt, NULL) == BS_OK && cnt == 0);
    CHECK(bs_check_feasible_noalloc(u, l, 8, 8, 64, BS_NOALLOC_MAX_BATCH + 1, NULL, BS_FP32,
                                    &cnt) == BS_ERR_ARG);
    for (int s = BS_OK; s <= BS_ERR_INPUT; ++s)
        CHECK(bs_strerror((bs_status)s) != NULL && strlen(bs_strerror((bs_status)s)) > 0);
    CHECK(bs_launch_count() >= 0);
    return fails;
}

#ifdef WITH_CUDA
static int gpu_example_a(void) {
    /* example A: chain 0-1-2-3 with (0,2) known; unknown pairs [1, 100] */
    const float U0[16] = {0, 4, 7, 100,  4, 0, 4, 100,  7, 4, 0, 4,  100, 100, 4, 0};
    const float L0[16] = {0, 3, 6.5f, 1,  3, 0, 3, 1,  6.5f, 3, 0, 3,  1, 1, 3, 0};
    const float Ux[16] = {0, 4, 7, 11,  4, 0, 4, 8,  7, 4, 0, 4,  11, 8, 4, 0};
    const float Lx[16] = {0, 3, 6.5f, 2.5f,  3, 0, 3, 1,  6.5f, 3, 0, 3,  2.5f, 1, 3, 0};
    float *dU, *dL, U[16], L[16];
    long long flags = -1;
    CHECK(cudaMalloc((void **)&dU, sizeof U0) == cudaSuccess);
    CHECK(cudaMalloc((void **)&dL, sizeof L0) == cudaSuccess);
    CHECK(cudaMemcpy(dU, U0, sizeof U0, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dL, L0, sizeof L0, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(bs_smooth_bounds(dU, dL, 4, 4, NULL, BS_FP32 | BS_VALIDATE) == BS_OK);
    CHECK(bs_check_feasible(dU, dL, 4, 4, NULL, BS_FP32, &flags, NULL) == BS_OK && flags == 0);
    CHECK(cudaMemcpy(U, dU, sizeof U, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(L, dL, sizeof L, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(memcmp(U, Ux, sizeof U) == 0);
    CHECK(memcmp(L, Lx, sizeof L) == 0);
    cudaFree(dU);
    cudaFree(dL);
    return fails;
}
#endif

int main(int argc, char **argv) {
#ifdef WITH_CUDA
    if (argc > 1 && strcmp(argv[1], "gpu") == 0)
        gpu_example_a();
    else
        host_checks();
#else
    (void)argc;
    (void)argv;
    host_checks();
#endif
    printf(fails ? "abi_caller: %d failure(s)\n" : "abi_caller: ok\n", fails);
    return fails ? 1 : 0;
}
