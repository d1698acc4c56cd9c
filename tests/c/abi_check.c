/*
 * A plain C caller of libptoc.so: allocates its own buffers with the CUDA
 * runtime, runs TREDUCE (Sum, Max, Min) over ranks holding base + 100 r (the
 * TREDUCE article's own test, section 7.1), in the register form and in the
 * staged form (PTOC_REDUCE_STAGING), and an all_to_all_v with clamped counts,
 * checks the results against the closed forms, and reads the wait-fault
 * count. Exit status 0 when everything matches; the first mismatch is printed.
 */
#define _POSIX_C_SOURCE 200112L
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ptoc.h"

#define N 4
#define ROWS 37
#define COLS 50
#define LD 56

static int fail(const char* what, long i, long got, long want)
{
    printf("mismatch: %s at %ld: got %ld want %ld\n", what, i, got, want);
    return 1;
}

int main(void)
{
    size_t bytes = (size_t)ROWS * LD * sizeof(int32_t);
    int32_t* host = (int32_t*)malloc(bytes);
    void* src[N];
    void* dst;
    for (int r = 0; r < N; ++r) {
        for (int i = 0; i < ROWS; ++i)
            for (int j = 0; j < LD; ++j)
                host[i * LD + j] = ((7 * i + 3 * j) % 11) - 5 + 100 * r;
        if (cudaMalloc(&src[r], bytes) != cudaSuccess) return 2;
        cudaMemcpy(src[r], host, bytes, cudaMemcpyHostToDevice);
    }
    if (cudaMalloc(&dst, bytes) != cudaSuccess) return 2;
    ptoc_group g = {src, N, 0};
    const ptoc_reduce_op ops[3] = {PTOC_SUM, PTOC_MAX, PTOC_MIN};
    const char* forms[2] = {"regs", "bulk"};
    for (int f = 0; f < 6; ++f) {
        const int o = f % 3;
        setenv("PTOC_REDUCE_STAGING", forms[f / 3], 1);
        cudaMemset(dst, 0xFF, bytes);
        ptoc_status st = ptoc_treduce(&g, dst, ROWS, COLS, ROWS, COLS, LD, ops[o], PTOC_I32, 0);
        if (st != PTOC_OK) {
            printf("ptoc_treduce: %s\n", ptoc_status_string(st));
            return 1;
        }
        cudaMemcpy(host, dst, bytes, cudaMemcpyDeviceToHost);
        for (int i = 0; i < ROWS; ++i)
            for (int j = 0; j < LD; ++j) {
                long base = ((7 * i + 3 * j) % 11) - 5;
                long want = j >= COLS ? -1
                          : o == 0 ? N * base + 100 * N * (N - 1) / 2
                          : o == 1 ? base + 100 * (N - 1) : base;
                if (host[i * LD + j] != want) return fail("treduce", i * LD + j, host[i * LD + j], want);
            }
    }
    unsetenv("PTOC_REDUCE_STAGING");
    uint32_t faults = 1;
    if (ptoc_wait_faults(&faults) != PTOC_OK || faults != 0) return fail("wait faults", 0, (long)faults, 0);
    /* bad arguments come back as status codes, nothing launched */
    if (ptoc_treduce(&g, dst, ROWS, COLS, ROWS, COLS, LD, PTOC_PROD, PTOC_I32, 0) != PTOC_ERR_UNSUPPORTED)
        return fail("prod status", 0, 0, PTOC_ERR_UNSUPPORTED);
    if (ptoc_treduce(&g, src[1], ROWS, COLS, ROWS, COLS, LD, PTOC_SUM, PTOC_I32, 0) != PTOC_ERR_ALIAS)
        return fail("alias status", 0, 0, PTOC_ERR_ALIAS);

    /* all_to_all_v: 2 ranks, 6 target rows (MAX_RECV 3), 4 int32 per row */
    enum { R = 2, TR = 6, SZ = 4 };
    int32_t in_h[R][TR * SZ], out_h[TR * SZ];
    int32_t sc_h[R][R] = {{-1, 5}, {2, 3}};
    void *in_d[R], *tg_d[R];
    int32_t *sc_d[R], *rc_d[R];
    for (int s = 0; s < R; ++s) {
        for (int k = 0; k < TR * SZ; ++k) in_h[s][k] = 1000 * s + k;
        cudaMalloc(&in_d[s], sizeof(in_h[s]));
        cudaMalloc(&tg_d[s], sizeof(in_h[s]));
        cudaMalloc((void**)&sc_d[s], sizeof(sc_h[s]));
        cudaMalloc((void**)&rc_d[s], sizeof(sc_h[s]));
        cudaMemcpy(in_d[s], in_h[s], sizeof(in_h[s]), cudaMemcpyHostToDevice);
        cudaMemcpy(sc_d[s], sc_h[s], sizeof(sc_h[s]), cudaMemcpyHostToDevice);
        cudaMemset(tg_d[s], 0xFF, sizeof(in_h[s]));
    }
    ptoc_group gi = {in_d, R, 0}, gt = {tg_d, R, 0};
    ptoc_status st = ptoc_all_to_all_v(&gi, &gt, (const int32_t* const*)sc_d, rc_d, TR, SZ, PTOC_I32, 0);
    if (st != PTOC_OK) {
        printf("ptoc_all_to_all_v: %s\n", ptoc_status_string(st));
        return 1;
    }
    for (int d = 0; d < R; ++d) {
        int32_t rc[R];
        cudaMemcpy(rc, rc_d[d], sizeof(rc), cudaMemcpyDeviceToHost);
        cudaMemcpy(out_h, tg_d[d], sizeof(out_h), cudaMemcpyDeviceToHost);
        for (int s = 0; s < R; ++s) {
            long c = sc_h[s][d] < 0 ? 0 : (sc_h[s][d] > 3 ? 3 : sc_h[s][d]);
            if (rc[s] != c) return fail("recv_counts", d * R + s, rc[s], c);
            for (int i = 0; i < 3; ++i)
                for (int k = 0; k < SZ; ++k) {
                    long got = out_h[(s * 3 + i) * SZ + k];
                    long want = i < c ? in_h[s][(d * 3 + i) * SZ + k] : -1;
                    if (got != want) return fail("target", (s * 3 + i) * SZ + k, got, want);
                }
        }
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    printf("abi_check: ok\n");
    return 0;
}
