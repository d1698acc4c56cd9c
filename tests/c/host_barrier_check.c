/*
 * A plain C caller of ptoc_credit_barrier_host ("Distributed Operators (N6)",
 * Barrier-signal protocol) with POSIX threads as ranks; no GPU is needed.
 * 1. Eight ranks, 500 generations, three calls in a row: every rank reports
 *    0 and every cell is back at zero after each call.
 * 2. Rank 5 never calls: the other seven give up in generation 1, and each
 *    of them has left exactly one credit in every other window (rank 5's
 *    included), none in its own.
 * Exit status 0 when everything matches; the first mismatch is printed.
 */
#include <pthread.h>
#include <stdio.h>
#include <string.h>

#include "ptoc.h"

#define N 8

static int32_t cells[N][N];
static int32_t status_of[N];
static void* windows[N];
static ptoc_group group;
static int32_t generations;
static int64_t timeout_ns;

static void* rank_main(void* arg)
{
    int32_t r = (int32_t)(long)arg;
    if (ptoc_credit_barrier_host(&group, r, generations, timeout_ns, &status_of[r]) != PTOC_OK)
        status_of[r] = -100;
    return NULL;
}

static void run(int absent)
{
    pthread_t t[N];
    for (int r = 0; r < N; ++r) status_of[r] = -1;
    for (int r = 0; r < N; ++r)
        if (r != absent) pthread_create(&t[r], NULL, rank_main, (void*)(long)r);
    for (int r = 0; r < N; ++r)
        if (r != absent) pthread_join(t[r], NULL);
}

int main(void)
{
    for (int r = 0; r < N; ++r) windows[r] = cells[r];
    group.tensors = windows;
    group.nranks = N;
    group.root = 0;

    generations = 500;
    timeout_ns = 20LL * 1000 * 1000 * 1000;
    for (int call = 0; call < 3; ++call) {
        run(-1);
        for (int r = 0; r < N; ++r)
            if (status_of[r] != 0) {
                printf("mismatch: complete call %d, rank %d status %d\n", call, r, status_of[r]);
                return 1;
            }
        for (int p = 0; p < N; ++p)
            for (int s = 0; s < N; ++s)
                if (cells[p][s] != 0) {
                    printf("mismatch: complete call %d, cell [%d][%d] = %d\n", call, p, s, cells[p][s]);
                    return 1;
                }
    }

    const int absent = 5;
    generations = 3;
    timeout_ns = 100LL * 1000 * 1000;
    run(absent);
    for (int r = 0; r < N; ++r)
        if (r != absent && status_of[r] != 1) {
            printf("mismatch: absent rank, rank %d status %d\n", r, status_of[r]);
            return 1;
        }
    for (int p = 0; p < N; ++p)
        for (int s = 0; s < N; ++s) {
            int want = (s != absent && s != p) ? 1 : 0;
            if (cells[p][s] != want) {
                printf("mismatch: absent rank, cell [%d][%d] = %d, want %d\n", p, s, cells[p][s], want);
                return 1;
            }
        }

    if (ptoc_credit_barrier_host(&group, N, 1, timeout_ns, &status_of[0]) != PTOC_ERR_INVALID_ARG) {
        printf("mismatch: rank out of range accepted\n");
        return 1;
    }
    printf("host barrier: ok\n");
    return 0;
}
