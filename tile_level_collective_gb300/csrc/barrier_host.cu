// The self-clearing credit barrier ("Distributed Operators (N6)",
// Barrier-signal protocol) for ranks that are host threads or processes.
//
// The protocol is the one the cooperative kernel runs for ranks on the GPU:
// rank r's window holds one int32 cell per source rank, and a call of G
// generations is, for rank r,
//   for g = 1..G:  cell [p][r] += 1 for every peer p != r   (release)
//                  wait until cell [r][s] >= g for every s != r   (acquire)
//   epilogue:      cell [r][s] -= G for every s != r
// Here every rank is the thread that calls ptoc_credit_barrier_host for it;
// the cells are plain host memory (one process's, or a mapping shared between
// processes) updated with lock-free 32-bit atomics. A wait is bounded by a
// deadline on the steady clock; a rank that gives up records the generation it
// was waiting in and skips its epilogue, leaving its credits, as the page
// describes for an aborted call. No CUDA call is made.
#include <chrono>
#include <cstdint>
#include <thread>

#include <nvtx3/nvToolsExt.h>

#include "ptoc.h"
#include "ptoc_internal.h"

namespace {

inline void credit_add(int32_t* cell, int32_t v) { __atomic_fetch_add(cell, v, __ATOMIC_RELEASE); }

inline int32_t credit_load(const int32_t* cell) { return __atomic_load_n(cell, __ATOMIC_ACQUIRE); }

constexpr uint32_t kSpinPolls = 64;   // polls before the waiting thread starts yielding

bool ranges_overlap(uintptr_t a, uintptr_t an, uintptr_t b, uintptr_t bn)
{
    return an > 0 && bn > 0 && a < b + bn && b < a + an;
}

}  // namespace

static ptoc_status credit_barrier_host(const ptoc_group* signals, int32_t rank, int32_t generations,
                                       int64_t timeout_ns, int32_t* status)
{
    if (!signals || !signals->tensors || !status) return PTOC_ERR_INVALID_ARG;
    const int n = signals->nranks;
    if (n < 1 || n > ptoc::kMaxRanks) return PTOC_ERR_INVALID_ARG;
    if (rank < 0 || rank >= n) return PTOC_ERR_INVALID_ARG;
    if (generations < 0 || generations > (1 << 30)) return PTOC_ERR_INVALID_ARG;
    if (timeout_ns <= 0 || timeout_ns > (int64_t)60 * 1000 * 1000 * 1000) return PTOC_ERR_INVALID_ARG;
    if ((uintptr_t)status % 4 != 0) return PTOC_ERR_INVALID_ARG;
    int32_t* sig[ptoc::kMaxRanks];
    for (int r = 0; r < n; ++r) {
        sig[r] = (int32_t*)signals->tensors[r];
        if (!sig[r] || (uintptr_t)sig[r] % 4 != 0) return PTOC_ERR_INVALID_ARG;
    }
    const uintptr_t wb = (uintptr_t)n * 4u;
    for (int a = 0; a < n; ++a) {
        if (ranges_overlap((uintptr_t)sig[a], wb, (uintptr_t)status, 4)) return PTOC_ERR_ALIAS;
        for (int b = a + 1; b < n; ++b)
            if (ranges_overlap((uintptr_t)sig[a], wb, (uintptr_t)sig[b], wb)) return PTOC_ERR_ALIAS;
    }

    const int me = rank;
    const auto start = std::chrono::steady_clock::now();
    const auto limit = std::chrono::nanoseconds(timeout_ns);
    int32_t st = 0;
    for (int g = 1; g <= generations && st == 0; ++g) {
        for (int peer = 0; peer < n; ++peer)
            if (peer != me) credit_add(sig[peer] + me, 1);
        uint32_t polls = 0;
        while (true) {
            bool ready = true;
            for (int s = 0; s < n && ready; ++s)
                if (s != me && credit_load(sig[me] + s) < g) ready = false;
            if (ready) break;
            if (std::chrono::steady_clock::now() - start > limit) {
                st = g;
                break;
            }
            if (++polls > kSpinPolls) std::this_thread::yield();
        }
    }
    if (st == 0)
        for (int s = 0; s < n; ++s)
            if (s != me) credit_add(sig[me] + s, -generations);
    *status = st;
    return PTOC_OK;
}

extern "C" ptoc_status ptoc_credit_barrier_host(const ptoc_group* signals, int32_t rank, int32_t generations,
                                                int64_t timeout_ns, int32_t* status)
{
    nvtxRangePushA("ptoc_credit_barrier_host");
    const ptoc_status st = credit_barrier_host(signals, rank, generations, timeout_ns, status);
    nvtxRangePop();
    return st;
}
