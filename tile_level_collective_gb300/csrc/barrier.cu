// The self-clearing credit barrier ("Distributed Operators (N6)",
// Barrier-signal protocol) for ranks simulated on one GPU.
//
// Rank r's signal window holds one int32 cell per source rank. A call of G
// generations is, for rank r:
//   for g = 1..G:  notify every peer p != r: cell [p][r] += 1  (atomic add,
//                  release: earlier writes are visible before the credit)
//                  wait until cell [r][s] >= g for every s != r (acquire)
//   epilogue:      cell [r][s] -= G for every s != r
// Adds are commutative, so a complete call leaves every cell at zero whatever
// the interleaving, and the next call starts from zero.
//
// All ranks that take part run in ONE cooperative launch (one warp each, all
// co-resident), so the waits only ever wait on warps of the same grid. A rank
// that is not launched never notifies; the others then time out. Every wait is
// bounded by a deadline on %globaltimer and by an iteration cap; a timed-out
// rank records the generation it was waiting in and returns without its
// epilogue, leaving its credits behind (the page: an aborted call leaves the
// signal non-zero until a host-side reset).
#include <cuda_runtime.h>

#include "ptoc_internal.h"

namespace ptoc {

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void credit_add(int32_t* cell, int32_t v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(cell), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t credit_load(const int32_t* cell)
{
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cell) : "memory");
    return v;
}

constexpr uint32_t kMaxPolls = 1u << 24;   // iteration cap behind the deadline
constexpr uint32_t kSpinPolls = 64;        // polls before the nanosleep back-off starts

__global__ void __launch_bounds__(32) credit_barrier_kernel(const __grid_constant__ BarrierParams p)
{
    const int me = p.local[blockIdx.x];
    const int n = p.nranks;
    const int lane = threadIdx.x;
    const unsigned full = 0xffffffffu;
    const uint64_t start = global_ns();
    int32_t status = 0;

    for (int g = 1; g <= p.generations && status == 0; ++g) {
        for (int peer = lane; peer < n; peer += 32)
            if (peer != me) credit_add(p.sig[peer] + me, 1);
        uint32_t polls = 0;
        unsigned pause = 32;
        while (true) {
            bool ready = true;
            for (int s = lane; s < n; s += 32)
                if (s != me && credit_load(p.sig[me] + s) < g) ready = false;
            if (__all_sync(full, ready)) break;
            // warp-uniform give-up decision
            const bool late = (global_ns() - start > (uint64_t)p.timeout_ns) || (++polls > kMaxPolls);
            if (__any_sync(full, late)) {
                status = g;
                break;
            }
            if (polls > kSpinPolls) {
                __nanosleep(pause);
                if (pause < 1024) pause <<= 1;
            }
        }
    }
    if (status == 0)
        for (int s = lane; s < n; s += 32)
            if (s != me) credit_add(p.sig[me] + s, -p.generations);
    if (lane == 0) p.status[blockIdx.x] = status;
}

cudaError_t launch_credit_barrier(const BarrierParams& p, cudaStream_t s)
{
    void* args[] = {(void*)&p};
    return cudaLaunchCooperativeKernel((const void*)credit_barrier_kernel, dim3((unsigned)p.nlocal), dim3(32),
                                       args, 0, s);
}

}  // namespace ptoc
