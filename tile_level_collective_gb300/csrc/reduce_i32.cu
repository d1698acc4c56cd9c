// TREDUCE / reduce_scatter / allreduce kernels for int32_t elements (one translation unit
// per element type so the library builds in parallel).
#include <atomic>

#include "reduce_async.cuh"
#include "reduce_impl.cuh"

namespace ptoc {

cudaError_t launch_reduce_i32(const ReduceParams& p, int op, int vb, int unroll, dim3 grid, cudaStream_t s)
{
    return launch_reduce_t<int32_t>(p, op, vb, unroll, grid, s);
}

int occupancy_reduce_i32(int op, int vb, int unroll) { return occupancy_t<int32_t>(op, vb, unroll); }

cudaError_t launch_async_i32(const ReduceParams& p, int op, int cfg, int grid, cudaStream_t s)
{
    return launch_async_t<int32_t>(p, op, cfg, grid, s);
}

// Resident CTAs per SM of the pipelined kernel on device `dev`, cached; the
// first query of a device also opts the kernel into its shared-memory size.
int occupancy_async_i32(int op, int cfg, int dev)
{
    static std::atomic<int> cache[kMaxDevices][4][kAsyncCfgs];
    if (dev < 0 || dev >= kMaxDevices || op < 0 || op > 3 || cfg < 0 || cfg >= kAsyncCfgs)
        return async_occupancy_t<int32_t>(op, cfg);
    int v = cache[dev][op][cfg].load(std::memory_order_relaxed);
    if (v == 0) {
        v = async_occupancy_t<int32_t>(op, cfg);
        cache[dev][op][cfg].store(v > 0 ? v : -1, std::memory_order_relaxed);
    }
    return v > 0 ? v : 0;
}

}  // namespace ptoc
