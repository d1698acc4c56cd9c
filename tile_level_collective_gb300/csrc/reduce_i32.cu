// TREDUCE / reduce_scatter kernels for int32_t elements (one translation unit
// per element type so the library builds in parallel).
#include "reduce_impl.cuh"

namespace ptoc {

cudaError_t launch_reduce_i32(const ReduceParams& p, int op, int vb, int unroll, dim3 grid, cudaStream_t s)
{
    return launch_reduce_t<int32_t>(p, op, vb, unroll, grid, s);
}

int occupancy_reduce_i32(int op, int vb, int unroll) { return occupancy_t<int32_t>(op, vb, unroll); }

}  // namespace ptoc
