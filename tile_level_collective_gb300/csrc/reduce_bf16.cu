// TREDUCE / reduce_scatter kernels for __nv_bfloat16 elements (one translation unit
// per element type so the library builds in parallel).
#include "reduce_impl.cuh"

namespace ptoc {

cudaError_t launch_reduce_bf16(const ReduceParams& p, int op, int vb, int unroll, dim3 grid, cudaStream_t s)
{
    return launch_reduce_t<__nv_bfloat16>(p, op, vb, unroll, grid, s);
}

int occupancy_reduce_bf16(int op, int vb, int unroll) { return occupancy_t<__nv_bfloat16>(op, vb, unroll); }

}  // namespace ptoc
