// TREDUCE / reduce_scatter / allreduce kernels for float elements (one translation unit
// per element type so the library builds in parallel).
#include "reduce_forms.cuh"

namespace ptoc {

cudaError_t launch_reduce_f32(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s)
{
    return launch_reduce_t<float>(p, op, vb, grid, s);
}

cudaError_t launch_tma_reduce_f32(const TmaReduceParams& p, int op, cudaStream_t s)
{
    return launch_tma_reduce_t<float>(p, op, s);
}

cudaError_t take_stage_faults_f32(uint32_t* count)
{
    return take_stage_faults(count);
}

}  // namespace ptoc
