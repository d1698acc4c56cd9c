// TREDUCE / reduce_scatter / allreduce kernels for __nv_bfloat16 elements (one translation unit
// per element type so the library builds in parallel).
#include "reduce_forms.cuh"

namespace ptoc {

cudaError_t launch_reduce_bf16(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s)
{
    return launch_reduce_t<__nv_bfloat16>(p, op, vb, grid, s);
}

cudaError_t launch_tma_reduce_bf16(const TmaReduceParams& p, int op, cudaStream_t s)
{
    return launch_tma_reduce_t<__nv_bfloat16>(p, op, s);
}

cudaError_t take_stage_faults_bf16(uint32_t* count)
{
    return take_stage_faults(count);
}

}  // namespace ptoc
