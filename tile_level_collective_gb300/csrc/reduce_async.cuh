// TREDUCE / reduce_scatter / allreduce, pipelined through shared memory.
//
// Same arithmetic as reduce_kernel (root first, then ascending ranks; binary32
// accumulation; raw-encoding select for 16-bit Max / Min). What differs is how
// the bytes are kept in flight: the register kernel holds its loads in
// registers, which caps it at two resident CTAs per SM and drains the memory
// pipe at every tile boundary. Here each thread streams its 16-byte vectors
// with cp.async (global -> shared, L1 bypass) into a ring of S stages; a stage
// holds G ranks of one tile. While the thread reduces stage i it already has
// stages i+1 .. i+S-1 in flight, so the loads of later ranks and tiles overlap
// the reduction of the current one, and in-flight bytes are bounded by shared
// memory (S * G * 4 KiB per CTA) rather than by registers.
//
// Each thread reads back only the shared-memory slots it filled itself, so
// cp.async.wait_group alone orders the copy before the read: no CTA barrier,
// no spin loop. The grid is persistent (CTAs = SMs x resident CTAs per SM)
// and walks the tile list round robin.
#pragma once

#include "reduce_impl.cuh"

namespace ptoc {

__device__ __forceinline__ void cp_async16(uint4* smem, const void* gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int K>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory"); }

__device__ __forceinline__ Words<4> lds128(const uint4* p)
{
    const uint4 v = *p;
    Words<4> r;
    r.w[0] = v.x;
    r.w[1] = v.y;
    r.w[2] = v.z;
    r.w[3] = v.w;
    return r;
}

// Cursor over this CTA's work items (tile m, rank group g), in issue order.
struct ItemCursor {
    int64_t row, seg;     // tile coordinates
    int g;                // rank group
    int64_t left;         // items not yet visited
};

__device__ __forceinline__ void cursor_init(ItemCursor& c, const ReduceParams& p, int64_t items)
{
    c.row = (int64_t)blockIdx.x / p.tpr;
    c.seg = (int64_t)blockIdx.x - c.row * p.tpr;
    c.g = 0;
    c.left = items;
}

// Advance by one item: next group, or the CTA's next tile (t += gridDim.x),
// done with the precomputed quotient / remainder of gridDim.x by tpr.
__device__ __forceinline__ void cursor_next(ItemCursor& c, const ReduceParams& p, int ngroups,
                                            int64_t dq, int64_t dr)
{
    --c.left;
    if (++c.g == ngroups) {
        c.g = 0;
        c.seg += dr;
        c.row += dq;
        if (c.seg >= p.tpr) {
            c.seg -= p.tpr;
            ++c.row;
        }
    }
}

template <class T, int OP, int S, int G, int B>
__global__ void __launch_bounds__(B, 512 / B) reduce_async_kernel(const __grid_constant__ ReduceParams p)
{
    extern __shared__ uint4 stage[];          // [S][G][B] 16-byte slots
    pdl_enter();
    constexpr int VE = 16 / (int)sizeof(T);
    const int n = p.nranks;
    const int ngroups = (n + G - 1) / G;
    const int64_t my_tiles =
        (p.ntiles > (int64_t)blockIdx.x) ? (p.ntiles - 1 - (int64_t)blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t items = my_tiles * ngroups;
    const int64_t dq = (int64_t)gridDim.x / p.tpr;
    const int64_t dr = (int64_t)gridDim.x - dq * p.tpr;

    ItemCursor in, out;
    cursor_init(in, p, items);
    cursor_init(out, p, items);
    int in_slot = 0, out_slot = 0;

    // issue the copies of the item under the `in` cursor (an empty group when
    // there is none, so that every iteration commits exactly one group)
    auto issue = [&]() {
        if (in.left > 0) {
            const int64_t v = in.seg * B + threadIdx.x;
            if (v < p.vpr) {
                const int64_t off = in.row * p.ld * (int64_t)sizeof(T) + v * 16;
                uint4* slot = stage + (size_t)in_slot * G * B + threadIdx.x;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const int r = in.g * G + j;
                    if (r < n) cp_async16(slot + j * B, (const char*)p.src[r] + off);
                }
            }
            cursor_next(in, p, ngroups, dq, dr);
            in_slot = (in_slot + 1 == S) ? 0 : in_slot + 1;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue();

    VecAcc<T, OP, 4> acc;
    for (int64_t i = 0; i < items; ++i) {
        issue();
        cp_async_wait<S - 1>();          // this thread's copies of item i have landed
        const int64_t v = out.seg * B + threadIdx.x;
        const bool last_group = (out.g == ngroups - 1);
        if (v < p.vpr) {
            const uint4* slot = stage + (size_t)out_slot * G * B + threadIdx.x;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int r = out.g * G + j;
                if (r < n) {
                    const Words<4> x = lds128(slot + j * B);
                    if (r == 0) acc.init(x);
                    else acc.add(x);
                }
            }
            if (last_group)
                store_result<4>(p, out.row, out.row * p.ld * (int64_t)sizeof(T) + v * 16, acc.out());
        }
        if (last_group && p.tail > 0 && out.seg == p.tpr - 1) {
            using Raw = typename Scalar<T>::Raw;
            for (int c = threadIdx.x; c < p.tail; c += B) {
                const int64_t e = out.row * p.ld + p.vpr * VE + c;
                store_elem<Raw>(p, out.row, e, reduce_one<T, OP>(p, e));
            }
        }
        cursor_next(out, p, ngroups, dq, dr);
        out_slot = (out_slot + 1 == S) ? 0 : out_slot + 1;
    }
    cp_async_wait<0>();
}

template <class T, int OP, int C>
cudaError_t launch_async_cfg(const ReduceParams& p, int grid, cudaStream_t s)
{
    return launch_kernel(reduce_async_kernel<T, OP, kAsyncS[C], kAsyncG[C], kAsyncB[C]>, dim3((unsigned)grid),
                         (unsigned)kAsyncB[C], async_smem_bytes(C), s, p);
}

// Resident CTAs per SM of one pipelined kernel (sets the shared-memory opt-in
// of the instantiation first).
template <class T, int OP, int C>
int async_occupancy_cfg()
{
    auto k = reduce_async_kernel<T, OP, kAsyncS[C], kAsyncG[C], kAsyncB[C]>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)async_smem_bytes(C)) !=
        cudaSuccess)
        return 0;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kAsyncB[C], async_smem_bytes(C)) != cudaSuccess)
        return 0;
    return b;
}

template <class T, int OP>
cudaError_t launch_async_op(const ReduceParams& p, int cfg, int grid, cudaStream_t s)
{
    switch (cfg) {
    case 1: return launch_async_cfg<T, OP, 1>(p, grid, s);
    case 2: return launch_async_cfg<T, OP, 2>(p, grid, s);
    case 3: return launch_async_cfg<T, OP, 3>(p, grid, s);
    case 4: return launch_async_cfg<T, OP, 4>(p, grid, s);
    case 5: return launch_async_cfg<T, OP, 5>(p, grid, s);
    default: return launch_async_cfg<T, OP, 0>(p, grid, s);
    }
}

template <class T, int OP>
int async_occupancy_op(int cfg)
{
    switch (cfg) {
    case 1: return async_occupancy_cfg<T, OP, 1>();
    case 2: return async_occupancy_cfg<T, OP, 2>();
    case 3: return async_occupancy_cfg<T, OP, 3>();
    case 4: return async_occupancy_cfg<T, OP, 4>();
    case 5: return async_occupancy_cfg<T, OP, 5>();
    default: return async_occupancy_cfg<T, OP, 0>();
    }
}

template <class T>
cudaError_t launch_async_t(const ReduceParams& p, int op, int cfg, int grid, cudaStream_t s)
{
    switch (op) {
    case kSum: return launch_async_op<T, kSum>(p, cfg, grid, s);
    case kMax: return launch_async_op<T, kMax>(p, cfg, grid, s);
    case kProd: return launch_async_op<T, kProd>(p, cfg, grid, s);
    default: return launch_async_op<T, kMin>(p, cfg, grid, s);
    }
}

template <class T>
int async_occupancy_t(int op, int cfg)
{
    switch (op) {
    case kSum: return async_occupancy_op<T, kSum>(cfg);
    case kMax: return async_occupancy_op<T, kMax>(cfg);
    case kProd: return async_occupancy_op<T, kProd>(cfg);
    default: return async_occupancy_op<T, kMin>(cfg);
    }
}

}  // namespace ptoc
