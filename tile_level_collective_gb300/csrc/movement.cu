// Window-layout data movement ("Distributed Operators (N6)"): allgather,
// broadcast, all_to_all_v, symmetric all_to_all and the all_to_all_v combine.
//
// allgather (op table): row chunk r of window r is copied into row chunk r of
// every other window. broadcast (op table): the root's rows are copied into
// every other window. One read, N-1 writes per element: each thread loads its
// vectors once and stores them N-1 times.
//
// all_to_all_v (pld.tensor.all_to_all_v): for every (sender s, destination
// d) the clamped count c = clamp(send_counts[s][d], 0, MAX_RECV) is published
// to recv_counts[d][s], and c packed rows move from input s (rows
// d*MAX_RECV ..) to target d (rows s*MAX_RECV ..). The symmetric all_to_all
// (op table) is the same exchange with every count equal to MAX_RECV. The
// combine (pld.tensor.put / remote_store with AtomicType kAdd) is the return
// leg: rank d pushes the recv_counts[d][s] rows it holds from s back to s's
// output, overwriting or adding. Because the rows of one pair are contiguous
// on both sides, each pair is one contiguous copy of c * row_bytes bytes. The
// counts live on the device, so the grid is sized for the largest possible
// run: grid.y is the pair, grid.x the tile of the pair's run, one tile per
// block. A block reads its pair's count (one L2-resident integer), publishes
// it if it is the pair's first block, and exits at once when its tile lies
// past the run; the hardware block scheduler hands out the live tiles in
// order as blocks retire.
#include <cuda_runtime.h>

#include "ptoc_internal.h"
#include "reduce_impl.cuh"

namespace ptoc {

// ---------------------------------------------------------------------------
// allgather
// ---------------------------------------------------------------------------

template <int EB>
struct ElemRaw;
template <>
struct ElemRaw<2> {
    using T = uint16_t;
};
template <>
struct ElemRaw<4> {
    using T = uint32_t;
};

template <int EB, int VB>
__global__ void __launch_bounds__(kBlock) gather_kernel(const __grid_constant__ GatherParams p)
{
    using C = Chunk<VB>;
    constexpr int VE = VB / EB;
    const int n = p.nranks;
    pdl_enter();
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const int64_t row = t / p.tpr;
        const int64_t seg = t - row * p.tpr;
        const int owner = p.root >= 0 ? p.root : row_owner(row, n, p.rows);
        const int64_t row_byte = row * p.ld * EB;
        const int64_t v = seg * kBlock + threadIdx.x;
        if (v < p.vpr) {
            const int64_t off = row_byte + v * VB;
            const typename C::type x = C::load((const char*)p.win[owner] + off);
            for (int s = 0; s < n; ++s)
                if (s != owner) C::store((char*)p.win[s] + off, x);
        }
        if (p.tail > 0 && seg == p.tpr - 1) {
            using Raw = typename ElemRaw<EB>::T;
            for (int c = threadIdx.x; c < p.tail; c += kBlock) {
                const int64_t e = row * p.ld + p.vpr * VE + c;
                const Raw x = reinterpret_cast<const Raw*>(p.win[owner])[e];
                for (int s = 0; s < n; ++s)
                    if (s != owner) reinterpret_cast<Raw*>(p.win[s])[e] = x;
            }
        }
    }
}

template <int EB>
static cudaError_t launch_gather_eb(const GatherParams& p, int vb, dim3 grid, cudaStream_t s)
{
    if (vb == 16) return launch_kernel(gather_kernel<EB, 16>, grid, kBlock, 0, s, p);
    if (vb == 8) return launch_kernel(gather_kernel<EB, 8>, grid, kBlock, 0, s, p);
    if (vb == 4) return launch_kernel(gather_kernel<EB, 4>, grid, kBlock, 0, s, p);
    if constexpr (EB == 2) return launch_kernel(gather_kernel<2, 2>, grid, kBlock, 0, s, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gather(const GatherParams& p, int elem_bytes, int vb, dim3 grid, cudaStream_t s)
{
    return elem_bytes == 2 ? launch_gather_eb<2>(p, vb, grid, s) : launch_gather_eb<4>(p, vb, grid, s);
}

// ---------------------------------------------------------------------------
// all_to_all_v
// ---------------------------------------------------------------------------

__device__ __forceinline__ int32_t clamp_count(int32_t c, int64_t max_recv)
{
    int64_t v = c;
    v = v < 0 ? 0 : v;
    return (int32_t)(v > max_recv ? max_recv : v);
}

// Moves one chunk of VB bytes: a copy, or (AddMover) out += in per element.
template <int VB>
struct CopyMover {
    using C = Chunk<VB>;
    using V = typename C::type;
    static __device__ __forceinline__ V load(const char* src, const char*) { return C::load(src); }
    static __device__ __forceinline__ void store(char* dst, const V& v) { C::store(dst, v); }
};

template <class T, int VB>
struct AddMover {
    static constexpr int W = VB / 4;
    using V = Words<W>;
    // loads both operands and returns the sum, ready to store
    static __device__ __forceinline__ V load(const char* src, const char* dst)
    {
        VecAcc<T, kSum, W> acc;
        acc.init(load_words<W>(dst));
        acc.add(load_words<W>(src));
        return acc.out();
    }
    static __device__ __forceinline__ void store(char* dst, const V& v) { store_words<W>(dst, v); }
};

// 16-bit data that is only 2-byte aligned: one element at a time.
template <class T>
struct AddMover1 {
    using V = Elem16;
    static __device__ __forceinline__ V load(const char* src, const char* dst)
    {
        const float a = Scalar<T>::widen(Chunk<2>::load(dst).h);
        const float b = Scalar<T>::widen(Chunk<2>::load(src).h);
        V r;
        r.h = Scalar<T>::narrow(__fadd_rn(a, b));
        return r;
    }
    static __device__ __forceinline__ void store(char* dst, const V& v) { Chunk<2>::store(dst, v); }
};

// U chunks of VB bytes per thread per tile: tile_bytes = U * kBlock * VB.
// Block (x, q) moves bytes [x * tile_bytes, (x + 1) * tile_bytes) of pair
// q = a * N + b: from input a, rows b * MAX_RECV .., to output b, rows
// a * MAX_RECV .. (a grid-stride loop over x covers grids capped below the
// run's tile count).
template <class M, int VB, int U>
__global__ void __launch_bounds__(kBlock) pairs_kernel(const __grid_constant__ A2avParams p)
{
    const int n = p.nranks;
    const int q = blockIdx.y;
    const int a = q / n, b = q - a * n;
    pdl_enter();
    const int32_t c = p.full ? (int32_t)p.max_recv : clamp_count(p.cnt[a][b], p.max_recv);
    if (p.publish && blockIdx.x == 0 && threadIdx.x == 0) p.pub[b][a] = c;
    const int64_t bytes = (int64_t)c * p.row_bytes;
    const char* src0 = (const char*)p.in[a] + b * p.max_recv * p.row_bytes;
    char* dst0 = (char*)p.out[b] + a * p.max_recv * p.row_bytes;

    for (int64_t beg = (int64_t)blockIdx.x * p.tile_bytes; beg < bytes; beg += (int64_t)gridDim.x * p.tile_bytes) {
        const int64_t len = min(p.tile_bytes, bytes - beg);
        const char* src = src0 + beg;
        char* dst = dst0 + beg;
        typename M::V x[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t o = ((int64_t)k * kBlock + threadIdx.x) * VB;
            if (o < len) x[k] = M::load(src + o, dst + o);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t o = ((int64_t)k * kBlock + threadIdx.x) * VB;
            if (o < len) M::store(dst + o, x[k]);
        }
    }
}

template <int U>
static cudaError_t launch_a2av_u(const A2avParams& p, int vb, dim3 grid, cudaStream_t s)
{
    if (vb == 16) return launch_kernel(pairs_kernel<CopyMover<16>, 16, U>, grid, kBlock, 0, s, p);
    if (vb == 8) return launch_kernel(pairs_kernel<CopyMover<8>, 8, U>, grid, kBlock, 0, s, p);
    if (vb == 4) return launch_kernel(pairs_kernel<CopyMover<4>, 4, U>, grid, kBlock, 0, s, p);
    return launch_kernel(pairs_kernel<CopyMover<2>, 2, U>, grid, kBlock, 0, s, p);
}

cudaError_t launch_a2av(const A2avParams& p, int vb, int unroll, dim3 grid, cudaStream_t s)
{
    if (unroll == 16) return launch_a2av_u<16>(p, vb, grid, s);
    return unroll == 4 ? launch_a2av_u<4>(p, vb, grid, s) : launch_a2av_u<8>(p, vb, grid, s);
}

// The combine with kAdd: 4 chunks per thread per tile (each chunk loads both
// operands).
constexpr int kAddUnroll = 4;

template <class T>
static cudaError_t launch_add_t(const A2avParams& p, int vb, dim3 grid, cudaStream_t s)
{
    if (vb == 16) return launch_kernel(pairs_kernel<AddMover<T, 16>, 16, kAddUnroll>, grid, kBlock, 0, s, p);
    if (vb == 8) return launch_kernel(pairs_kernel<AddMover<T, 8>, 8, kAddUnroll>, grid, kBlock, 0, s, p);
    if (vb == 4) return launch_kernel(pairs_kernel<AddMover<T, 4>, 4, kAddUnroll>, grid, kBlock, 0, s, p);
    if constexpr (sizeof(T) == 2)
        return launch_kernel(pairs_kernel<AddMover1<T>, 2, kAddUnroll>, grid, kBlock, 0, s, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_pairs_add(const A2avParams& p, int dtype, int vb, dim3 grid, cudaStream_t s)
{
    switch (dtype) {
    case PTOC_F32: return launch_add_t<float>(p, vb, grid, s);
    case PTOC_I32: return launch_add_t<int32_t>(p, vb, grid, s);
    case PTOC_F16: return launch_add_t<__half>(p, vb, grid, s);
    default: return launch_add_t<__nv_bfloat16>(p, vb, grid, s);
    }
}

}  // namespace ptoc
