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
// on both sides, each pair is one contiguous copy of c * row_bytes bytes.
//
// When every count is MAX_RECV (the symmetric all_to_all) the host knows the
// tiles: grid.y is the pair, grid.x the tile of its run, one tile per block,
// and the hardware block scheduler hands them out in order as blocks retire.
// When the counts live on the device (all_to_all_v, the combine) a grid sized
// for the largest runs would launch a block per possible tile, and empty
// blocks cost about a nanosecond each: a sparse exchange would pay for its
// capacity. So one wave of blocks is launched instead. Each block rebuilds the
// pair counts and their tile prefix sums in shared memory, then claims the
// live tiles one at a time, in order, from a counter that starts at zero.
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

// Per-pair state in shared memory: cnt[q] = clamped count of pair q
// (q = a * N + b), pre[q] = tiles of pairs 0..q-1, pre[np] = all live tiles.
// Each thread sums a contiguous run of pairs; the runs are combined with a
// warp-shuffle scan and a pass over the warp totals. Block 0 also publishes
// the counts when asked (all_to_all_v's recv_counts).
__device__ void build_pairs(const A2avParams& p, int32_t* cnt, int32_t* pre, int32_t* warp_tot)
{
    const int n = p.nranks;
    const int np = n * n;
    const int per = (np + kBlock - 1) / kBlock;
    const int q0 = threadIdx.x * per;
    const int q1 = min(q0 + per, np);
    int32_t run = 0;
    for (int q = q0; q < q1; ++q) {
        const int a = q / n, b = q - (q / n) * n;
        const int32_t c = p.full ? (int32_t)p.max_recv : clamp_count(p.cnt[a][b], p.max_recv);
        if (p.publish && blockIdx.x == 0) p.pub[b][a] = c;
        cnt[q] = c;
        const int32_t tiles = (int32_t)(((int64_t)c * p.row_bytes + p.tile_bytes - 1) / p.tile_bytes);
        pre[q] = tiles;                 // this pair's tiles, until the scan below
        run += tiles;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int w = 0; w < kBlock / 32; ++w) {
            const int32_t t = warp_tot[w];
            warp_tot[w] = acc;
            acc += t;
        }
        pre[np] = acc;
    }
    __syncthreads();
    int32_t excl = warp_tot[warp] + incl - run;
    for (int q = q0; q < q1; ++q) {
        const int32_t tiles = pre[q];
        pre[q] = excl;
        excl += tiles;
    }
    __syncthreads();
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

// The same moves, claimed: tile t (counted over the live tiles of all pairs
// in pair order) is pair q's tile t - pre[q], where pre[q] <= t < pre[q + 1].
template <class M, int VB, int U>
__global__ void __launch_bounds__(kBlock) pairs_claim_kernel(const __grid_constant__ A2avParams p)
{
    extern __shared__ int32_t smem[];
    __shared__ int32_t warp_tot[kBlock / 32];
    __shared__ int32_t claimed;
    const int n = p.nranks;
    const int np = n * n;
    int32_t* cnt = smem;                    // np entries
    int32_t* pre = smem + np;               // np + 1 entries
    pdl_enter();
    build_pairs(p, cnt, pre, warp_tot);
    const int32_t total = pre[np];

    while (true) {
        if (threadIdx.x == 0) claimed = (int32_t)atomicAdd(p.claim, 1u);
        __syncthreads();
        const int32_t t = claimed;
        __syncthreads();                    // all have read it before the next claim
        if (t >= total) break;
        int lo = 0, hi = np;                // invariant: pre[lo] <= t < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= t) lo = mid;
            else hi = mid;
        }
        const int q = lo;
        const int a = q / n, b = q - (q / n) * n;
        const int64_t bytes = (int64_t)cnt[q] * p.row_bytes;
        const int64_t beg = (int64_t)(t - pre[q]) * p.tile_bytes;
        const int64_t len = min(p.tile_bytes, bytes - beg);
        const char* src = (const char*)p.in[a] + b * p.max_recv * p.row_bytes + beg;
        char* dst = (char*)p.out[b] + a * p.max_recv * p.row_bytes + beg;
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

size_t pairs_claim_smem_bytes(int nranks) { return (size_t)(2 * nranks * nranks + 1) * sizeof(int32_t); }

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

// ---- claiming launches --------------------------------------------------------

template <class M, int VB, int U>
static int claim_occupancy(size_t smem)
{
    int b = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, pairs_claim_kernel<M, VB, U>, kBlock, smem);
    return (e == cudaSuccess && b > 0) ? b : 1;
}

template <class M, int VB, int U>
static cudaError_t claim_launch(const A2avParams& p, int grid, size_t smem, cudaStream_t s)
{
    return launch_kernel(pairs_claim_kernel<M, VB, U>, dim3((unsigned)grid), kBlock, smem, s, p);
}

// The kernel family of one (add, dtype, vb, unroll): copies or kAdd adds.
template <class F>
static auto with_claim_kernel(bool add, int dtype, int vb, int unroll, F&& f)
{
    if (add) {
        switch (dtype) {
        case PTOC_F32:
            if (vb == 16) return f.template go<AddMover<float, 16>, 16, kAddUnroll>();
            if (vb == 8) return f.template go<AddMover<float, 8>, 8, kAddUnroll>();
            return f.template go<AddMover<float, 4>, 4, kAddUnroll>();
        case PTOC_I32:
            if (vb == 16) return f.template go<AddMover<int32_t, 16>, 16, kAddUnroll>();
            if (vb == 8) return f.template go<AddMover<int32_t, 8>, 8, kAddUnroll>();
            return f.template go<AddMover<int32_t, 4>, 4, kAddUnroll>();
        case PTOC_F16:
            if (vb == 16) return f.template go<AddMover<__half, 16>, 16, kAddUnroll>();
            if (vb == 8) return f.template go<AddMover<__half, 8>, 8, kAddUnroll>();
            if (vb == 4) return f.template go<AddMover<__half, 4>, 4, kAddUnroll>();
            return f.template go<AddMover1<__half>, 2, kAddUnroll>();
        default:
            if (vb == 16) return f.template go<AddMover<__nv_bfloat16, 16>, 16, kAddUnroll>();
            if (vb == 8) return f.template go<AddMover<__nv_bfloat16, 8>, 8, kAddUnroll>();
            if (vb == 4) return f.template go<AddMover<__nv_bfloat16, 4>, 4, kAddUnroll>();
            return f.template go<AddMover1<__nv_bfloat16>, 2, kAddUnroll>();
        }
    }
    if (unroll == 16) {
        if (vb == 16) return f.template go<CopyMover<16>, 16, 16>();
        if (vb == 8) return f.template go<CopyMover<8>, 8, 16>();
        if (vb == 4) return f.template go<CopyMover<4>, 4, 16>();
        return f.template go<CopyMover<2>, 2, 16>();
    }
    if (unroll == 4) {
        if (vb == 16) return f.template go<CopyMover<16>, 16, 4>();
        if (vb == 8) return f.template go<CopyMover<8>, 8, 4>();
        if (vb == 4) return f.template go<CopyMover<4>, 4, 4>();
        return f.template go<CopyMover<2>, 2, 4>();
    }
    if (vb == 16) return f.template go<CopyMover<16>, 16, 8>();
    if (vb == 8) return f.template go<CopyMover<8>, 8, 8>();
    if (vb == 4) return f.template go<CopyMover<4>, 4, 8>();
    return f.template go<CopyMover<2>, 2, 8>();
}

struct ClaimOccupancy {
    size_t smem;
    template <class M, int VB, int U>
    int go() const { return claim_occupancy<M, VB, U>(smem); }
};

struct ClaimLaunch {
    const A2avParams& p;
    int grid;
    size_t smem;
    cudaStream_t s;
    template <class M, int VB, int U>
    cudaError_t go() const { return claim_launch<M, VB, U>(p, grid, smem, s); }
};

int pairs_claim_blocks_per_sm(bool add, int dtype, int vb, int unroll, int nranks)
{
    return with_claim_kernel(add, dtype, vb, unroll, ClaimOccupancy{pairs_claim_smem_bytes(nranks)});
}

cudaError_t launch_pairs_claim(const A2avParams& p, bool add, int dtype, int vb, int unroll, int grid,
                               cudaStream_t s)
{
    return with_claim_kernel(add, dtype, vb, unroll, ClaimLaunch{p, grid, pairs_claim_smem_bytes(p.nranks), s});
}

}  // namespace ptoc
