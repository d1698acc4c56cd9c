// Window-layout data movement: allgather and all_to_all_v.
//
// allgather ("Distributed Operators (N6)", op table): row chunk r of window r
// is copied into row chunk r of every other window. One read, N-1 writes per
// element: each thread loads its vectors once and stores them N-1 times.
//
// all_to_all_v ("Distributed Operators (N6)", pld.tensor.all_to_all_v): for
// every (sender s, destination d) the clamped count c = clamp(send_counts[s][d],
// 0, MAX_RECV) is published to recv_counts[d][s], and c packed rows move from
// input s (rows d*MAX_RECV ..) to target d (rows s*MAX_RECV ..). Because the
// rows of one pair are contiguous on both sides, each pair is one contiguous
// copy of c * row_bytes bytes. The counts live on the device, so the grid
// cannot be sized from them: a persistent grid walks a list of fixed-size
// tiles, and every CTA rebuilds the per-pair tile prefix sums in shared memory
// from the N^2 counts (a few hundred integers, L2-resident) before it starts.
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
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const int64_t row = t / p.tpr;
        const int64_t seg = t - row * p.tpr;
        const int owner = row_owner(row, n, p.rows);
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
    if (vb == 16) gather_kernel<EB, 16><<<grid, kBlock, 0, s>>>(p);
    else if (vb == 8) gather_kernel<EB, 8><<<grid, kBlock, 0, s>>>(p);
    else if (vb == 4) gather_kernel<EB, 4><<<grid, kBlock, 0, s>>>(p);
    else if constexpr (EB == 2) gather_kernel<2, 2><<<grid, kBlock, 0, s>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
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
// (q = s * N + d), pre[q] = tiles of pairs 0..q-1 (exclusive prefix), pre[np]
// = total. Each thread scans a contiguous run of pairs; the run totals are
// combined with a warp-shuffle scan and a pass over the warp totals. Block 0
// also publishes the counts to recv_counts.
__device__ void build_pairs(const A2avParams& p, int32_t* cnt, int32_t* pre, int32_t* warp_tot)
{
    const int n = p.nranks;
    const int np = n * n;
    const int per = (np + kBlock - 1) / kBlock;
    const int q0 = threadIdx.x * per;
    const int q1 = min(q0 + per, np);

    int32_t run = 0;
    for (int q = q0; q < q1; ++q) {
        const int s = q / n, d = q - (q / n) * n;
        const int32_t c = clamp_count(p.sc[s][d], p.max_recv);
        if (blockIdx.x == 0) p.rc[d][s] = c;
        cnt[q] = c;
        const int32_t tiles = (int32_t)(((int64_t)c * p.row_bytes + p.tile_bytes - 1) / p.tile_bytes);
        pre[q] = tiles;                 // temporarily: this pair's tile count
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
    int32_t excl = warp_tot[warp] + incl - run;   // tiles before this thread's run
    for (int q = q0; q < q1; ++q) {
        const int32_t tiles = pre[q];
        pre[q] = excl;
        excl += tiles;
    }
    __syncthreads();
}

// U chunks of VB bytes per thread per tile: tile_bytes = U * kBlock * VB.
template <int VB, int U>
__global__ void __launch_bounds__(kBlock) a2av_kernel(const __grid_constant__ A2avParams p)
{
    extern __shared__ int32_t smem[];
    __shared__ int32_t warp_tot[kBlock / 32];
    using C = Chunk<VB>;
    const int n = p.nranks;
    const int np = n * n;
    int32_t* cnt = smem;                    // np entries
    int32_t* pre = smem + np;               // np + 1 entries
    build_pairs(p, cnt, pre, warp_tot);
    const int32_t total = pre[np];

    for (int32_t t = blockIdx.x; t < total; t += gridDim.x) {
        // the pair q with pre[q] <= t < pre[q + 1]
        int lo = 0, hi = np;                // invariant: pre[lo] <= t < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= t) lo = mid;
            else hi = mid;
        }
        const int q = lo;
        const int s = q / n, d = q - (q / n) * n;
        const int64_t bytes = (int64_t)cnt[q] * p.row_bytes;
        const int64_t beg = (int64_t)(t - pre[q]) * p.tile_bytes;
        const int64_t len = min(p.tile_bytes, bytes - beg);
        const char* src = (const char*)p.in[s] + d * p.max_recv * p.row_bytes + beg;
        char* dst = (char*)p.tgt[d] + s * p.max_recv * p.row_bytes + beg;

        typename C::type x[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t o = ((int64_t)k * kBlock + threadIdx.x) * VB;
            if (o < len) x[k] = C::load(src + o);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t o = ((int64_t)k * kBlock + threadIdx.x) * VB;
            if (o < len) C::store(dst + o, x[k]);
        }
    }
}

size_t a2av_smem_bytes(int nranks) { return (size_t)(2 * nranks * nranks + 1) * sizeof(int32_t); }

template <int U>
static cudaError_t launch_a2av_u(const A2avParams& p, int vb, dim3 grid, cudaStream_t s)
{
    const size_t smem = a2av_smem_bytes(p.nranks);
    if (vb == 16) a2av_kernel<16, U><<<grid, kBlock, smem, s>>>(p);
    else if (vb == 8) a2av_kernel<8, U><<<grid, kBlock, smem, s>>>(p);
    else if (vb == 4) a2av_kernel<4, U><<<grid, kBlock, smem, s>>>(p);
    else a2av_kernel<2, U><<<grid, kBlock, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_a2av(const A2avParams& p, int vb, int unroll, dim3 grid, cudaStream_t s)
{
    return unroll == 8 ? launch_a2av_u<8>(p, vb, grid, s) : launch_a2av_u<4>(p, vb, grid, s);
}

template <int U>
static int a2av_occupancy_u(int vb, size_t smem)
{
    int b = 0;
    cudaError_t e = vb == 16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, a2av_kernel<16, U>, kBlock, smem)
                  : vb == 8 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, a2av_kernel<8, U>, kBlock, smem)
                  : vb == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, a2av_kernel<4, U>, kBlock, smem)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, a2av_kernel<2, U>, kBlock, smem);
    return (e == cudaSuccess && b > 0) ? b : 1;
}

int a2av_blocks_per_sm(int vb, int unroll, int nranks)
{
    const size_t smem = a2av_smem_bytes(nranks);
    return unroll == 8 ? a2av_occupancy_u<8>(vb, smem) : a2av_occupancy_u<4>(vb, smem);
}

}  // namespace ptoc
