// The shared-memory forms of the TREDUCE / reduce_scatter / allreduce
// reduction, and the per-element-type dispatch between the forms (included
// only by the reduction translation units, reduce_{f32,i32,f16,bf16}.cu).
//
// The staged form takes the register form's tiles (one row segment of kBlock
// 16-byte vectors per block) and stages them through shared memory with the
// bulk-copy (TMA) engine: per tile, one `cp.async.bulk` per rank lands the
// rank's 4 KiB segment and completes on that rank's mbarrier, so the fold of
// rank r runs while the copies of ranks r+1.. are still in flight (the GPU
// form of the page's ping-pong between two UB tiles, TREDUCE article §4.4).
// Grid, tile order, arithmetic and stores are those of the register form;
// only the path of the loads differs. The tensor form (TREDUCE only) loads
// 2-D boxes of the valid box through tensor maps and stores the result box
// back through one, clipped to the valid box.
#pragma once

#include "reduce_impl.cuh"

namespace ptoc {

// ---- the staged form ----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Arm the mbarrier at `bar` for `bytes` and start one bulk copy of `bytes`
// from global `src` into shared `dst` that completes on it.
__device__ __forceinline__ void stage_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ Words<4> stage_load(uint32_t addr)
{
    Words<4> r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "r"(addr)
                 : "memory");
    return r;
}

__device__ __forceinline__ bool stage_ready(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Every wait on a copy is bounded: a deadline on %globaltimer behind an
// iteration cap. A copy of valid memory always completes long before either.
// The fold's waits take the launch's bound (wait_ns, 2 s unless the caller's
// process sets PTOC_WAIT_NS); the one wait of a block that gave up, for its
// own copies still in flight, always takes kStageWaitNs, so that no block
// leaves while a copy into its shared memory may still land.
// Tiles whose wait gave up are counted here (one counter per translation
// unit, zero at load; ptoc_wait_faults reads and clears them).
static __device__ uint32_t g_stage_faults;
constexpr uint64_t kStageWaitNs = 2000000000ull;
constexpr uint32_t kStageWaitPolls = 1u << 26;

// try_wait with a bound on how long the thread may stay suspended in it
__device__ __forceinline__ bool stage_ready_within(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Bounds below this are passed to try_wait as its suspend-time limit, and the
// deadline is then checked after every poll: try_wait may otherwise stay
// suspended until the copy lands, well past a short bound.
constexpr uint64_t kHintedWaitNs = 1000000ull;

__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, uint64_t deadline, uint64_t bound_ns)
{
    const uint32_t hint = bound_ns < kHintedWaitNs ? (uint32_t)bound_ns : 0u;
    for (uint32_t i = 0; i < kStageWaitPolls; ++i) {
        if (hint ? stage_ready_within(bar, parity, hint) : stage_ready(bar, parity)) return true;
        if ((hint || (i & 31) == 31) && globaltimer_ns() > deadline) return false;
    }
    return false;
}

// The fold of one staged tile for the calling thread: its 16 bytes of rank
// r's segment sit at `mine` + r * kBlock * 16 in shared memory, and rank r's
// copy completes on bars[r]. Waits for the ranks in order (each bounded by
// the launch's bound), folding each as it lands; false if a wait gave up.
template <class T, int OP>
__device__ __forceinline__ bool fold_staged(const uint64_t* bars, int n, uint32_t parity, uint32_t mine,
                                            uint64_t bound_ns, Words<4>& out)
{
    const uint64_t deadline = globaltimer_ns() + bound_ns;
    VecAcc<T, OP, 4> acc;
    if (!stage_wait(smem_u32(&bars[0]), parity, deadline, bound_ns)) return false;
    acc.init(stage_load(mine));
    for (int r = 1; r < n; ++r) {
        if (!stage_wait(smem_u32(&bars[r]), parity, deadline, bound_ns)) return false;
        acc.add(stage_load(mine + (uint32_t)(r * kBlock * 16)));
    }
    out = acc.out();
    return true;
}

// A block one of whose waits gave up: count the fault, wait (with the full
// bound) for each rank's copy still in flight, so that no copy lands in shared
// memory the block no longer owns, and meet the block before it returns.
__device__ __forceinline__ void give_up_tile(const uint64_t* bars, int n, uint32_t parity)
{
    if (threadIdx.x == 0) atomicAdd(&g_stage_faults, 1u);
    if ((int)threadIdx.x < n)
        stage_wait(smem_u32(&bars[threadIdx.x]), parity, globaltimer_ns() + kStageWaitNs, kStageWaitNs);
    __syncthreads();
}

// Tiles as in reduce_kernel (one row segment of kBlock 16-byte vectors), the
// sources staged in dynamic shared memory: rank r's segment at r * kBlock
// vectors. Thread r < n owns rank r's mbarrier and starts that rank's copy
// (the block's first tile before the block-wide barrier, so the copies are on
// their way while the other warps arrive); every thread with a vector then
// waits for rank 0's copy, initialises its accumulator, and folds ranks
// 1..n-1 as their copies land, in rank order; the stores are those of the
// register form. A wait that gives up (with the default bound it never does
// on valid memory) adds 1 to g_stage_faults, and the block waits once more,
// with the full bound, for its copies in flight and returns without storing
// that tile or any later one.
template <class T, int OP>
__global__ void __launch_bounds__(kBlock) reduce_staged_kernel(const __grid_constant__ ReduceParams p)
{
    extern __shared__ __align__(128) Words<4> stage[];
    __shared__ __align__(8) uint64_t bars[kGroup];
    const int n = p.nranks;
    const int tid = threadIdx.x;
    const int64_t total = p.ntiles + p.tail_blocks;
    // Vectors of tile w (0 for a row shorter than one vector, whose tail
    // block covers it); its row and the byte offset of its first vector.
    auto tile = [&](int64_t w, int64_t& row, int64_t& off0) -> int {
        row = w / p.tpr;
        const int64_t v0 = (w - row * p.tpr) * kBlock;
        off0 = row * p.ld * (int64_t)sizeof(T) + v0 * 16;
        return (int)(p.vpr - v0 < kBlock ? p.vpr - v0 : kBlock);
    };
    auto issue = [&](int64_t off0, int nv) {
        stage_copy(smem_u32(stage + tid * kBlock), (const char*)p.src[tid] + off0, (uint32_t)nv * 16u,
                   smem_u32(&bars[tid]));
    };
    if (tid < n) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[tid])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_enter();
    bool issued = false;          // the copies of the next tile are already on their way
    if (blockIdx.x < p.ntiles) {
        int64_t row, off0;
        const int nv = tile(blockIdx.x, row, off0);
        if (nv > 0) {
            if (tid < n) issue(off0, nv);
            issued = true;
        }
    }
    __syncthreads();              // every mbarrier is initialised before anyone waits on it
    uint32_t parity = 0;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        if (w >= p.ntiles) {
            reduce_tail_block<T, OP, 16>(p, w - p.ntiles);
            continue;
        }
        int64_t row, off0;
        const int nv = tile(w, row, off0);
        if (nv <= 0) continue;
        if (!issued && tid < n) {
            // the stage was last read through the generic proxy (previous tile)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(off0, nv);
        }
        issued = false;
        bool ok = true;
        if (tid < nv) {
            Words<4> v;
            ok = fold_staged<T, OP>(bars, n, parity, smem_u32(stage + tid), p.wait_ns, v);
            if (ok) store_result<4>(p, row, off0 + (int64_t)tid * 16, v);
        }
        // every thread is done with the stage before it is refilled
        if (!__syncthreads_and(ok)) {
            give_up_tile(bars, n, parity);
            return;
        }
        parity ^= 1u;
    }
}

// ---- the tensor form (TREDUCE) -----------------------------------------------

// One box of 256 threads x 16 bytes = 4 KiB per rank: kTmaBoxCols elements
// wide, this many rows high (4 for 4-byte elements, 8 for 2-byte ones).
template <class T>
constexpr int kTmaBoxRows = kBlock * 16 / (kTmaBoxCols * (int)sizeof(T));

// Arm the mbarrier at `bar` for one 4 KiB box and load the box at (x, y) of
// the tensor map `map` (a kernel-parameter address) into shared `dst`.
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kBlock * 16) : "memory");
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// Store the 4 KiB box in shared `src` at (x, y) of `map`, clipped to the
// map's extent; returns once shared memory has been read.
__device__ __forceinline__ void tma_store_box(const CUtensorMap* map, int x, int y, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// TREDUCE over 2 to kGroup ranks through tensor maps. Tile w is one box of
// the valid box: threads 0..n-1 each load their rank's box into shared
// memory (rank r at r * kBlock vectors), completing on that rank's mbarrier;
// every thread folds its 16 bytes of the box over the ranks in order as the
// boxes land (parts of a box outside the valid box were filled with zeros
// and fold to values that are never stored), writes the result over rank 0's
// box, and thread 0 stores the box, which the map clips to the valid box.
// Waits are bounded as in the staged form; a block that gives up counts a
// fault and returns without storing.
template <class T, int OP>
__global__ void __launch_bounds__(kBlock) reduce_tma2d_kernel(const __grid_constant__ TmaReduceParams p)
{
    extern __shared__ __align__(128) Words<4> stage[];
    __shared__ __align__(8) uint64_t bars[kGroup];
    constexpr int kRows = kTmaBoxRows<T>;
    const int n = p.nranks;
    const int tid = threadIdx.x;
    // the boxes need 128-byte-aligned shared memory: refuse rather than copy
    if (smem_u32(stage) & 127u) {
        if (tid == 0) atomicAdd(&g_stage_faults, 1u);
        return;
    }
    auto issue = [&](int64_t w) {
        const int x = (int)(w % p.tiles_x) * kTmaBoxCols;
        const int y = (int)(w / p.tiles_x) * kRows;
        tma_load_box(smem_u32(stage + tid * kBlock), &p.src[tid], x, y, smem_u32(&bars[tid]));
    };
    if (tid < n) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[tid])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_enter();
    if (blockIdx.x < p.ntiles && tid < n) issue(blockIdx.x);
    __syncthreads();              // every mbarrier is initialised before anyone waits on it
    uint32_t parity = 0;
    bool first = true;
    for (int64_t w = blockIdx.x; w < p.ntiles; w += gridDim.x) {
        if (!first && tid < n) {
            // the stage was last read through the generic proxy (previous tile)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(w);
        }
        first = false;
        const uint32_t mine = smem_u32(stage + tid);
        Words<4> v;
        const bool ok = fold_staged<T, OP>(bars, n, parity, mine, p.wait_ns, v);
        if (ok)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                         ::"r"(mine), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                         : "memory");
        // the result box is complete (and visible to the async proxy) before
        // thread 0 stores it; a failed wait anywhere skips the store
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!__syncthreads_and(ok)) {
            give_up_tile(bars, n, parity);
            return;
        }
        if (tid == 0)
            tma_store_box(&p.dst, (int)(w % p.tiles_x) * kTmaBoxCols, (int)(w / p.tiles_x) * kRows,
                          smem_u32(stage));
        __syncthreads();          // the store has read the stage before it is refilled
        parity ^= 1u;
    }
}

template <class T>
cudaError_t launch_tma_reduce_t(const TmaReduceParams& p, int op, cudaStream_t s)
{
    if (p.nranks < 2 || p.nranks > kGroup || p.ntiles < 1) return cudaErrorInvalidValue;
    const int64_t cap = (int64_t)1 << 30;
    const dim3 grid((unsigned)(p.ntiles < cap ? p.ntiles : cap));
    const size_t smem = (size_t)p.nranks * kBlock * 16;
    switch (op) {
    case kSum: return launch_kernel(reduce_tma2d_kernel<T, kSum>, grid, kBlock, smem, s, p);
    case kMax: return launch_kernel(reduce_tma2d_kernel<T, kMax>, grid, kBlock, smem, s, p);
    case kMin: return launch_kernel(reduce_tma2d_kernel<T, kMin>, grid, kBlock, smem, s, p);
    default: return cudaErrorInvalidValue;
    }
}

// The rank form follows the rank count; kWide runs on vectors of at most 8
// bytes (the host narrows 16-byte vectors for 9 to 16 ranks).
template <class T, int OP, int VB>
cudaError_t launch_reduce_vb(const ReduceParams& p, dim3 grid, cudaStream_t s)
{
    if constexpr (VB == 16) {
        // up to one group of ranks: the staged form when selected
        if (p.nranks >= 2 && p.nranks <= kGroup && p.staged)
            return launch_kernel(reduce_staged_kernel<T, OP>, grid, kBlock,
                                 (size_t)p.nranks * kBlock * 16, s, p);
    }
    if constexpr (VB >= 4) {
        if (p.nranks > 2 * kGroup) return launch_kernel(reduce_kernel<T, OP, VB, kGroups>, grid, kBlock, 0, s, p);
        if (p.nranks > kGroup) {
            if constexpr (VB == 16) {
                if (p.nranks <= 12) return launch_kernel(reduce_kernel<T, OP, VB, kWide12>, grid, kBlock, 0, s, p);
                return cudaErrorInvalidValue;
            } else {
                return launch_kernel(reduce_kernel<T, OP, VB, kWide>, grid, kBlock, 0, s, p);
            }
        }
    }
    return launch_kernel(reduce_kernel<T, OP, VB, kOneGroup>, grid, kBlock, 0, s, p);
}

template <class T, int OP>
cudaError_t launch_reduce_op(const ReduceParams& p, int vb, dim3 grid, cudaStream_t s)
{
    switch (vb) {
    case 16: return launch_reduce_vb<T, OP, 16>(p, grid, s);
    case 8: return launch_reduce_vb<T, OP, 8>(p, grid, s);
    case 4: return launch_reduce_vb<T, OP, 4>(p, grid, s);
    default:
        if constexpr (sizeof(T) == 2) return launch_reduce_vb<T, OP, 2>(p, grid, s);
        return cudaErrorInvalidValue;
    }
}

// This translation unit's staged-wait fault count: read, then reset.
static inline cudaError_t take_stage_faults(uint32_t* count)
{
    const uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(count, g_stage_faults, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_stage_faults, &zero, sizeof(zero));
    return e;
}

template <class T>
cudaError_t launch_reduce_t(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s)
{
    switch (op) {
    case kSum: return launch_reduce_op<T, kSum>(p, vb, grid, s);
    case kMax: return launch_reduce_op<T, kMax>(p, vb, grid, s);
    case kProd: return launch_reduce_op<T, kProd>(p, vb, grid, s);
    default: return launch_reduce_op<T, kMin>(p, vb, grid, s);
    }
}

}  // namespace ptoc
