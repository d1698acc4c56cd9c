// TREDUCE / reduce_scatter / allreduce kernel template.
//
// What it computes (TREDUCE article, "CANN PTO-ISA TREDUCE 指令详解", §1.1,
// §4.3): for every element of the valid box, acc = src[root]; then for every
// other rank in ascending order acc = acc (+) src[r]; store. The host passes
// the sources already in that order (src[0] is the root), so the kernel only
// walks src[0..n-1]. (+) is Sum, Max, Min, or Prod (the allreduce family's
// kProd, "Distributed Operators (N6)", ABI enums). The result goes to one
// dst (TREDUCE), to the window that owns the row (reduce_scatter) or to every
// window (allreduce).
//
// How (GB300 design, not the page's UB ping-pong): the op is HBM-bound
// (N reads + 1 write per element, at most one ALU op per loaded element), so
// the kernel is a streaming engine. Each block reduces one tile (a row
// segment of kBlock vectors of VB bytes, one per thread); each thread issues
// the loads of a group of up to kGroup ranks back to back (kGroup independent
// 16-byte loads in flight per thread) and only then folds them into its
// accumulator in rank order (9 to 12 ranks: 12 slots of 16 bytes; 13 to 16:
// 8-byte vectors, all 16 loads in flight; more ranks: one group after
// another). The grid has one block per tile, so as blocks retire the hardware
// block scheduler hands the next tiles, in order, to whichever SM has room.
// Accumulation is binary32 for every floating type (one RNE narrowing at the
// store); 16-bit Max / Min compare packed pairs and select the raw encodings,
// so their result is the selected input bit for bit.
//
// The shared-memory forms of the same reduction and the per-type dispatch
// between the forms are in reduce_forms.cuh; this file also serves the
// data-movement kernels (loads, stores, accumulators, launch helpers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <type_traits>

#include "ptoc_internal.h"

namespace ptoc {


template <int W>
struct Words {
    uint32_t w[W];
};

template <class To, class From>
__device__ __forceinline__ To bitcast(const From& f)
{
    static_assert(sizeof(To) == sizeof(From), "bitcast size");
    To t;
    memcpy(&t, &f, sizeof(To));
    return t;
}

// ---- vector loads and stores (L1 bypass: every byte is touched once) -------
// The loads are volatile and clobber memory, like the stores and the wait of
// a programmatic dependent launch: the compiler keeps every load after that
// wait, so no load can read a source before the previous kernel's writes.

template <int W>
__device__ __forceinline__ Words<W> load_words(const char* p);

template <>
__device__ __forceinline__ Words<4> load_words<4>(const char* p)
{
    Words<4> r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "l"(p) : "memory");
    return r;
}
template <>
__device__ __forceinline__ Words<2> load_words<2>(const char* p)
{
    Words<2> r;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p) : "memory");
    return r;
}
template <>
__device__ __forceinline__ Words<1> load_words<1>(const char* p)
{
    Words<1> r;
    asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p) : "memory");
    return r;
}

template <int W>
__device__ __forceinline__ void store_words(char* p, const Words<W>& v);

template <>
__device__ __forceinline__ void store_words<4>(char* p, const Words<4>& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]) : "memory");
}
template <>
__device__ __forceinline__ void store_words<2>(char* p, const Words<2>& v)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(v.w[0]), "r"(v.w[1]) : "memory");
}
template <>
__device__ __forceinline__ void store_words<1>(char* p, const Words<1>& v)
{
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(v.w[0]) : "memory");
}

// Copy units of VB bytes for the pure data-movement kernels (VB = 2: one
// 16-bit element).
struct Elem16 {
    uint16_t h;
};
template <int VB>
struct Chunk {
    using type = Words<VB / 4>;
    static __device__ __forceinline__ type load(const char* p) { return load_words<VB / 4>(p); }
    static __device__ __forceinline__ void store(char* p, const type& v) { store_words<VB / 4>(p, v); }
};
template <>
struct Chunk<2> {
    using type = Elem16;
    static __device__ __forceinline__ type load(const char* p)
    {
        Elem16 r;
        asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(r.h) : "l"(p) : "memory");
        return r;
    }
    static __device__ __forceinline__ void store(char* p, const type& v)
    {
        asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(v.h) : "memory");
    }
};

// ---- vector accumulators ----------------------------------------------------
// init(x): acc = x (the root's vector); add(x): acc = acc (+) x; out(): encode.

template <class T, int OP, int W>
struct VecAcc;

template <int OP, int W>
struct VecAcc<float, OP, W> {
    float a[W];
    __device__ __forceinline__ void init(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] = __uint_as_float(x.w[i]);
    }
    __device__ __forceinline__ void add(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const float v = __uint_as_float(x.w[i]);
            if constexpr (OP == kSum) a[i] = __fadd_rn(a[i], v);
            else if constexpr (OP == kProd) a[i] = __fmul_rn(a[i], v);
            else if constexpr (OP == kMax) a[i] = (v > a[i]) ? v : a[i];
            else a[i] = (v < a[i]) ? v : a[i];
        }
    }
    __device__ __forceinline__ Words<W> out() const
    {
        Words<W> r;
#pragma unroll
        for (int i = 0; i < W; ++i) r.w[i] = __float_as_uint(a[i]);
        return r;
    }
};

template <int OP, int W>
struct VecAcc<int32_t, OP, W> {
    uint32_t a[W];
    __device__ __forceinline__ void init(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] = x.w[i];
    }
    __device__ __forceinline__ void add(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            if constexpr (OP == kSum) a[i] = a[i] + x.w[i];   // wraps modulo 2^32
            else if constexpr (OP == kProd) a[i] = a[i] * x.w[i];   // wraps modulo 2^32
            else if constexpr (OP == kMax) a[i] = ((int32_t)x.w[i] > (int32_t)a[i]) ? x.w[i] : a[i];
            else a[i] = ((int32_t)x.w[i] < (int32_t)a[i]) ? x.w[i] : a[i];
        }
    }
    __device__ __forceinline__ Words<W> out() const
    {
        Words<W> r;
#pragma unroll
        for (int i = 0; i < W; ++i) r.w[i] = a[i];
        return r;
    }
};

// 16-bit Sum / Prod: each word holds two elements (low half = lower
// address); widened exactly to binary32, accumulated there, narrowed with RNE.
template <class T>
struct Pair16;
template <>
struct Pair16<__half> {
    using P = __half2;
    static __device__ __forceinline__ float2 widen(uint32_t w) { return __half22float2(bitcast<__half2>(w)); }
    // lo += widen(low half of w), hi += widen(high half): Blackwell's
    // mixed-precision add converts the 16-bit operand exactly to binary32 and
    // adds with round-to-nearest-even, which is widen() then __fadd_rn.
    static __device__ __forceinline__ void add_widened(float& lo, float& hi, uint32_t w)
    {
        asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.f16 %0, l, %0; add.rn.f32.f16 %1, h, %1; }"
            : "+f"(lo), "+f"(hi)
            : "r"(w));
    }
    static __device__ __forceinline__ uint32_t narrow(float lo, float hi)
    {
        return bitcast<uint32_t>(__floats2half2_rn(lo, hi));
    }
    static __device__ __forceinline__ uint32_t gt_mask(uint32_t x, uint32_t a)
    {
        return __hgt2_mask(bitcast<__half2>(x), bitcast<__half2>(a));
    }
    static __device__ __forceinline__ uint32_t lt_mask(uint32_t x, uint32_t a)
    {
        return __hlt2_mask(bitcast<__half2>(x), bitcast<__half2>(a));
    }
};
template <>
struct Pair16<__nv_bfloat16> {
    using P = __nv_bfloat162;
    static __device__ __forceinline__ float2 widen(uint32_t w) { return __bfloat1622float2(bitcast<__nv_bfloat162>(w)); }
    static __device__ __forceinline__ void add_widened(float& lo, float& hi, uint32_t w)
    {
        asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.bf16 %0, l, %0; add.rn.f32.bf16 %1, h, %1; }"
            : "+f"(lo), "+f"(hi)
            : "r"(w));
    }
    static __device__ __forceinline__ uint32_t narrow(float lo, float hi)
    {
        return bitcast<uint32_t>(__floats2bfloat162_rn(lo, hi));
    }
    static __device__ __forceinline__ uint32_t gt_mask(uint32_t x, uint32_t a)
    {
        return __hgt2_mask(bitcast<__nv_bfloat162>(x), bitcast<__nv_bfloat162>(a));
    }
    static __device__ __forceinline__ uint32_t lt_mask(uint32_t x, uint32_t a)
    {
        return __hlt2_mask(bitcast<__nv_bfloat162>(x), bitcast<__nv_bfloat162>(a));
    }
};

template <class T, int W, int OP = kSum>
struct Acc16Sum {
    float a[2 * W];
    __device__ __forceinline__ void init(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const float2 f = Pair16<T>::widen(x.w[i]);
            a[2 * i] = f.x;
            a[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ void add(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            if constexpr (OP == kProd) {
                const float2 f = Pair16<T>::widen(x.w[i]);
                a[2 * i] = __fmul_rn(a[2 * i], f.x);
                a[2 * i + 1] = __fmul_rn(a[2 * i + 1], f.y);
            } else {
                Pair16<T>::add_widened(a[2 * i], a[2 * i + 1], x.w[i]);
            }
        }
    }
    __device__ __forceinline__ Words<W> out() const
    {
        Words<W> r;
#pragma unroll
        for (int i = 0; i < W; ++i) r.w[i] = Pair16<T>::narrow(a[2 * i], a[2 * i + 1]);
        return r;
    }
};

// 16-bit Max / Min: an IEEE comparison per lane (false on NaN), then a
// bitwise select of the raw encodings: x replaces acc only where strictly
// greater (smaller).
template <class T, int OP, int W>
struct Acc16Sel {
    uint32_t a[W];
    __device__ __forceinline__ void init(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] = x.w[i];
    }
    __device__ __forceinline__ void add(const Words<W>& x)
    {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const uint32_t m = (OP == kMax) ? Pair16<T>::gt_mask(x.w[i], a[i])
                                            : Pair16<T>::lt_mask(x.w[i], a[i]);
            a[i] = (x.w[i] & m) | (a[i] & ~m);
        }
    }
    __device__ __forceinline__ Words<W> out() const
    {
        Words<W> r;
#pragma unroll
        for (int i = 0; i < W; ++i) r.w[i] = a[i];
        return r;
    }
};

template <int W> struct VecAcc<__half, kSum, W> : Acc16Sum<__half, W> {};
template <int W> struct VecAcc<__half, kProd, W> : Acc16Sum<__half, W, kProd> {};
template <int W> struct VecAcc<__half, kMax, W> : Acc16Sel<__half, kMax, W> {};
template <int W> struct VecAcc<__half, kMin, W> : Acc16Sel<__half, kMin, W> {};
template <int W> struct VecAcc<__nv_bfloat16, kSum, W> : Acc16Sum<__nv_bfloat16, W> {};
template <int W> struct VecAcc<__nv_bfloat16, kProd, W> : Acc16Sum<__nv_bfloat16, W, kProd> {};
template <int W> struct VecAcc<__nv_bfloat16, kMax, W> : Acc16Sel<__nv_bfloat16, kMax, W> {};
template <int W> struct VecAcc<__nv_bfloat16, kMin, W> : Acc16Sel<__nv_bfloat16, kMin, W> {};

// ---- one element at a time (row tails, 2-byte-aligned buffers) ------------

template <class T>
struct Scalar;
template <>
struct Scalar<float> {
    using Raw = uint32_t;
};
template <>
struct Scalar<int32_t> {
    using Raw = uint32_t;
};
template <>
struct Scalar<__half> {
    using Raw = uint16_t;
    static __device__ __forceinline__ float widen(uint16_t h) { return __half2float(bitcast<__half>(h)); }
    static __device__ __forceinline__ uint16_t narrow(float f) { return bitcast<uint16_t>(__float2half_rn(f)); }
};
template <>
struct Scalar<__nv_bfloat16> {
    using Raw = uint16_t;
    static __device__ __forceinline__ float widen(uint16_t h) { return __bfloat162float(bitcast<__nv_bfloat16>(h)); }
    static __device__ __forceinline__ uint16_t narrow(float f) { return bitcast<uint16_t>(__float2bfloat16_rn(f)); }
};

// Element `e` (offset in elements) of the reduction over src[0..n-1].
template <class T, int OP>
__device__ __forceinline__ typename Scalar<T>::Raw reduce_one(const ReduceParams& p, int64_t e)
{
    using Raw = typename Scalar<T>::Raw;
    const int n = p.nranks;
    Raw acc = reinterpret_cast<const Raw*>(p.src[0])[e];
    if constexpr (std::is_same<T, float>::value) {
        float a = __uint_as_float(acc);
        for (int r = 1; r < n; ++r) {
            const float v = __uint_as_float(reinterpret_cast<const Raw*>(p.src[r])[e]);
            if constexpr (OP == kSum) a = __fadd_rn(a, v);
            else if constexpr (OP == kProd) a = __fmul_rn(a, v);
            else if constexpr (OP == kMax) a = (v > a) ? v : a;
            else a = (v < a) ? v : a;
        }
        return __float_as_uint(a);
    } else if constexpr (std::is_same<T, int32_t>::value) {
        for (int r = 1; r < n; ++r) {
            const uint32_t v = reinterpret_cast<const Raw*>(p.src[r])[e];
            if constexpr (OP == kSum) acc = acc + v;
            else if constexpr (OP == kProd) acc = acc * v;
            else if constexpr (OP == kMax) acc = ((int32_t)v > (int32_t)acc) ? v : acc;
            else acc = ((int32_t)v < (int32_t)acc) ? v : acc;
        }
        return acc;
    } else {
        float a = Scalar<T>::widen(acc);
        for (int r = 1; r < n; ++r) {
            const Raw raw = reinterpret_cast<const Raw*>(p.src[r])[e];
            const float v = Scalar<T>::widen(raw);
            if constexpr (OP == kSum) {
                a = __fadd_rn(a, v);
            } else if constexpr (OP == kProd) {
                a = __fmul_rn(a, v);
            } else if ((OP == kMax && v > a) || (OP == kMin && v < a)) {
                a = v;
                acc = raw;
            }
        }
        if constexpr (OP == kSum || OP == kProd) return Scalar<T>::narrow(a);
        return acc;
    }
}

// Rank that owns row `row` under the balanced bounds floor(r * rows / n):
// the largest r with floor(r * rows / n) <= row, i.e. ((row + 1) n - 1) / rows.
__device__ __forceinline__ int row_owner(int64_t row, int n, int64_t rows)
{
    return (int)(((row + 1) * (int64_t)n - 1) / rows);
}

// The one destination of a row (kDstOne, kDstOwner); kDstAll rows go to every
// window and use store_all / put_all instead.
__device__ __forceinline__ char* row_dst(const ReduceParams& p, int64_t row)
{
    return (char*)(p.dst_mode == kDstOwner ? p.dst[row_owner(row, p.nranks, p.rows)] : p.dst[0]);
}

// Store one result vector at byte offset `off` of its destination(s).
template <int W>
__device__ __forceinline__ void store_result(const ReduceParams& p, int64_t row, int64_t off, const Words<W>& v)
{
    if (p.dst_mode == kDstAll) {
        for (int r = 0; r < p.nranks; ++r) store_words<W>((char*)p.dst[r] + off, v);
    } else {
        store_words<W>(row_dst(p, row) + off, v);
    }
}

// Store one result element at element offset `e` of its destination(s).
template <class Raw>
__device__ __forceinline__ void store_elem(const ReduceParams& p, int64_t row, int64_t e, Raw v)
{
    if (p.dst_mode == kDstAll) {
        for (int r = 0; r < p.nranks; ++r) reinterpret_cast<Raw*>(p.dst[r])[e] = v;
    } else {
        reinterpret_cast<Raw*>(row_dst(p, row))[e] = v;
    }
}

// ---- programmatic dependent launch -----------------------------------------

// Called first by every data kernel: wait until the previous grid in the
// stream has completed and its writes are visible (a no-op for an ordinary
// launch), then allow the next programmatic launch to start scheduling.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// Launch `kernel` on `s`, as a programmatic dependent launch when enabled:
// the launch may overlap the tail of the previous kernel of the stream, which
// pdl_enter then waits for.
template <class K, class P>
cudaError_t launch_kernel(K kernel, dim3 grid, unsigned block, size_t smem, cudaStream_t s, const P& p)
{
    if (!programmatic_launch()) {
        kernel<<<grid, block, smem, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// ---- the kernel --------------------------------------------------------------

// How a thread covers the ranks (chosen on the host from the rank count):
//   kOneGroup  up to kGroup ranks: all loads issued back to back, then folded.
//   kWide12    9 to 12 ranks on 16-byte vectors: the same with 12 slots
//              (80 registers: three blocks per SM, up to 192 bytes of loads in
//              flight per thread).
//   kWide      up to 2 * kGroup ranks on vectors of at most 8 bytes: all
//              2 * kGroup loads in flight (the host narrows 16-byte vectors to
//              8 for 13 to 16 ranks, so the registers stay those of one group).
//   kGroups    more ranks: groups of kGroup, each issued and then folded.
enum RankForm : int { kOneGroup = 0, kWide = 1, kGroups = 2, kWide12 = 3 };

template <int FORM>
constexpr int kSlots = FORM == kWide ? 2 * kGroup : FORM == kWide12 ? 12 : kGroup;

// One tile: kBlock vectors of VB bytes of one row segment, one per thread,
// folded in rank order 0, 1, 2, ... whatever the form.
template <class T, int OP, int VB, int FORM>
__device__ __forceinline__ void reduce_vector_tile(const ReduceParams& p, int64_t t)
{
    constexpr int W = VB / 4;
    constexpr int S = kSlots<FORM>;
    const int n = p.nranks;
    const int64_t row = t / p.tpr;
    const int64_t seg = t - row * p.tpr;
    const int64_t v = seg * kBlock + threadIdx.x;
    if (v >= p.vpr) return;
    const int64_t off = row * p.ld * (int64_t)sizeof(T) + v * VB;

    VecAcc<T, OP, W> acc;
    {
        Words<W> x[S];
#pragma unroll
        for (int j = 0; j < S; ++j)
            if (j < n) x[j] = load_words<W>((const char*)p.src[j] + off);
        acc.init(x[0]);
#pragma unroll
        for (int j = 1; j < S; ++j)
            if (j < n) acc.add(x[j]);
    }
    if constexpr (FORM == kGroups) {
        for (int g0 = S; g0 < n; g0 += S) {
            Words<W> x[S];
#pragma unroll
            for (int j = 0; j < S; ++j)
                if (g0 + j < n) x[j] = load_words<W>((const char*)p.src[g0 + j] + off);
#pragma unroll
            for (int j = 0; j < S; ++j)
                if (g0 + j < n) acc.add(x[j]);
        }
    }
    store_result<W>(p, row, off, acc.out());
}

// One element per thread: 16-bit data that is only 2-byte aligned (vpr is
// then the row's element count and there is no tail).
template <class T, int OP>
__device__ __forceinline__ void reduce_element_tile(const ReduceParams& p, int64_t t)
{
    using Raw = typename Scalar<T>::Raw;
    const int64_t row = t / p.tpr;
    const int64_t seg = t - row * p.tpr;
    const int64_t v = seg * kBlock + threadIdx.x;
    if (v < p.vpr) {
        const int64_t e = row * p.ld + v;
        store_elem<Raw>(p, row, e, reduce_one<T, OP>(p, e));
    }
}

// Tail block b: the elements after the last full vector of each row (fewer
// than one vector per row), rows * tail of them, one per thread.
template <class T, int OP, int VB>
__device__ __forceinline__ void reduce_tail_block(const ReduceParams& p, int64_t b)
{
    using Raw = typename Scalar<T>::Raw;
    constexpr int VE = VB / (int)sizeof(T);
    const int64_t i = b * kBlock + threadIdx.x;
    if (i >= p.rows * p.tail) return;
    const int64_t row = i / p.tail;
    const int64_t c = i - row * p.tail;
    const int64_t e = row * p.ld + p.vpr * VE + c;
    store_elem<Raw>(p, row, e, reduce_one<T, OP>(p, e));
}

// Work item w < ntiles is vector tile w, the rest are tail blocks. The grid
// normally has one block per work item, so the hardware block scheduler hands
// out the tiles in order as blocks retire; a grid-stride loop covers grids
// capped below the item count.
// Before it waits for the previous kernel of the stream, a block of the first
// wave asks L2 for its first tile (one bulk prefetch per rank, on 16-byte
// vectors): a programmatic dependent launch starts these blocks while the
// previous kernel's last blocks still run, and the prefetch lets DRAM fetch
// the tile meanwhile. A prefetch returns no data, and L2 is where every write
// to device memory lands, so the loads after the wait still see the previous
// kernel's writes.
template <class T, int VB>
__device__ __forceinline__ void prefetch_first_tile(const ReduceParams& p)
{
    if constexpr (VB == 16) {
        if (blockIdx.x < (unsigned)p.prefetch_blocks && blockIdx.x < p.ntiles && (int)threadIdx.x < p.nranks) {
            const int64_t row = blockIdx.x / p.tpr;
            const int64_t v0 = (blockIdx.x - row * p.tpr) * kBlock;
            const int64_t nv = p.vpr - v0 < kBlock ? p.vpr - v0 : kBlock;
            if (nv > 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                             ::"l"((const char*)p.src[threadIdx.x] + row * p.ld * (int64_t)sizeof(T) + v0 * 16),
                               "r"((uint32_t)(nv * 16))
                             : "memory");
        }
    }
}

template <class T, int OP, int VB, int FORM>
__global__ void __launch_bounds__(kBlock) reduce_kernel(const __grid_constant__ ReduceParams p)
{
    prefetch_first_tile<T, VB>(p);
    pdl_enter();
    const int64_t total = p.ntiles + p.tail_blocks;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        if (w < p.ntiles) {
            if constexpr (VB < 4) reduce_element_tile<T, OP>(p, w);
            else reduce_vector_tile<T, OP, VB, FORM>(p, w);
        } else {
            if constexpr (VB >= 4) reduce_tail_block<T, OP, VB>(p, w - p.ntiles);
        }
    }
}

}  // namespace ptoc
