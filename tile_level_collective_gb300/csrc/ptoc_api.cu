// C-ABI entry points of libptoc.so: argument validation, operand ordering,
// vector-width and grid selection, and the launch. Every check runs on the
// host before any CUDA call, so a rejected call launches nothing and needs no
// GPU. Semantics and citations are in include/ptoc.h.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "ptoc.h"
#include "ptoc_internal.h"

namespace ptoc {

// A named NVTX range around the host side of every entry point (checks and
// launches), so that timeline tools show the library's calls by name. With
// no tool attached a range costs a few nanoseconds.
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

// The documented switch PTOC_PDL=0 turns programmatic dependent launch off.
bool programmatic_launch()
{
    const char* e = getenv("PTOC_PDL");
    return !(e && strcmp(e, "0") == 0);
}

// Which form a reduction over 2 to 8 ranks with 16-byte vectors takes: the
// staged form when the launch moves at least kStagedMinBytes (N reads plus
// its writes), the register form below. Measured on GB300: from about 1.8 GB
// per launch up the staged form is 1-5 % faster; at 0.6-1.2 GB the register
// form is up to 8 % faster on a single launch after a cold L2. The
// documented switch PTOC_REDUCE_STAGING=bulk|regs forces one form.
constexpr int64_t kStagedMinBytes = (int64_t)3 << 29;   // 1.5 GiB

bool staged_reduction(int64_t bytes)
{
    const char* e = getenv("PTOC_REDUCE_STAGING");
    if (e && strcmp(e, "bulk") == 0) return true;
    if (e && (strcmp(e, "regs") == 0 || strcmp(e, "tma") == 0)) return false;
    return bytes >= kStagedMinBytes;
}

namespace {
int sm_count();
}

int32_t first_wave_prefetch(int64_t bytes)
{
    constexpr int64_t kPrefetchBelowBytes = (int64_t)512 << 20;
    const char* e = getenv("PTOC_L2_PREFETCH");
    if ((e && strcmp(e, "0") == 0) || bytes >= kPrefetchBelowBytes) return 0;
    return 8 * sm_count();
}

uint64_t copy_wait_ns()
{
    const uint64_t dflt = 2000000000ull, most = 60000000000ull;
    const char* e = getenv("PTOC_WAIT_NS");
    if (!e || !*e) return dflt;
    char* end = nullptr;
    const unsigned long long v = strtoull(e, &end, 10);
    if (!end || *end || v < 1) return dflt;
    return v > most ? most : (uint64_t)v;
}

// Whether TREDUCE takes the tensor form (PTOC_REDUCE_STAGING=tma) where it
// applies.
bool tensor_form_selected()
{
    const char* e = getenv("PTOC_REDUCE_STAGING");
    return e && strcmp(e, "tma") == 0;
}

namespace {

int elem_size(int dtype)
{
    switch (dtype) {
    case PTOC_F32: case PTOC_I32: return 4;
    case PTOC_F16: case PTOC_BF16: return 2;
    default: return 0;
    }
}

bool valid_dtype(int dtype) { return elem_size(dtype) != 0; }

// op of TREDUCE: Sum / Max / Min ([TR] §1.3); Prod belongs to the allreduce
// family only.
ptoc_status check_op(int op)
{
    if (op == PTOC_SUM || op == PTOC_MAX || op == PTOC_MIN) return PTOC_OK;
    if (op == PTOC_PROD) return PTOC_ERR_UNSUPPORTED;
    return PTOC_ERR_INVALID_ARG;
}

// op of the allreduce family (reduce_scatter, allreduce): all four.
ptoc_status check_op_allreduce(int op)
{
    return (op >= PTOC_SUM && op <= PTOC_PROD) ? PTOC_OK : PTOC_ERR_INVALID_ARG;
}

// Byte range [lo, hi) a buffer occupies.
struct Range {
    uintptr_t lo, hi;
};

bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi; }

// Footprint in bytes of a [rows, cols] box with pitch ld, or -1 on overflow.
int64_t footprint(int64_t rows, int64_t cols, int64_t ld, int eb)
{
    if (rows == 0 || cols == 0) return 0;
    const int64_t lim = INT64_MAX / 8;
    if (rows > lim / (ld > 0 ? ld : 1)) return -1;
    const int64_t elems = (rows - 1) * ld + cols;
    if (elems > lim / eb) return -1;
    return elems * eb;
}

// The widest vector (16, 8, 4 or 2 bytes) that every address and the pitch
// allow, never narrower than one element (addresses are element-aligned).
int pick_vector_bytes(uintptr_t addr_or, int64_t pitch_bytes, int eb)
{
    const uintptr_t m = addr_or | (uintptr_t)pitch_bytes;
    for (int vb = 16; vb > eb; vb >>= 1)
        if ((m & (uintptr_t)(vb - 1)) == 0) return vb;
    return eb;
}

std::atomic<int> g_sm_count[kMaxDevices];

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    return dev;
}

int sm_count()
{
    const int dev = current_device();
    if (dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int c = 1;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1) c = 1;
    if (dev < kMaxDevices) g_sm_count[dev].store(c, std::memory_order_relaxed);
    return c;
}

// The 4-byte tile counters of the claiming exchanges come from one small
// memory pool per device, created on first use, that never returns its memory
// to the driver: it only ever holds the counters of calls in flight (one
// granule). A pool that releases at synchronization (the default pool does)
// would have to map memory again on the next call, which measured ~100 us of
// host time. During stream capture the default pool is used, so that the
// allocation becomes a graph memory node.
std::atomic<cudaMemPool_t> g_scratch_pool[kMaxDevices];
std::mutex g_scratch_pool_mu;

cudaMemPool_t scratch_pool(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    cudaMemPool_t pool = g_scratch_pool[dev].load(std::memory_order_acquire);
    if (pool) return pool;
    std::lock_guard<std::mutex> lock(g_scratch_pool_mu);
    pool = g_scratch_pool[dev].load(std::memory_order_relaxed);
    if (pool) return pool;
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = ~(uint64_t)0;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_scratch_pool[dev].store(pool, std::memory_order_release);
    return pool;
}

// A zeroed 4-byte counter in stream order on `stream`, or nullptr.
uint32_t* zeroed_counter(cudaStream_t stream)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
    void* ptr = nullptr;
    cudaError_t e;
    cudaMemPool_t pool = cap == cudaStreamCaptureStatusActive ? nullptr : scratch_pool(current_device());
    if (pool) e = cudaMallocFromPoolAsync(&ptr, sizeof(uint32_t), pool, stream);
    else e = cudaMallocAsync(&ptr, sizeof(uint32_t), stream);   // capture, or no pool of our own
    if (e != cudaSuccess) return nullptr;
    if (cudaMemsetAsync(ptr, 0, sizeof(uint32_t), stream) != cudaSuccess) {
        cudaFreeAsync(ptr, stream);
        return nullptr;
    }
    return (uint32_t*)ptr;
}

// Chunks per thread per tile of the exchanges' copy kernel: the documented
// switch PTOC_A2AV_UNROLL=4|16, else 8 (32 KiB tiles for 16-byte vectors).
int a2av_unroll()
{
    const char* e = getenv("PTOC_A2AV_UNROLL");
    if (e && strcmp(e, "4") == 0) return 4;
    if (e && strcmp(e, "16") == 0) return 16;
    return 8;
}

// Tile description of a [rows, cols] box with pitch ld for vectors of vb
// bytes and tiles of `tile_vec` vectors.
struct Box {
    int64_t rows, ld, vpr, tpr, ntiles;
    int32_t tail;
};

Box make_box(int64_t rows, int64_t cols, int64_t ld, int eb, int vb, int tile_vec)
{
    Box b;
    b.rows = rows;
    b.ld = ld;
    const int ve = vb / eb;
    b.vpr = cols / ve;
    b.tail = (int32_t)(cols - b.vpr * ve);
    b.tpr = (b.vpr + tile_vec - 1) / tile_vec;
    if (b.tpr == 0) b.tpr = 1;
    b.ntiles = rows * b.tpr;
    return b;
}

dim3 grid_for(int64_t ntiles)
{
    // One tile per CTA; the hardware block scheduler balances the tail. Very
    // large boxes fall back to a grid-stride loop inside the kernel.
    const int64_t cap = (int64_t)1 << 30;
    return dim3((unsigned)(ntiles < cap ? (ntiles > 0 ? ntiles : 1) : cap));
}

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (the library links no driver library); null if the driver lacks it.
using TensorMapEncoder = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TensorMapEncoder tensor_map_encoder()
{
    static std::once_flag once;
    static TensorMapEncoder fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = (TensorMapEncoder)f;
    });
    return fn;
}

// A tensor map over the valid box of a slice: {valid_cols, valid_rows}
// elements, rows ld * eb bytes apart, boxes of kTmaBoxCols x (4 KiB / row
// bytes) elements, zero fill outside. False if the driver refuses it.
bool encode_valid_box(CUtensorMap* m, const void* base, int eb, int64_t valid_rows, int64_t valid_cols, int64_t ld)
{
    const TensorMapEncoder enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)valid_cols, (cuuint64_t)valid_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * eb)};
    const cuuint32_t box[2] = {(cuuint32_t)kTmaBoxCols, (cuuint32_t)(kBlock * 16 / (kTmaBoxCols * eb))};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(m, eb == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
               const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TREDUCE in the tensor form, if it applies: 2 to kGroup ranks, every base
// pointer, the row pitch and a row of the valid box a multiple of 16 bytes
// (a tensor store clips a row at 16-byte granularity, so a valid row that
// ends inside a 16-byte unit would have its padding overwritten), extents
// that fit a tensor map. Returns false (nothing launched) when it does not
// apply; otherwise the launch status in *e.
bool launch_tensor_form(int dtype, const void* const* src, void* dst, int n, int op, int64_t valid_rows,
                        int64_t valid_cols, int64_t ld, int eb, cudaStream_t stream, cudaError_t* e)
{
    if (n < 2 || n > kGroup) return false;
    if (((uintptr_t)dst & 15u) || ((ld * eb) & 15) || ((valid_cols * eb) & 15)) return false;
    for (int r = 0; r < n; ++r)
        if ((uintptr_t)src[r] & 15u) return false;
    if (valid_cols > ((int64_t)1 << 32) || valid_rows > ((int64_t)1 << 32) || ld * eb >= ((int64_t)1 << 40))
        return false;
    TmaReduceParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r)
        if (!encode_valid_box(&p.src[r], src[r], eb, valid_rows, valid_cols, ld)) return false;
    if (!encode_valid_box(&p.dst, dst, eb, valid_rows, valid_cols, ld)) return false;
    const int64_t box_rows = kBlock * 16 / (kTmaBoxCols * eb);
    const int64_t tiles_x = (valid_cols + kTmaBoxCols - 1) / kTmaBoxCols;
    const int64_t tiles_y = (valid_rows + box_rows - 1) / box_rows;
    if (tiles_x > INT32_MAX) return false;
    p.tiles_x = (int32_t)tiles_x;
    p.ntiles = tiles_x * tiles_y;
    p.nranks = n;
    p.wait_ns = copy_wait_ns();
    switch (dtype) {
    case PTOC_F32: *e = launch_tma_reduce_f32(p, op, stream); break;
    case PTOC_I32: *e = launch_tma_reduce_i32(p, op, stream); break;
    case PTOC_F16: *e = launch_tma_reduce_f16(p, op, stream); break;
    default: *e = launch_tma_reduce_bf16(p, op, stream); break;
    }
    return true;
}

cudaError_t launch_reduce_regs(int dtype, const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s)
{
    switch (dtype) {
    case PTOC_F32: return launch_reduce_f32(p, op, vb, grid, s);
    case PTOC_I32: return launch_reduce_i32(p, op, vb, grid, s);
    case PTOC_F16: return launch_reduce_f16(p, op, vb, grid, s);
    default: return launch_reduce_bf16(p, op, vb, grid, s);
    }
}

// Tile a [rows, cols] box with pitch ld and launch one reduction over it
// (p.src, p.dst, p.nranks and p.dst_mode already filled in): one block per
// tile of kBlock vectors of vb bytes, then the row-tail blocks.
cudaError_t launch_reduction(int dtype, ReduceParams& p, int op, int64_t rows, int64_t cols, int64_t ld,
                             int eb, int vb, cudaStream_t s)
{
    p.ld = ld;
    p.rows = rows;
    // 13 to 16 ranks: 8-byte vectors, so all their loads fit in flight at
    // once in the registers of one group of 16-byte loads (9 to 12 ranks keep
    // 16-byte vectors in a 12-slot form)
    if (p.nranks > 12 && p.nranks <= 2 * kGroup && vb > 8) vb = 8;
    const Box b = make_box(rows, cols, ld, eb, vb, kBlock);
    p.vpr = b.vpr;
    p.tail = b.tail;
    p.tpr = b.tpr;
    p.ntiles = b.ntiles;
    p.tail_blocks = b.tail > 0 ? (rows * b.tail + kBlock - 1) / kBlock : 0;
    // bytes the launch moves: N reads and one write per element (N writes to
    // every window for allreduce)
    const int64_t writes = p.dst_mode == kDstAll ? p.nranks : 1;
    const int64_t elems = rows > 0 && cols > 0 ? rows * cols : 0;
    const int64_t per_elem = (p.nranks + writes) * eb;
    const int64_t bytes = elems > INT64_MAX / per_elem ? INT64_MAX : per_elem * elems;
    p.staged = staged_reduction(bytes) ? 1 : 0;
    p.prefetch_blocks = p.staged ? 0 : first_wave_prefetch(bytes);
    p.wait_ns = copy_wait_ns();
    return launch_reduce_regs(dtype, p, op, vb, grid_for(p.ntiles + p.tail_blocks), s);
}

ptoc_status check_group(const ptoc_group* g, bool need_root)
{
    if (!g || !g->tensors) return PTOC_ERR_INVALID_ARG;
    if (g->nranks < 1 || g->nranks > kMaxRanks) return PTOC_ERR_INVALID_ARG;
    if (need_root && (g->root < 0 || g->root >= g->nranks)) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < g->nranks; ++r)
        if (!g->tensors[r]) return PTOC_ERR_INVALID_ARG;
    return PTOC_OK;
}

bool aligned(const void* p, int eb) { return ((uintptr_t)p % (uintptr_t)eb) == 0; }

// Shared checks of the window collectives (reduce_scatter, allgather,
// allreduce, broadcast): group, dtype, sizes, alignment, disjoint windows.
ptoc_status check_windows(const ptoc_group* w, int64_t rows, int64_t cols, int64_t ld, int dtype,
                          int64_t* fp_out)
{
    ptoc_status st = check_group(w, false);
    if (st != PTOC_OK) return st;
    if (!valid_dtype(dtype)) return PTOC_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ld < 0 || (rows > 0 && cols > ld)) return PTOC_ERR_INVALID_ARG;
    const int eb = elem_size(dtype);
    const int64_t fp = footprint(rows, cols, ld, eb);
    if (fp < 0) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < w->nranks; ++r)
        if (!aligned(w->tensors[r], eb)) return PTOC_ERR_INVALID_ARG;
    for (int a = 0; a < w->nranks; ++a)
        for (int b = a + 1; b < w->nranks; ++b) {
            const Range ra{(uintptr_t)w->tensors[a], (uintptr_t)w->tensors[a] + (uintptr_t)fp};
            const Range rb{(uintptr_t)w->tensors[b], (uintptr_t)w->tensors[b] + (uintptr_t)fp};
            if (overlap(ra, rb)) return PTOC_ERR_ALIAS;
        }
    *fp_out = fp;
    return PTOC_OK;
}

// Shared checks of the pairwise exchanges over [target_rows, size] buffers
// (all_to_all_v, all_to_all, the combine). `writes` are the spans the call
// writes, `reads` the ones it only reads; outputs must not overlap anything,
// inputs may overlap each other.
struct Span {
    const void* p;
    uintptr_t bytes;
};

ptoc_status check_disjoint_outputs(const Span* writes, int nw, const Span* reads, int nr)
{
    for (int a = 0; a < nw; ++a) {
        const Range ra{(uintptr_t)writes[a].p, (uintptr_t)writes[a].p + writes[a].bytes};
        for (int b = a + 1; b < nw; ++b) {
            const Range rb{(uintptr_t)writes[b].p, (uintptr_t)writes[b].p + writes[b].bytes};
            if (overlap(ra, rb)) return PTOC_ERR_ALIAS;
        }
        for (int b = 0; b < nr; ++b) {
            const Range rb{(uintptr_t)reads[b].p, (uintptr_t)reads[b].p + reads[b].bytes};
            if (overlap(ra, rb)) return PTOC_ERR_ALIAS;
        }
    }
    return PTOC_OK;
}

// Vector width and tile of a pairwise exchange (sets p.tile_bytes); `add`
// selects the combine's add mover, which moves 4 chunks per thread.
struct PairsPlan {
    int vb, unroll;
    int64_t run_tiles;   // tiles of the longest possible run (MAX_RECV rows)
};

PairsPlan plan_pairs(A2avParams& p, const void* const* a, const void* const* b, int n, int eb, bool add)
{
    uintptr_t addr_or = 0;
    for (int r = 0; r < n; ++r) addr_or |= (uintptr_t)a[r] | (uintptr_t)b[r];
    PairsPlan pl;
    pl.vb = pick_vector_bytes(addr_or, p.row_bytes, eb);
    pl.unroll = add ? 4 : a2av_unroll();
    p.tile_bytes = (int64_t)pl.vb * kBlock * pl.unroll;
    const int64_t run = p.max_recv * p.row_bytes;
    pl.run_tiles = (run + p.tile_bytes - 1) / p.tile_bytes;
    return pl;
}

// Tile indices are int32 in the claiming kernel.
bool claim_fits(int n, const PairsPlan& pl) { return (int64_t)n * n * (pl.run_tiles + 1) < INT32_MAX; }

// One wave of blocks claiming the live tiles from `counter`, which the
// stream has zeroed before this launch.
cudaError_t launch_claimed(A2avParams& p, const PairsPlan& pl, int n, int dtype, bool add, uint32_t* counter,
                           cudaStream_t stream)
{
    const int grid = sm_count() * pairs_claim_blocks_per_sm(add, dtype, pl.vb, pl.unroll, n);
    p.claim = counter;
    return launch_pairs_claim(p, add, dtype, pl.vb, pl.unroll, grid, stream);
}

ptoc_status launch_pairs(A2avParams& p, const void* const* a, const void* const* b, int n, int eb, int dtype,
                         bool add, cudaStream_t stream)
{
    const PairsPlan pl = plan_pairs(p, a, b, n, eb, add);
    if (p.full) {
        // every count is MAX_RECV: grid.y = the N^2 pairs, grid.x = the tiles of a run
        const int64_t cap = (int64_t)1 << 30;
        const int64_t gx = pl.run_tiles < 1 ? 1 : (pl.run_tiles > cap ? cap : pl.run_tiles);
        const dim3 grid((unsigned)gx, (unsigned)(n * n));
        const cudaError_t e = add ? launch_pairs_add(p, dtype, pl.vb, grid, stream)
                                  : launch_a2av(p, pl.vb, pl.unroll, grid, stream);
        return e == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
    }
    // counts on the device: one wave of blocks claims the live tiles from a
    // zeroed counter (a 4-byte stream-ordered allocation, freed in stream
    // order after the launch)
    if (!claim_fits(n, pl)) return PTOC_ERR_UNSUPPORTED;
    uint32_t* claim = zeroed_counter(stream);
    if (!claim) return PTOC_ERR_CUDA;
    const cudaError_t e = launch_claimed(p, pl, n, dtype, add, claim, stream);
    const cudaError_t f = cudaFreeAsync(claim, stream);
    return (e == cudaSuccess && f == cudaSuccess) ? PTOC_OK : PTOC_ERR_CUDA;
}

ptoc_status check_pair_group(const ptoc_group* a, const ptoc_group* b)
{
    ptoc_status st = check_group(a, false);
    if (st != PTOC_OK) return st;
    st = check_group(b, false);
    if (st != PTOC_OK) return st;
    return a->nranks == b->nranks ? PTOC_OK : PTOC_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace ptoc

using namespace ptoc;

extern "C" ptoc_status ptoc_treduce(const ptoc_group* group, void* dst, int64_t rows, int64_t cols,
                                    int64_t valid_rows, int64_t valid_cols, int64_t ld,
                                    ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_treduce");
    ptoc_status st = check_group(group, true);
    if (st != PTOC_OK) return st;
    if (!dst) return PTOC_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return PTOC_ERR_INVALID_ARG;
    st = check_op(op);
    if (st != PTOC_OK) return st;
    if (rows < 0 || cols < 0 || valid_rows < 0 || valid_cols < 0 || ld < 0) return PTOC_ERR_INVALID_ARG;
    if (valid_rows > rows || valid_cols > cols || (rows > 0 && cols > ld)) return PTOC_ERR_INVALID_ARG;
    const int eb = elem_size(dtype);
    if (footprint(rows, cols, ld, eb) < 0) return PTOC_ERR_INVALID_ARG;
    const int n = group->nranks;
    if (!aligned(dst, eb)) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r)
        if (!aligned(group->tensors[r], eb)) return PTOC_ERR_INVALID_ARG;

    // Empty valid region: nothing is read or written (TREDUCE article §4.1).
    if (valid_rows == 0 || valid_cols == 0) return PTOC_OK;

    // dst may be exactly the root's slice (in place); any other overlap of the
    // valid footprints is an alias.
    const int64_t fp = footprint(valid_rows, valid_cols, ld, eb);
    const Range rd{(uintptr_t)dst, (uintptr_t)dst + (uintptr_t)fp};
    for (int r = 0; r < n; ++r) {
        const void* s = group->tensors[r];
        if (s == dst && r == group->root) continue;
        const Range rs{(uintptr_t)s, (uintptr_t)s + (uintptr_t)fp};
        if (overlap(rd, rs)) return PTOC_ERR_ALIAS;
    }

    ReduceParams p;
    memset(&p, 0, sizeof(p));
    // Reduction order (TREDUCE article §4.3): root first, then ascending.
    int k = 0;
    p.src[k++] = group->tensors[group->root];
    for (int r = 0; r < n; ++r)
        if (r != group->root) p.src[k++] = group->tensors[r];
    p.dst[0] = dst;
    p.nranks = n;
    p.dst_mode = kDstOne;
    // One rank: a bit copy (TREDUCE article §4.3). Max with a single operand
    // is exactly that, NaN payloads included.
    const int eff_op = (n == 1) ? PTOC_MAX : (int)op;

    if (tensor_form_selected()) {
        cudaError_t e = cudaSuccess;
        if (launch_tensor_form(dtype, p.src, dst, n, eff_op, valid_rows, valid_cols, ld, eb, stream, &e))
            return e == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
    }

    // Contiguous valid box (full rows, or a single row): one flat row.
    const bool flat = (valid_cols == ld) || (valid_rows == 1);
    const int64_t frows = flat ? 1 : valid_rows;
    const int64_t fcols = flat ? valid_rows * ld - (ld - valid_cols) : valid_cols;
    const int64_t fld = flat ? fcols : ld;
    uintptr_t addr_or = (uintptr_t)dst;
    for (int r = 0; r < n; ++r) addr_or |= (uintptr_t)group->tensors[r];
    const int vb = pick_vector_bytes(addr_or, flat ? 0 : ld * eb, eb);
    cudaError_t e = launch_reduction(dtype, p, eff_op, frows, fcols, fld, eb, vb, stream);
    return e == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
}

// reduce_scatter (dst_mode kDstOwner) and allreduce (kDstAll) over windows.
static ptoc_status window_reduction(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                                    ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream, int dst_mode)
{
    int64_t fp = 0;
    ptoc_status st = check_windows(windows, rows, cols, ld, dtype, &fp);
    if (st != PTOC_OK) return st;
    st = check_op_allreduce(op);
    if (st != PTOC_OK) return st;
    const int n = windows->nranks;
    // Nothing to do: an empty box, or one rank (its window already holds the
    // reduction of itself).
    if (rows == 0 || cols == 0 || n == 1) return PTOC_OK;
    const int eb = elem_size(dtype);

    ReduceParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) {
        p.src[r] = windows->tensors[r];     // rank order 0..N-1
        p.dst[r] = windows->tensors[r];
    }
    p.nranks = n;
    p.dst_mode = dst_mode;
    uintptr_t addr_or = 0;
    for (int r = 0; r < n; ++r) addr_or |= (uintptr_t)windows->tensors[r];
    // allreduce writes every window with the same value: when the windows are
    // whole rows it is one flat row
    const bool flat = (dst_mode == kDstAll) && (cols == ld || rows == 1);
    const int64_t frows = flat ? 1 : rows;
    const int64_t fcols = flat ? rows * ld - (ld - cols) : cols;
    const int64_t fld = flat ? fcols : ld;
    const int vb = pick_vector_bytes(addr_or, flat ? 0 : ld * eb, eb);
    cudaError_t e = launch_reduction(dtype, p, (int)op, frows, fcols, fld, eb, vb, stream);
    return e == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
}

extern "C" ptoc_status ptoc_reduce_scatter(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                                           ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_reduce_scatter");
    return window_reduction(windows, rows, cols, ld, op, dtype, stream, kDstOwner);
}

extern "C" ptoc_status ptoc_allreduce(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                                      ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_allreduce");
    return window_reduction(windows, rows, cols, ld, op, dtype, stream, kDstAll);
}

// allgather (root < 0: row i comes from its owner window) and broadcast
// (every row comes from window `root`).
static ptoc_status window_copy(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                               ptoc_dtype dtype, cudaStream_t stream, int root)
{
    const int n = windows->nranks;
    const int eb = elem_size(dtype);
    GatherParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) p.win[r] = windows->tensors[r];
    p.nranks = n;
    p.root = root;
    uintptr_t addr_or = 0;
    for (int r = 0; r < n; ++r) addr_or |= (uintptr_t)windows->tensors[r];
    // broadcast copies the same rows to every window: whole rows are one flat row
    const bool flat = (root >= 0) && (cols == ld || rows == 1);
    const int64_t frows = flat ? 1 : rows;
    const int64_t fcols = flat ? rows * ld - (ld - cols) : cols;
    const int64_t fld = flat ? fcols : ld;
    const int vb = pick_vector_bytes(addr_or, flat ? 0 : ld * eb, eb);
    const Box b = make_box(frows, fcols, fld, eb, vb, kBlock);
    p.ld = fld;
    p.rows = frows;
    p.vpr = b.vpr;
    p.tail = b.tail;
    p.tpr = b.tpr;
    p.ntiles = b.ntiles;
    cudaError_t e = launch_gather(p, eb, vb, grid_for(p.ntiles), stream);
    return e == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
}

extern "C" ptoc_status ptoc_allgather(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                                      ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_allgather");
    int64_t fp = 0;
    ptoc_status st = check_windows(windows, rows, cols, ld, dtype, &fp);
    if (st != PTOC_OK) return st;
    if (rows == 0 || cols == 0 || windows->nranks == 1) return PTOC_OK;
    return window_copy(windows, rows, cols, ld, dtype, stream, -1);
}

extern "C" ptoc_status ptoc_broadcast(const ptoc_group* windows, int64_t rows, int64_t cols, int64_t ld,
                                      ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_broadcast");
    ptoc_status st = check_group(windows, true);
    if (st != PTOC_OK) return st;
    int64_t fp = 0;
    st = check_windows(windows, rows, cols, ld, dtype, &fp);
    if (st != PTOC_OK) return st;
    if (rows == 0 || cols == 0 || windows->nranks == 1) return PTOC_OK;
    return window_copy(windows, rows, cols, ld, dtype, stream, windows->root);
}

// Checks and kernel parameters of an all_to_all_v call (no CUDA call).
static ptoc_status a2av_setup(const ptoc_group* inputs, const ptoc_group* targets,
                              const int32_t* const* send_counts, int32_t* const* recv_counts,
                              int64_t target_rows, int64_t size, ptoc_dtype dtype, A2avParams& p, int& eb)
{
    ptoc_status st = check_pair_group(inputs, targets);
    if (st != PTOC_OK) return st;
    if (!send_counts || !recv_counts) return PTOC_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return PTOC_ERR_INVALID_ARG;
    if (target_rows < 0 || size < 0) return PTOC_ERR_INVALID_ARG;
    const int n = inputs->nranks;
    eb = elem_size(dtype);
    const int64_t fp = footprint(target_rows, size, size, eb);
    if (fp < 0) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r) {
        if (!send_counts[r] || !recv_counts[r]) return PTOC_ERR_INVALID_ARG;
        if (!aligned(send_counts[r], 4) || !aligned(recv_counts[r], 4)) return PTOC_ERR_INVALID_ARG;
        if (!aligned(inputs->tensors[r], eb) || !aligned(targets->tensors[r], eb)) return PTOC_ERR_INVALID_ARG;
    }
    // Outputs (targets, recv_counts) must not overlap anything (the page
    // requires the five operands to be pairwise-distinct allocations); inputs
    // may share memory.
    Span writes[2 * kMaxRanks] = {}, reads[2 * kMaxRanks] = {};
    for (int r = 0; r < n; ++r) {
        writes[r] = Span{targets->tensors[r], (uintptr_t)fp};
        writes[n + r] = Span{recv_counts[r], (uintptr_t)n * 4u};
        reads[r] = Span{inputs->tensors[r], (uintptr_t)fp};
        reads[n + r] = Span{send_counts[r], (uintptr_t)n * 4u};
    }
    st = check_disjoint_outputs(writes, 2 * n, reads, 2 * n);
    if (st != PTOC_OK) return st;

    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) {
        p.in[r] = inputs->tensors[r];
        p.out[r] = targets->tensors[r];
        p.cnt[r] = send_counts[r];
        p.pub[r] = recv_counts[r];
    }
    p.nranks = n;
    p.max_recv = target_rows / n;
    p.row_bytes = size * eb;
    p.full = 0;
    p.publish = 1;
    return PTOC_OK;
}

extern "C" ptoc_status ptoc_all_to_all_v(const ptoc_group* inputs, const ptoc_group* targets,
                                         const int32_t* const* send_counts, int32_t* const* recv_counts,
                                         int64_t target_rows, int64_t size, ptoc_dtype dtype,
                                         cudaStream_t stream)
{
    const TraceRange trace("ptoc_all_to_all_v");
    A2avParams p;
    int eb = 0;
    const ptoc_status st = a2av_setup(inputs, targets, send_counts, recv_counts, target_rows, size, dtype, p, eb);
    if (st != PTOC_OK) return st;
    return launch_pairs(p, inputs->tensors, targets->tensors, inputs->nranks, eb, dtype, false, stream);
}

// ---- all_to_all_v without allocation ------------------------------------------

// The scratch of ptoc_all_to_all_v_noalloc: a fixed 256-byte block of device
// memory in the library image (zero at load). A call needs one 4-byte tile
// counter from it; calls in flight at the same time share it and race.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

namespace {

// Per-device cache of the block's address. Like the other per-device caches
// of the library (SM counts, the counter pool), it assumes the device's
// primary context lives as long as the process: after a cudaDeviceReset the
// cached values are stale.
std::atomic<void*> g_noalloc_addr[kMaxDevices];

}  // namespace

// The scratch block's device address on the current device, looked up once
// per device (with that device current).
static uint32_t* noalloc_scratch()
{
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    void* a = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return nullptr;
        g_noalloc_addr[dev].store(a, std::memory_order_release);
    }
    return (uint32_t*)a;
}

extern "C" ptoc_status ptoc_all_to_all_v_noalloc(const ptoc_group* inputs, const ptoc_group* targets,
                                                 const int32_t* const* send_counts, int32_t* const* recv_counts,
                                                 int64_t target_rows, int64_t size, ptoc_dtype dtype,
                                                 cudaStream_t stream)
{
    const TraceRange trace("ptoc_all_to_all_v_noalloc");
    A2avParams p;
    int eb = 0;
    const ptoc_status st = a2av_setup(inputs, targets, send_counts, recv_counts, target_rows, size, dtype, p, eb);
    if (st != PTOC_OK) return st;
    const int n = inputs->nranks;
    const PairsPlan pl = plan_pairs(p, inputs->tensors, targets->tensors, n, eb, false);
    if (!claim_fits(n, pl)) return PTOC_ERR_UNSUPPORTED;
    const size_t need = sizeof(uint32_t);        // the tile counter
    if (need > kNoAllocScratchBytes) return PTOC_ERR_UNSUPPORTED;
    uint32_t* counter = noalloc_scratch();
    if (!counter) return PTOC_ERR_CUDA;
    // the counter must start at zero for every call
    if (cudaMemsetAsync(counter, 0, need, stream) != cudaSuccess) return PTOC_ERR_CUDA;
    return launch_claimed(p, pl, n, dtype, false, counter, stream) == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
}

extern "C" ptoc_status ptoc_all_to_all(const ptoc_group* inputs, const ptoc_group* targets,
                                       int64_t target_rows, int64_t size, ptoc_dtype dtype, cudaStream_t stream)
{
    const TraceRange trace("ptoc_all_to_all");
    ptoc_status st = check_pair_group(inputs, targets);
    if (st != PTOC_OK) return st;
    if (!valid_dtype(dtype)) return PTOC_ERR_INVALID_ARG;
    if (target_rows < 0 || size < 0) return PTOC_ERR_INVALID_ARG;
    const int n = inputs->nranks;
    const int eb = elem_size(dtype);
    const int64_t fp = footprint(target_rows, size, size, eb);
    if (fp < 0) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r)
        if (!aligned(inputs->tensors[r], eb) || !aligned(targets->tensors[r], eb)) return PTOC_ERR_INVALID_ARG;
    Span writes[kMaxRanks] = {}, reads[kMaxRanks] = {};
    for (int r = 0; r < n; ++r) {
        writes[r] = Span{targets->tensors[r], (uintptr_t)fp};
        reads[r] = Span{inputs->tensors[r], (uintptr_t)fp};
    }
    st = check_disjoint_outputs(writes, n, reads, n);
    if (st != PTOC_OK) return st;
    const int64_t chunk = target_rows / n;
    if (chunk == 0 || size == 0) return PTOC_OK;

    A2avParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) {
        p.in[r] = inputs->tensors[r];
        p.out[r] = targets->tensors[r];
    }
    p.nranks = n;
    p.max_recv = chunk;
    p.row_bytes = size * eb;
    p.full = 1;
    p.publish = 0;
    return launch_pairs(p, inputs->tensors, targets->tensors, n, eb, dtype, false, stream);
}

extern "C" ptoc_status ptoc_all_to_all_v_combine(const ptoc_group* windows, const ptoc_group* outputs,
                                                 const int32_t* const* recv_counts, int64_t target_rows,
                                                 int64_t size, ptoc_atomic_type atomic, ptoc_dtype dtype,
                                                 cudaStream_t stream)
{
    const TraceRange trace("ptoc_all_to_all_v_combine");
    ptoc_status st = check_pair_group(windows, outputs);
    if (st != PTOC_OK) return st;
    if (!recv_counts) return PTOC_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return PTOC_ERR_INVALID_ARG;
    if (atomic != PTOC_ATOMIC_NONE && atomic != PTOC_ATOMIC_ADD) return PTOC_ERR_INVALID_ARG;
    if (target_rows < 0 || size < 0) return PTOC_ERR_INVALID_ARG;
    const int n = windows->nranks;
    const int eb = elem_size(dtype);
    const int64_t fp = footprint(target_rows, size, size, eb);
    if (fp < 0) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r) {
        if (!recv_counts[r] || !aligned(recv_counts[r], 4)) return PTOC_ERR_INVALID_ARG;
        if (!aligned(windows->tensors[r], eb) || !aligned(outputs->tensors[r], eb)) return PTOC_ERR_INVALID_ARG;
    }
    Span writes[kMaxRanks] = {}, reads[2 * kMaxRanks] = {};
    for (int r = 0; r < n; ++r) {
        writes[r] = Span{outputs->tensors[r], (uintptr_t)fp};
        reads[r] = Span{windows->tensors[r], (uintptr_t)fp};
        reads[n + r] = Span{recv_counts[r], (uintptr_t)n * 4u};
    }
    st = check_disjoint_outputs(writes, n, reads, 2 * n);
    if (st != PTOC_OK) return st;
    if (target_rows / n == 0 || size == 0) return PTOC_OK;

    A2avParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) {
        p.in[r] = windows->tensors[r];      // pair (a = d, b = s): window d -> output s
        p.out[r] = outputs->tensors[r];
        p.cnt[r] = recv_counts[r];
    }
    p.nranks = n;
    p.max_recv = target_rows / n;
    p.row_bytes = size * eb;
    p.full = 0;
    p.publish = 0;
    return launch_pairs(p, windows->tensors, outputs->tensors, n, eb, dtype, atomic == PTOC_ATOMIC_ADD, stream);
}

extern "C" ptoc_status ptoc_credit_barrier(const ptoc_group* signals, const int32_t* local_ranks, int32_t n_local,
                                           int32_t generations, int64_t timeout_ns, int32_t* status,
                                           cudaStream_t stream)
{
    const TraceRange trace("ptoc_credit_barrier");
    ptoc_status st = check_group(signals, false);
    if (st != PTOC_OK) return st;
    const int n = signals->nranks;
    if (!local_ranks || !status) return PTOC_ERR_INVALID_ARG;
    if (n_local < 1 || n_local > n) return PTOC_ERR_INVALID_ARG;
    if (generations < 0 || generations > (1 << 30)) return PTOC_ERR_INVALID_ARG;
    if (timeout_ns <= 0 || timeout_ns > (int64_t)60 * 1000 * 1000 * 1000) return PTOC_ERR_INVALID_ARG;
    if (!aligned(status, 4)) return PTOC_ERR_INVALID_ARG;
    bool seen[kMaxRanks] = {false};
    for (int i = 0; i < n_local; ++i) {
        const int r = local_ranks[i];
        if (r < 0 || r >= n || seen[r]) return PTOC_ERR_INVALID_ARG;
        seen[r] = true;
    }
    for (int r = 0; r < n; ++r)
        if (!aligned(signals->tensors[r], 4)) return PTOC_ERR_INVALID_ARG;
    Span writes[kMaxRanks + 1] = {};
    for (int r = 0; r < n; ++r) writes[r] = Span{signals->tensors[r], (uintptr_t)n * 4u};
    writes[n] = Span{status, (uintptr_t)n_local * 4u};
    st = check_disjoint_outputs(writes, n + 1, nullptr, 0);
    if (st != PTOC_OK) return st;

    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, current_device()) != cudaSuccess || !coop)
        return PTOC_ERR_UNSUPPORTED;
    BarrierParams p;
    memset(&p, 0, sizeof(p));
    for (int r = 0; r < n; ++r) p.sig[r] = (int32_t*)signals->tensors[r];
    for (int i = 0; i < n_local; ++i) p.local[i] = local_ranks[i];
    p.status = status;
    p.timeout_ns = timeout_ns;
    p.nranks = n;
    p.nlocal = n_local;
    p.generations = generations;
    return launch_credit_barrier(p, stream) == cudaSuccess ? PTOC_OK : PTOC_ERR_CUDA;
}

extern "C" ptoc_status ptoc_signal_reset(const ptoc_group* signals, cudaStream_t stream)
{
    const TraceRange trace("ptoc_signal_reset");
    ptoc_status st = check_group(signals, false);
    if (st != PTOC_OK) return st;
    const int n = signals->nranks;
    for (int r = 0; r < n; ++r)
        if (!aligned(signals->tensors[r], 4)) return PTOC_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r)
        if (cudaMemsetAsync(signals->tensors[r], 0, (size_t)n * 4u, stream) != cudaSuccess) return PTOC_ERR_CUDA;
    return PTOC_OK;
}

extern "C" ptoc_status ptoc_wait_faults(uint32_t* count)
{
    const TraceRange trace("ptoc_wait_faults");
    if (!count) return PTOC_ERR_INVALID_ARG;
    uint32_t total = 0;
    cudaError_t (*const take[])(uint32_t*) = {take_stage_faults_f32, take_stage_faults_i32, take_stage_faults_f16,
                                               take_stage_faults_bf16};
    for (auto f : take) {
        uint32_t v = 0;
        if (f(&v) != cudaSuccess) return PTOC_ERR_CUDA;
        total += v;
    }
    *count = total;
    return PTOC_OK;
}

extern "C" const char* ptoc_status_string(ptoc_status s)
{
    switch (s) {
    case PTOC_OK: return "PTOC_OK";
    case PTOC_ERR_INVALID_ARG: return "PTOC_ERR_INVALID_ARG";
    case PTOC_ERR_UNSUPPORTED: return "PTOC_ERR_UNSUPPORTED";
    case PTOC_ERR_ALIAS: return "PTOC_ERR_ALIAS";
    case PTOC_ERR_CUDA: return "PTOC_ERR_CUDA";
    default: return "PTOC_ERR_UNKNOWN";
    }
}
