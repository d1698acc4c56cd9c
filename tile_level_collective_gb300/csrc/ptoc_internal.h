// Internal declarations shared by the library's translation units: kernel
// parameter blocks (passed by value, so they need no device memory) and the
// per-dtype launchers the C-ABI layer dispatches to.
#pragma once

#include <cstdint>
#include <cuda.h>              // CUtensorMap (a type only: the library links no driver library)
#include <cuda_runtime_api.h>

#include "ptoc.h"

namespace ptoc {

constexpr int kMaxRanks = PTOC_MAX_RANKS;
constexpr int kBlock = 256;          // threads per CTA for every streaming kernel
constexpr int kGroup = 8;            // ranks whose 16-byte loads a reduction thread issues together
constexpr int kMaxDevices = 64;      // per-device caches

enum Op : int { kSum = 0, kMax = 1, kMin = 2, kProd = 3 };

// Where a reduction writes: one dst, the owner window of each row
// (reduce_scatter), or every window (allreduce).
enum DstMode : int { kDstOne = 0, kDstOwner = 1, kDstAll = 2 };

// TREDUCE, reduce_scatter and allreduce. The box is `rows` rows of `vpr` full vectors of
// VB bytes plus `tail` trailing elements; one tile is one row segment of
// kBlock vectors; the row tails are reduced by tail_blocks extra blocks.
struct ReduceParams {
    const void* src[kMaxRanks];   // sources in reduction order (root first)
    void* dst[kMaxRanks];         // dst[0] for TREDUCE; window r for reduce_scatter / allreduce
    int64_t ld;                   // row pitch, elements
    int64_t rows;                 // rows of the box (also the scatter chunk basis)
    int64_t vpr;                  // full vectors per row
    int64_t tpr;                  // tiles per row
    int64_t ntiles;               // rows * tpr
    int64_t tail_blocks;          // blocks after the tiles that reduce the row tails
    int32_t tail;                 // elements after the last full vector of a row
    int32_t nranks;
    int32_t dst_mode;             // DstMode
    int32_t staged;               // 1: the staged form where it applies (host-side choice)
    int32_t prefetch_blocks;      // blocks below this prefetch their first tile into L2 (register form)
    uint64_t wait_ns;             // the staged form's bound on one wait for a copy
};

// TREDUCE through tensor maps (the tensor form): src[r] describes source r
// (reduction order, root first) and dst the destination, each over the valid
// box only: globalDim = {valid_cols, valid_rows}, row stride ld * element
// bytes, box = kTmaBoxCols elements x box_rows rows (4 KiB). Loads of a box
// that reaches past the valid box fill the outside with zeros; stores clip
// at it, so padding is never written. Tile w is the box at column
// (w % tiles_x) * kTmaBoxCols, row (w / tiles_x) * box_rows. Stores clip a
// row at 16-byte granularity, so the form needs valid rows of a multiple of
// 16 bytes (the host checks it). Passed by value
// as a __grid_constant__ parameter (tensor maps must live in parameter,
// constant or global memory).
constexpr int kTmaBoxCols = 256;
struct TmaReduceParams {
    CUtensorMap src[kGroup];
    CUtensorMap dst;
    int64_t ntiles;
    uint64_t wait_ns;             // bound on one wait for a box
    int32_t tiles_x;
    int32_t nranks;
};

// The bound, in nanoseconds, on one wait of the staged and tensor forms for a
// copy: 2 s, or the documented switch PTOC_WAIT_NS (1 ns to 60 s).
uint64_t copy_wait_ns();

// allgather / broadcast: same box description; win[r] is rank r's window.
// Row i is read from win[owner(i)] (allgather) or from win[root] when
// root >= 0 (broadcast), and written to every other window.
struct GatherParams {
    void* win[kMaxRanks];
    int64_t ld, rows, vpr, tpr, ntiles;
    int32_t tail, nranks, root;
};

// Pairwise exchanges over the flat [N * MAX_RECV, size] layout. Pair (a, b)
// moves count(a, b) rows from in[a] rows [b * MAX_RECV, ..) to out[b] rows
// [a * MAX_RECV, ..):
//   all_to_all_v : a = sender, b = destination, count = clamp(cnt[a][b]) with
//                  cnt = send_counts; publishes pub[b][a] = count.
//   all_to_all   : count = MAX_RECV for every pair (cnt unused).
//   combine      : a = the rank that received, b = the original sender,
//                  count = clamp(cnt[a][b]) with cnt = recv_counts; out is
//                  overwritten or added into (AtomicType).
// Each pair is one contiguous segment cut into tiles of tile_bytes. With every
// count known (full), block (x, q) of a 2-D launch moves tile x of pair q.
// With counts on the device, a persistent grid claims the live tiles in order
// from the counter at `claim`.
struct A2avParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    const int32_t* cnt[kMaxRanks];
    int32_t* pub[kMaxRanks];
    int64_t max_recv;             // target_rows / nranks
    int64_t row_bytes;            // size * element bytes
    int64_t tile_bytes;           // bytes one block moves (the last tile of a run is shorter)
    uint32_t* claim;              // tile counter of the claiming kernel (zeroed before the launch)
    int32_t nranks;
    int32_t full;                 // 1: every count is MAX_RECV
    int32_t publish;              // 1: write pub[b][a]
};

// The credit barrier: sig[p] is rank p's signal window (nranks int32 cells,
// cell s = credits from rank s); the launch runs the ranks local[0..nlocal),
// one warp each; status[i] receives local[i]'s result (0, or the generation it
// timed out in).
struct BarrierParams {
    int32_t* sig[kMaxRanks];
    int32_t local[kMaxRanks];
    int32_t* status;
    int64_t timeout_ns;
    int32_t nranks, nlocal, generations;
};

cudaError_t launch_credit_barrier(const BarrierParams& p, cudaStream_t s);

// Whether the data kernels are launched as programmatic dependent launches:
// a launch may then overlap the tail of the previous kernel of the stream,
// and the kernel itself waits for that kernel to complete (and its writes to
// be visible) before touching memory. On by default; the documented switch
// PTOC_PDL=0 turns it off.
bool programmatic_launch();

// How many of a register-form reduction's first blocks prefetch their first
// tile into L2 before waiting for the previous kernel of the stream: the
// first wave (8 blocks per SM) for launches that move less than 512 MiB,
// none for larger ones or when the documented switch PTOC_L2_PREFETCH=0 is
// set.
int32_t first_wave_prefetch(int64_t bytes);

// Whether a reduction that moves `bytes` per launch takes the staged form
// (sources copied into shared memory by the bulk-copy engine) where it
// applies (2 to kGroup ranks, 16-byte vectors) rather than the register form:
// by size, unless the documented switch PTOC_REDUCE_STAGING (bulk | regs)
// forces one.
bool staged_reduction(int64_t bytes);

// Launchers (one translation unit per element type for the reductions).
// `vb` is the vector width in bytes (16, 8 or 4; 2 for 16-bit data that is
// only 2-byte aligned). They return the launch status; they never allocate.
cudaError_t launch_reduce_f32(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s);
cudaError_t launch_reduce_i32(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s);
cudaError_t launch_reduce_f16(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s);
cudaError_t launch_reduce_bf16(const ReduceParams& p, int op, int vb, dim3 grid, cudaStream_t s);
// The tensor form of TREDUCE, per element type (4 or 2 bytes: the copies
// move bits, the fold is the type's).
cudaError_t launch_tma_reduce_f32(const TmaReduceParams& p, int op, cudaStream_t s);
cudaError_t launch_tma_reduce_i32(const TmaReduceParams& p, int op, cudaStream_t s);
cudaError_t launch_tma_reduce_f16(const TmaReduceParams& p, int op, cudaStream_t s);
cudaError_t launch_tma_reduce_bf16(const TmaReduceParams& p, int op, cudaStream_t s);
// Per element type: read the count of staged tiles whose wait on a copy gave
// up (in that translation unit's device memory) and reset it to zero.
cudaError_t take_stage_faults_f32(uint32_t* count);
cudaError_t take_stage_faults_i32(uint32_t* count);
cudaError_t take_stage_faults_f16(uint32_t* count);
cudaError_t take_stage_faults_bf16(uint32_t* count);
cudaError_t launch_gather(const GatherParams& p, int elem_bytes, int vb, dim3 grid, cudaStream_t s);
cudaError_t launch_a2av(const A2avParams& p, int vb, int unroll, dim3 grid, cudaStream_t s);
// Claiming launches (counts on the device): blocks per SM, and the launch
// with its dynamic shared memory (the pair counts and tile prefix sums).
int pairs_claim_blocks_per_sm(bool add, int dtype, int vb, int unroll, int nranks);
cudaError_t launch_pairs_claim(const A2avParams& p, bool add, int dtype, int vb, int unroll, int grid,
                               cudaStream_t s);
// The combine with AtomicType kAdd: out += in per element (binary32 for
// floating types, one RNE narrowing; int32 wraps).
cudaError_t launch_pairs_add(const A2avParams& p, int dtype, int vb, dim3 grid, cudaStream_t s);


}  // namespace ptoc
