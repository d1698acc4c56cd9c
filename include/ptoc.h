/*
 * ptoc.h - C ABI of the GB300 tile-level collective library (libptoc.so).
 *
 * The library computes the data-parallel core of the PTO communication ops on
 * N symmetric per-rank window buffers that all live in ONE GPU's memory: the
 * TREDUCE element-wise reduction and the window-layout data movement of
 * reduce_scatter, allgather and all_to_all_v. Sources, cited by page title and
 * section:
 *   [TR] "CANN PTO-ISA TREDUCE 指令详解" (TREDUCE instruction explained,
 *        lpnh.cn news 2291107), sections 1-8.
 *   [DO] "Distributed Operators (N6)" (pypto.ai dev/distributed_ops): the op
 *        table in "Overview", "ABI enums", "Barrier-signal protocol",
 *        "pld.tensor.all_to_all_v", "pld.tensor.allreduce", "pld.tensor.put",
 *        "pld.tile.remote_store".
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer on the calling thread's current
 *     CUDA device, except in ptoc_credit_barrier_host, whose windows and
 *     status are host memory. Pointer arrays (ptoc_group.tensors, send_counts,
 *     recv_counts) are HOST arrays of device pointers; they are read during
 *     the call and copied into kernel parameters, so the caller may free or
 *     reuse them as soon as the call returns.
 *   - The caller owns every buffer. The library keeps no per-call state.
 *     The only memory it takes is the 4-byte work counter of
 *     ptoc_all_to_all_v and ptoc_all_to_all_v_combine: allocated in stream
 *     order on `stream` (from a library-owned pool per device that never
 *     returns its memory; from the default pool during stream capture, where
 *     it becomes a graph memory node), zeroed, and freed in stream order
 *     after the call's kernel. An allocation failure is PTOC_ERR_CUDA.
 *   - Work is enqueued asynchronously on `stream` (0 = the legacy default
 *     stream). Completion is observed through the stream; results must not
 *     be read, and inputs must not be modified, before the stream reaches
 *     them. ptoc_credit_barrier_host, which has no stream, runs on the
 *     calling thread and returns when that rank is done.
 *   - Layout: a "slice" is row-major with a row pitch of `ld` ELEMENTS
 *     (ld >= cols). Element (i, j) is at offset i*ld + j. The footprint the
 *     library may touch is (rows-1)*ld + cols elements from the base pointer.
 *   - Every pointer must be aligned to its element size. Wider alignment
 *     (16 bytes for base pointers and ld*elem_size) selects faster kernels.
 *   - Errors are returned synchronously and NOTHING is launched when a call
 *     returns anything but PTOC_OK. A CUDA launch failure is PTOC_ERR_CUDA.
 *   - Floating point: accumulation in binary32 for f32, f16 and bf16 with one
 *     round-to-nearest-even narrowing per output element; subnormals kept;
 *     Sum adds one rank at a time in the documented rank order (no fused or
 *     reassociated arithmetic). int32 Sum wraps modulo 2^32.
 *   - Per-device state: the library caches, per device ordinal, the SM
 *     count, the counter pool above and the address of the no-allocation
 *     scratch block. They assume the device's primary context lives as long
 *     as the process; after cudaDeviceReset they are stale, so do not call
 *     the library on a device that has been reset.
 *
 * Environment switches (read at every call; results never depend on them)
 *   PTOC_PDL=0           launch the data kernels as ordinary launches. By
 *                        default they are programmatic dependent launches:
 *                        a launch may begin while the previous kernel of the
 *                        stream finishes, and waits for that kernel's
 *                        completion and writes before it touches memory.
 *                        Turning it off gives strict launch boundaries (for
 *                        tools that time or replay kernels one by one).
 *   PTOC_A2AV_UNROLL=4|16
 *                        16-byte chunks per thread in one tile of the
 *                        exchanges' copy kernel (ptoc_all_to_all_v, its
 *                        no-allocation twin, ptoc_all_to_all and the
 *                        PTOC_ATOMIC_NONE combine): 16 or 64 KiB tiles
 *                        instead of the default 32 KiB (8 chunks), for
 *                        16-byte-aligned rows (narrower vectors scale the
 *                        tiles down in proportion). It trades
 *                        scheduling granularity against per-tile overhead;
 *                        any other value means the default.
 *   PTOC_REDUCE_STAGING=bulk|regs|tma
 *                        how the reductions (ptoc_treduce, ptoc_reduce_scatter,
 *                        ptoc_allreduce) over 2 to 8 ranks with 16-byte-aligned
 *                        data load their sources: "bulk" stages each rank's
 *                        4 KiB tile segment in shared memory with the
 *                        bulk-copy (TMA) engine, "regs" loads it into
 *                        registers (same tiles, grid, arithmetic and stores).
 *                        "tma" runs ptoc_treduce through tensor maps over the
 *                        valid box: 2-D boxes of every rank loaded into shared
 *                        memory, the result box stored back by the tensor
 *                        engine, clipped to the valid box; it applies when
 *                        every base pointer, the pitch and a valid row are
 *                        multiples of 16 bytes (else, and for the window
 *                        reductions, the register form runs). Unset (or any
 *                        other value): "bulk" for launches that move at
 *                        least 1.5 GiB (N reads plus the writes), "regs"
 *                        below, the faster form at each size on GB300.
 *                        Results are identical in every form.
 *   PTOC_L2_PREFETCH=0   turn off the first-wave L2 prefetch of the register
 *                        form: by default, in a reduction that moves less than
 *                        512 MiB, each block of the first wave (8 per SM) asks
 *                        L2 for its first tile before it waits for the previous
 *                        kernel of the stream, so that back-to-back calls keep
 *                        DRAM busy across the boundary between them.
 *   PTOC_WAIT_NS=<ns>    the bound on one wait of the staged and tensor forms
 *                        for a copy to land (1 ns to 60 s; default 2 s). A
 *                        block whose wait runs out stores nothing more,
 *                        counts a fault (ptoc_wait_faults), waits (bounded,
 *                        2 s) for its own copies in flight and returns, so
 *                        part of that call's result is missing. Copies of
 *                        valid memory land in microseconds; tiny bounds serve
 *                        to exercise the detection path.
 */
#ifndef PTOC_H
#define PTOC_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest group the library accepts (kernel parameters hold one pointer per
 * rank). */
#define PTOC_MAX_RANKS 64

typedef enum {
    PTOC_OK = 0,
    PTOC_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, misalignment */
    PTOC_ERR_UNSUPPORTED = 2,   /* a valid enum value this library does not implement */
    PTOC_ERR_ALIAS = 3,         /* an output overlaps another operand */
    PTOC_ERR_CUDA = 4           /* the CUDA runtime reported an error at launch */
} ptoc_status;

/* Reduction operators. Values follow the ReduceOp ABI ([TR] §1.3: Sum = 0,
 * Max = 1, Min = 2; [DO] "ABI enums" appends kProd = 3 for the allreduce
 * family). TREDUCE takes Sum, Max and Min only (PTOC_PROD returns
 * PTOC_ERR_UNSUPPORTED there); reduce_scatter and allreduce take all four.
 * Prod multiplies in binary32 one rank at a time (int32 wraps modulo 2^32). */
typedef enum {
    PTOC_SUM = 0,
    PTOC_MAX = 1,
    PTOC_MIN = 2,
    PTOC_PROD = 3
} ptoc_reduce_op;

/* Element types. f16 / bf16 are IEEE binary16 and bfloat16 encodings. */
typedef enum {
    PTOC_F32 = 0,
    PTOC_F16 = 1,
    PTOC_BF16 = 2,
    PTOC_I32 = 3
} ptoc_dtype;

/* Store semantics of a put ([DO] "ABI enums", AtomicType): overwrite the
 * destination, or add into it (a combine, dst += src). */
typedef enum {
    PTOC_ATOMIC_NONE = 0,
    PTOC_ATOMIC_ADD = 1
} ptoc_atomic_type;

/* A rank group ([TR] §2.1, §3.3, §6: ParallelGroup{tensors, nranks, rootIdx}).
 * tensors: host array of nranks device pointers, tensors[r] = rank r's slice.
 * Requires 1 <= nranks <= PTOC_MAX_RANKS; root in [0, nranks) where used. All
 * slices share one shape and row pitch. */
typedef struct {
    void* const* tensors;
    int32_t nranks;
    int32_t root;
} ptoc_group;

/*
 * ptoc_treduce - TREDUCE ([TR] §1.1, §4).
 *   dst[i*ld + j] = (+)_{r} tensors[r][i*ld + j]
 * for i < valid_rows, j < valid_cols, with (+) = op. rows x cols is the
 * physical box of every slice and of dst (valid_rows <= rows,
 * valid_cols <= cols <= ld). Only the valid box is read, and only the valid
 * box of dst is written: padding is never touched ([TR] §3.4, §4.2).
 *
 * Order: the root's element starts the accumulation, then every other rank in
 * ascending order, skipping the root ([TR] §4.3). Max / Min keep the earlier
 * operand on ties (+0 / -0 included) and never let a NaN replace the
 * accumulator; their result is the selected input element, bit for bit.
 * nranks == 1 is a bit copy ([TR] §4.3). An empty valid box returns PTOC_OK
 * and launches nothing ([TR] §4.1).
 *
 * dst may be exactly tensors[root] (in place); any other overlap between dst's
 * valid footprint and a source's is PTOC_ERR_ALIAS. Sources may alias each
 * other.
 */
ptoc_status ptoc_treduce(const ptoc_group* group, void* dst,
                         int64_t rows, int64_t cols,
                         int64_t valid_rows, int64_t valid_cols, int64_t ld,
                         ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_reduce_scatter - reduce_scatter over N windows, in place ([DO] op
 * table: "reduce and scatter chunks across ranks"; the result is the window).
 * Window r's row chunk [floor(r*rows/N), floor((r+1)*rows/N)) (the balanced
 * segment bounds of [DO] "pld.tensor.allreduce", ring mode, applied to rows)
 * becomes the reduction over all windows of the same rows, columns
 * [0, cols), in rank order 0..N-1, binary32 accumulation. Every other element
 * of every window is left unchanged. windows->root is ignored. op: Sum, Max,
 * Min or Prod. Windows must not overlap one another (PTOC_ERR_ALIAS).
 */
ptoc_status ptoc_reduce_scatter(const ptoc_group* windows,
                                int64_t rows, int64_t cols, int64_t ld,
                                ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_allgather - allgather over N windows, in place ([DO] op table: "gather
 * data from all ranks via window"). Row chunk r (bounds as in
 * ptoc_reduce_scatter) of window r is copied bit for bit into row chunk r of
 * every other window, columns [0, cols). Called after ptoc_reduce_scatter
 * with the same arguments it leaves every window equal to the full reduction.
 * windows->root is ignored. Windows must not overlap (PTOC_ERR_ALIAS).
 */
ptoc_status ptoc_allgather(const ptoc_group* windows,
                           int64_t rows, int64_t cols, int64_t ld,
                           ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_allreduce - allreduce over N windows, in place ([DO]
 * "pld.tensor.allreduce": every participating rank's window slice is reduced
 * in place; Sum, Max, Min, Prod). Every window's [rows, cols] box becomes the
 * same value: the reduction over all windows in rank order 0..N-1 with binary32
 * accumulation, bit-identical to ptoc_reduce_scatter followed by
 * ptoc_allgather with the same arguments, done in one pass (each element is
 * read once from every window and written once to every window). Columns
 * [cols, ld) are untouched. windows->root is ignored. Windows must not overlap
 * (PTOC_ERR_ALIAS).
 */
ptoc_status ptoc_allreduce(const ptoc_group* windows,
                           int64_t rows, int64_t cols, int64_t ld,
                           ptoc_reduce_op op, ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_broadcast - broadcast into N windows, in place ([DO] op table:
 * "replicate root rank's data to all ranks"; the result is the window). The
 * [rows, cols] box of window windows->root is copied bit for bit into every
 * other window. Requires root in [0, N). Windows must not overlap
 * (PTOC_ERR_ALIAS).
 */
ptoc_status ptoc_broadcast(const ptoc_group* windows,
                           int64_t rows, int64_t cols, int64_t ld,
                           ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_all_to_all_v - variable-size all-to-all into flat staging windows
 * ([DO] "pld.tensor.all_to_all_v").
 *   inputs->tensors[s]  : rank s's packed input  [target_rows, size] (read)
 *   targets->tensors[d] : rank d's packed window [target_rows, size] (written)
 *   send_counts[s]      : host array of N device pointers, each int32[N]:
 *                         rows rank s sends to each destination (read)
 *   recv_counts[d]      : host array of N device pointers, each int32[N]
 *                         (the [NR, 1] column): written with the counts rank d
 *                         receives from each source.
 * With MAX_RECV = target_rows / N (floor), for every pair (s, d), s == d
 * included:
 *   c = clamp(send_counts[s][d], 0, MAX_RECV)            (two-sided clamp)
 *   recv_counts[d][s] = c
 *   targets[d] rows [s*MAX_RECV, s*MAX_RECV + c) = inputs[s] rows
 *                   [d*MAX_RECV, d*MAX_RECV + c)
 * Target rows outside the counts are never written. Counts live on the
 * device and are clamped there: out-of-range counts are not errors. The data
 * is moved bit for bit; dtype only fixes the element size.
 * inputs->nranks must equal targets->nranks; roots are ignored. Outputs
 * (targets, recv_counts) must not overlap each other or any input
 * (PTOC_ERR_ALIAS); inputs and send_counts may overlap one another.
 * The counts are read on the device, so the work is scheduled there: one
 * wave of blocks takes the moved tiles in order from a zeroed 4-byte counter
 * (see the conventions above), and a sparse exchange costs in proportion to
 * the rows it moves, not to the capacity of the windows. A call whose
 * windows would hold 2^31 or more tiles (32 KiB each for 16-byte-aligned
 * rows, less for narrower alignment) returns PTOC_ERR_UNSUPPORTED.
 */
ptoc_status ptoc_all_to_all_v(const ptoc_group* inputs, const ptoc_group* targets,
                              const int32_t* const* send_counts, int32_t* const* recv_counts,
                              int64_t target_rows, int64_t size, ptoc_dtype dtype,
                              cudaStream_t stream);

/*
 * ptoc_all_to_all_v_noalloc - ptoc_all_to_all_v without any allocation. The
 * pages have no counterpart of this entry point: it serves callers that may
 * not allocate during a call, at the price of one exchange in flight at a time.
 * Arguments, results, checks and errors are those of ptoc_all_to_all_v. Its
 * only scratch is a 4-byte tile counter taken from a fixed 256-byte block of
 * device memory inside the library (its address is looked up once per device).
 * Each call zeroes the counter with a stream-ordered memset; no call allocates
 * or frees memory. A call whose scratch would not fit in the block returns
 * PTOC_ERR_UNSUPPORTED (the counter always fits).
 * Calls whose kernels can overlap (on different streams, from different
 * threads, or through graph replays) share the counter and RACE: their
 * results are undefined. Serialize them, for instance on one stream.
 */
ptoc_status ptoc_all_to_all_v_noalloc(const ptoc_group* inputs, const ptoc_group* targets,
                                      const int32_t* const* send_counts, int32_t* const* recv_counts,
                                      int64_t target_rows, int64_t size, ptoc_dtype dtype,
                                      cudaStream_t stream);

/*
 * ptoc_all_to_all - symmetric all-to-all ([DO] op table: every rank pushes
 * its per-destination chunks to every peer's window; the window is the
 * result). Layout as ptoc_all_to_all_v with C = target_rows / N rows per
 * chunk: targets[d] rows [s*C, (s+1)*C) = inputs[s] rows [d*C, (d+1)*C) for
 * every (s, d). Rows at and past N*C are not written. Alias rules as
 * ptoc_all_to_all_v (targets must not overlap inputs or each other).
 */
ptoc_status ptoc_all_to_all(const ptoc_group* inputs, const ptoc_group* targets,
                            int64_t target_rows, int64_t size, ptoc_dtype dtype,
                            cudaStream_t stream);

/*
 * ptoc_all_to_all_v_combine - the return leg of ptoc_all_to_all_v: a put from
 * every rank d to every peer s ([DO] "pld.tensor.put", "pld.tile.remote_store":
 * AtomicType kAdd makes the push a combine, peer_region += src, what an
 * all-to-all combine needs).
 *   windows->tensors[d] : rank d's window [target_rows, size] holding the rows
 *                         it received (read)
 *   outputs->tensors[s] : rank s's output [target_rows, size] (written)
 *   recv_counts[d]      : host array of N device pointers, each int32[N]: the
 *                         rows rank d holds from each source (read; typically
 *                         the counts ptoc_all_to_all_v published)
 * With MAX_RECV = target_rows / N and c = clamp(recv_counts[d][s], 0,
 * MAX_RECV): outputs[s] rows [d*MAX_RECV, d*MAX_RECV + c) receive windows[d]
 * rows [s*MAX_RECV, s*MAX_RECV + c); PTOC_ATOMIC_NONE overwrites bit for bit,
 * PTOC_ATOMIC_ADD adds (binary32 add and one RNE narrowing per element for
 * floating types, wrapping for int32). Every output row has at most one
 * contributor, so the result does not depend on scheduling. Other output rows
 * are not written. Outputs must not overlap each other, the windows or the
 * counts (PTOC_ERR_ALIAS). Scheduled like ptoc_all_to_all_v (a 4-byte
 * work counter per call).
 */
ptoc_status ptoc_all_to_all_v_combine(const ptoc_group* windows, const ptoc_group* outputs,
                                      const int32_t* const* recv_counts,
                                      int64_t target_rows, int64_t size, ptoc_atomic_type atomic,
                                      ptoc_dtype dtype, cudaStream_t stream);

/*
 * ptoc_credit_barrier - the self-clearing credit barrier ([DO]
 * "Barrier-signal protocol") among ranks simulated on this GPU.
 *   signals->tensors[p] : rank p's signal window, N device int32 cells; cell s
 *                         counts the credits rank s has given rank p. All
 *                         cells must be zero when a call starts (they are
 *                         zero again after every complete call).
 *   local_ranks         : host array of the n_local distinct ranks that take
 *                         part in this launch (1 <= n_local <= N).
 *   status              : device int32[n_local]; status[i] = 0 if
 *                         local_ranks[i] completed, or g if it gave up
 *                         waiting in generation g.
 * For g = 1..generations every rank adds 1 (atomic, release) to its cell in
 * every peer's window and waits (acquire) until every cell of its own window
 * is >= g (Ge, not Eq: a fast peer may already be ahead); then it subtracts
 * `generations` from its own cells. All local ranks run in one cooperative
 * launch (one warp each). A rank that is not local never arrives, so the
 * others give up after timeout_ns nanoseconds (0 < timeout_ns <= 60 s) and
 * skip their epilogue, leaving credits in the windows, as the page describes
 * for an aborted call: clear them with ptoc_signal_reset before reuse.
 * Errors: invalid arguments, overlapping windows or status
 * (PTOC_ERR_ALIAS), no cooperative-launch support (PTOC_ERR_UNSUPPORTED).
 */
ptoc_status ptoc_credit_barrier(const ptoc_group* signals, const int32_t* local_ranks, int32_t n_local,
                                int32_t generations, int64_t timeout_ns, int32_t* status,
                                cudaStream_t stream);

/*
 * ptoc_credit_barrier_host - the same credit barrier ([DO] "Barrier-signal
 * protocol") for ranks that are host threads or host processes. The calling
 * thread runs rank `rank`'s part of one call; every rank that takes part
 * calls it once, with the same windows and `generations`.
 *   signals->tensors[p] : HOST pointer to rank p's window of N int32 cells
 *                         (memory every participant addresses: the memory
 *                         of one process shared by its threads, or a mapping
 *                         shared between processes). Cells are updated with
 *                         lock-free 32-bit atomics; all must be zero when a
 *                         call starts and are zero again after a complete
 *                         call. signals->root is ignored.
 *   status              : host int32; 0 if the rank completed, or g if it
 *                         gave up waiting in generation g.
 * Same steps as ptoc_credit_barrier (release adds, acquire waits for >= g,
 * the epilogue subtracts `generations`). A rank that never calls never
 * arrives: the others give up after timeout_ns (0 < timeout_ns <= 60 s, on
 * the steady clock) and leave their credits, so zero the windows before the
 * next call. Blocks the calling thread; makes no CUDA call and needs no GPU.
 * Errors: invalid arguments (rank outside [0, N), null or misaligned
 * pointers, sizes), overlapping windows or status (PTOC_ERR_ALIAS).
 */
ptoc_status ptoc_credit_barrier_host(const ptoc_group* signals, int32_t rank, int32_t generations,
                                     int64_t timeout_ns, int32_t* status);

/*
 * ptoc_signal_reset - zero every cell of every signal window on `stream`
 * (the host-side reset the page prescribes after an aborted call).
 */
ptoc_status ptoc_signal_reset(const ptoc_group* signals, cudaStream_t stream);

/*
 * ptoc_wait_faults - failure detection for the waits inside the library's
 * kernels (no counterpart in the pages). Every wait of the staged and tensor
 * reduction forms on a copy is bounded (2 s, or PTOC_WAIT_NS); a block whose
 * wait gives up stores nothing more and counts one fault on its device. *count receives the faults counted
 * on the current device since the previous call, and the count restarts at
 * zero. 0 means every staged tile of every earlier call was stored. The
 * read is a synchronous copy on the legacy default stream: call it when the
 * device is idle (after cudaDeviceSynchronize) to include every earlier call.
 * The credit barrier reports its own waits through its status array.
 */
ptoc_status ptoc_wait_faults(uint32_t* count);

/* A static, human-readable name for a status code. */
const char* ptoc_status_string(ptoc_status status);

#ifdef __cplusplus
}
#endif

#endif /* PTOC_H */
