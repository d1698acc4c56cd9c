/*
 * Oracle for the TREDUCE / window-collective hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU
 * restatement of what the operations compute. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference leg may load it; the
 * product (the CUDA library) never does, and the two share no code: no
 * header, helper, table or constant of the CUDA library is used here.
 *
 * Sources (cited by page title and section):
 *   [TR]  "CANN PTO-ISA TREDUCE 指令详解" (TREDUCE instruction explained,
 *         lpnh.cn news 2291107), sections 1 to 8 (一..八).
 *   [DO]  "Distributed Operators (N6)", pypto.ai dev/distributed_ops:
 *         the op table (Overview), "ABI enums", "Barrier-signal protocol",
 *         "pld.tensor.all_to_all_v", "pld.tensor.allreduce",
 *         "pld.tensor.put", "pld.tile.remote_store".
 *
 * Readings taken where the pages are silent or garbled are stated beside the
 * code that takes them. Every function here is pinned by tests that do not
 * call back into this file for the expected values (closed forms, brute
 * force, library conversions, hand-worked examples).
 *
 * Floating point: compiled with -ffp-contract=off and without fast-math, so
 * each `+` below is one IEEE-754 binary32 addition in the order written.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ReduceOp values: [TR] §1.3 (Sum = 0, Max = 1, Min = 2); [DO] "ABI enums"
 * appends kProd = 3 for the allreduce family. */
enum { ORC_SUM = 0, ORC_MAX = 1, ORC_MIN = 2, ORC_PROD = 3 };
/* AtomicType values ([DO] "ABI enums"): plain store, or add into the
 * destination. */
enum { ORC_ATOMIC_NONE = 0, ORC_ATOMIC_ADD = 1 };
/* Element types the oracle accepts (its own numbering, passed by the tests). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_I32 = 3 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1 };

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

static size_t elem_bytes(int dtype)
{
    switch (dtype) {
    case ORC_F32: case ORC_I32: return 4;
    case ORC_F16: case ORC_BF16: return 2;
    default: return 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Conversions, from the IEEE-754 encodings.                                 */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of a binary32 encoding: widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/*
 * binary32 -> bfloat16, round to nearest, ties to even. Keep the upper 16
 * bits; look at the 16 dropped bits: above half an ulp rounds up, exactly half
 * rounds up only if the kept value is odd. Adding 1 to the kept encoding
 * carries from the mantissa into the exponent, which is the correct next
 * representable value (and turns the largest finite value into infinity).
 * NaN keeps its sign and top payload bits and is made quiet.
 */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u = f32_bits(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

/* binary16 -> binary32 (exact): value = (-1)^s * m * 2^-24 for subnormals,
 * (-1)^s * (1024 + m) * 2^(e - 25) for normals. NaN payloads are not kept. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);
    return sign ? -v : v;
}

/*
 * binary32 -> binary16, round to nearest, ties to even, subnormals kept.
 * A finite binary32 is S * 2^(e-23) with S in [2^23, 2^24). The binary16
 * result is an integer multiple M of its quantum q: q = 2^(e-10) when the
 * value is in the normal range (e >= -14), q = 2^-24 below it. So
 * M = S / 2^shift with shift = 13 (normal) or -1 - e (subnormal), rounded
 * to nearest even on the dropped bits.
 */
uint16_t oracle_f32_to_f16(float x)
{
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    int32_t E = (int32_t)(a >> 23);
    uint32_t frac = a & 0x007FFFFFu;
    if (E == 255)
        return (uint16_t)(sign | (frac ? 0x7E00u : 0x7C00u));
    if (E == 0)                      /* |x| < 2^-126: rounds to zero */
        return sign;
    int32_t e = E - 127;
    if (e > 15)                      /* |x| >= 2^16: overflow */
        return (uint16_t)(sign | 0x7C00u);
    uint32_t S = frac | 0x00800000u;
    int shift = (e >= -14) ? 13 : (-1 - e);
    if (shift > 24)                  /* below half of the smallest subnormal */
        return sign;
    uint32_t M = S >> shift;
    uint32_t rem = S & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (M & 1u)))
        M += 1u;
    uint32_t bits;
    if (e >= -14)                    /* M in [1024, 2048]; 2048 carries into the exponent */
        bits = ((uint32_t)(e + 15) << 10) + (M - 1024u);
    else                             /* subnormal; M == 1024 encodes the smallest normal */
        bits = M;
    if (bits >= 0x7C00u)             /* rounded past 65504 */
        bits = 0x7C00u;
    return (uint16_t)(sign | bits);
}

/* Array forms, for the exhaustive conversion checks. */
void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}
void oracle_f32_to_f16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_f16(x[i]);
}
void oracle_f16_to_f32_array(const uint16_t* x, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f16_to_f32(x[i]);
}
void oracle_bf16_to_f32_array(const uint16_t* x, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_to_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* TREDUCE                                                                   */
/* ------------------------------------------------------------------------ */

/* W(): widen a floating element to binary32 (exact for all three types). */
static float widen(int dtype, const void* base, int64_t k)
{
    if (dtype == ORC_F32) return ((const float*)base)[k];
    if (dtype == ORC_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[k]);
    return oracle_f16_to_f32(((const uint16_t*)base)[k]);
}

/* N(): narrow the binary32 accumulator to the destination type (RNE). */
static void narrow_store(int dtype, void* base, int64_t k, float acc)
{
    if (dtype == ORC_F32) ((float*)base)[k] = acc;
    else if (dtype == ORC_BF16) ((uint16_t*)base)[k] = oracle_f32_to_bf16(acc);
    else ((uint16_t*)base)[k] = oracle_f32_to_f16(acc);
}

/*
 * The rank order of the reduction ([TR] §4.3): the root's element is loaded
 * into the accumulator first, then every other rank in ascending order,
 * skipping the root. order[0] = root, order[1..N-1] = the rest ascending.
 */
static void rank_order(int nranks, int root, int* order)
{
    int n = 0;
    order[n++] = root;
    for (int r = 0; r < nranks; ++r)
        if (r != root) order[n++] = r;
}

/* One output element (row-major offset k) of TREDUCE. */
static void treduce_element(const void* const* src, const int* order, int nranks,
                            void* dst, int64_t k, int op, int dtype)
{
    size_t b = elem_bytes(dtype);

    /* nranks == 1: a plain copy of the root's element ([TR] §4.3). */
    if (nranks == 1) {
        memcpy((char*)dst + k * b, (const char*)src[order[0]] + k * b, b);
        return;
    }

    if (dtype == ORC_I32) {
        /* int32: Sum wraps modulo 2^32 (reading: the pages are silent), so it
         * is computed in uint32; Max and Min compare as signed int32. */
        int32_t acc = ((const int32_t*)src[order[0]])[k];
        for (int t = 1; t < nranks; ++t) {
            int32_t x = ((const int32_t*)src[order[t]])[k];
            if (op == ORC_SUM) acc = (int32_t)((uint32_t)acc + (uint32_t)x);
            else if (op == ORC_PROD) acc = (int32_t)((uint32_t)acc * (uint32_t)x);   /* wraps too */
            else if (op == ORC_MAX) acc = (x > acc) ? x : acc;
            else acc = (x < acc) ? x : acc;
        }
        ((int32_t*)dst)[k] = acc;
        return;
    }

    if (op == ORC_SUM || op == ORC_PROD) {
        /* acc = W(root); acc = acc + W(src_r) (or acc * W(src_r)) for the rest
         * in order; one RNE narrowing at the end. Accumulation in binary32 for
         * every floating type (reading: the pages make the accumulator tile the
         * destination type; the fp32 accumulator is the library's stated
         * contract). */
        float acc = widen(dtype, src[order[0]], k);
        for (int t = 1; t < nranks; ++t) {
            if (op == ORC_SUM) acc = acc + widen(dtype, src[order[t]], k);
            else acc = acc * widen(dtype, src[order[t]], k);
        }
        narrow_store(dtype, dst, k, acc);
        return;
    }

    /* Max / Min ([TR] §1.3, TMAX / TMIN; tie and NaN rules are a reading):
     * x replaces the accumulator only if strictly greater (smaller). Equal
     * values, +0 against -0 included, keep the earlier operand; a NaN x never
     * replaces; a NaN root stays. The result is the selected operand itself,
     * bit for bit. */
    int sel = order[0];
    float acc = widen(dtype, src[sel], k);
    for (int t = 1; t < nranks; ++t) {
        float x = widen(dtype, src[order[t]], k);
        if ((op == ORC_MAX && x > acc) || (op == ORC_MIN && x < acc)) {
            acc = x;
            sel = order[t];
        }
    }
    memcpy((char*)dst + k * b, (const char*)src[sel] + k * b, b);
}

/*
 * TREDUCE ([TR] §1.1): dst[i,j] = (+)_{r} src^(r)[i,j] over the valid region
 * i < valid_rows, j < valid_cols. Every slice and dst share one row pitch `ld`
 * (elements) ([TR] §3.3: all tensors share shape and strides). Nothing outside
 * the valid region is written. An empty region returns at once without writing
 * ([TR] §4.1, §7.2).
 */
int oracle_treduce(const void* const* src, int nranks, int root, void* dst,
                   int64_t valid_rows, int64_t valid_cols, int64_t ld, int op, int dtype)
{
    if (nranks <= 0 || root < 0 || root >= nranks) return ORC_BAD_ARG;   /* [TR] §3.3 */
    if (op != ORC_SUM && op != ORC_MAX && op != ORC_MIN && op != ORC_PROD) return ORC_BAD_ARG;
    if (elem_bytes(dtype) == 0) return ORC_BAD_ARG;
    if (valid_rows < 0 || valid_cols < 0 || (valid_cols > ld && valid_rows > 0)) return ORC_BAD_ARG;
    if (valid_rows == 0 || valid_cols == 0) return ORC_OK;

    int* order = (int*)malloc(sizeof(int) * (size_t)nranks);
    if (!order) return ORC_BAD_ARG;
    rank_order(nranks, root, order);
    for (int64_t i = 0; i < valid_rows; ++i)
        for (int64_t j = 0; j < valid_cols; ++j)
            treduce_element(src, order, nranks, dst, i * ld + j, op, dtype);
    free(order);
    return ORC_OK;
}

/*
 * TREDUCE Sum under the other reading of the accumulator's precision: [TR]
 * §3.1 declares the accumulator tile with the destination's element type, so
 * every partial sum is rounded (RNE) to that type before the next rank is
 * added. Ranks in the same order as oracle_treduce. For f32 the two readings
 * coincide; Max and Min select an operand and are not affected. This is test
 * infrastructure that measures what the binary32 accumulator changes; the
 * library implements only the binary32 accumulator.
 */
int oracle_treduce_sum_native_acc(const void* const* src, int nranks, int root, void* dst,
                                  int64_t valid_rows, int64_t valid_cols, int64_t ld, int dtype)
{
    if (nranks <= 0 || root < 0 || root >= nranks) return ORC_BAD_ARG;
    if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16) return ORC_BAD_ARG;
    if (valid_rows < 0 || valid_cols < 0 || (valid_cols > ld && valid_rows > 0)) return ORC_BAD_ARG;
    if (valid_rows == 0 || valid_cols == 0) return ORC_OK;

    int* order = (int*)malloc(sizeof(int) * (size_t)nranks);
    if (!order) return ORC_BAD_ARG;
    rank_order(nranks, root, order);
    for (int64_t i = 0; i < valid_rows; ++i)
        for (int64_t j = 0; j < valid_cols; ++j) {
            const int64_t k = i * ld + j;
            float acc = widen(dtype, src[order[0]], k);
            for (int t = 1; t < nranks; ++t) {
                const float sum = acc + widen(dtype, src[order[t]], k);
                /* the accumulator tile holds the destination type */
                if (dtype == ORC_BF16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(sum));
                else if (dtype == ORC_F16) acc = oracle_f16_to_f32(oracle_f32_to_f16(sum));
                else acc = sum;
            }
            narrow_store(dtype, dst, k, acc);
        }
    free(order);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* reduce_scatter and allgather over N windows                               */
/* ------------------------------------------------------------------------ */

/* Row chunk of rank r: [floor(r*rows/N), floor((r+1)*rows/N)). Reading: the
 * pages give the balanced floor(i*SIZE/NR) segment bounds for the fp32 ring
 * ([DO] pld.tensor.allreduce, "ring"); applied to rows here. */
static int64_t chunk_lo(int64_t r, int64_t rows, int64_t nranks) { return (r * rows) / nranks; }

/*
 * reduce_scatter ([DO] op table: "reduce and scatter chunks across ranks",
 * result is the window itself): window r's rows in chunk r become the
 * reduction, over every window in rank order 0..N-1, of those same rows. The
 * other rows of window r are left as they were. Computed from a snapshot of
 * all windows taken before any write.
 */
int oracle_reduce_scatter(void* const* win, int nranks, int64_t rows, int64_t cols,
                          int64_t ld, int op, int dtype)
{
    if (nranks <= 0 || rows < 0 || cols < 0 || (cols > ld && rows > 0)) return ORC_BAD_ARG;
    size_t b = elem_bytes(dtype);
    if (b == 0 || (op != ORC_SUM && op != ORC_MAX && op != ORC_MIN && op != ORC_PROD)) return ORC_BAD_ARG;
    if (rows == 0 || cols == 0) return ORC_OK;

    size_t footprint = (size_t)((rows - 1) * ld + cols) * b;
    void** snap = (void**)malloc(sizeof(void*) * (size_t)nranks);
    for (int r = 0; r < nranks; ++r) {
        snap[r] = malloc(footprint);
        memcpy(snap[r], win[r], footprint);
    }
    for (int r = 0; r < nranks; ++r) {
        int64_t lo = chunk_lo(r, rows, nranks), hi = chunk_lo(r + 1, rows, nranks);
        if (hi <= lo) continue;
        const void** src = (const void**)malloc(sizeof(void*) * (size_t)nranks);
        for (int s = 0; s < nranks; ++s) src[s] = (const char*)snap[s] + (size_t)(lo * ld) * b;
        oracle_treduce(src, nranks, 0, (char*)win[r] + (size_t)(lo * ld) * b,
                       hi - lo, cols, ld, op, dtype);
        free(src);
    }
    for (int r = 0; r < nranks; ++r) free(snap[r]);
    free(snap);
    return ORC_OK;
}

/*
 * allgather ([DO] op table: "gather data from all ranks via window"): chunk r
 * of window r is copied, bit for bit, into chunk r of every other window.
 */
int oracle_allgather(void* const* win, int nranks, int64_t rows, int64_t cols,
                     int64_t ld, int dtype)
{
    if (nranks <= 0 || rows < 0 || cols < 0 || (cols > ld && rows > 0)) return ORC_BAD_ARG;
    size_t b = elem_bytes(dtype);
    if (b == 0) return ORC_BAD_ARG;
    for (int r = 0; r < nranks; ++r) {
        int64_t lo = chunk_lo(r, rows, nranks), hi = chunk_lo(r + 1, rows, nranks);
        for (int s = 0; s < nranks; ++s) {
            if (s == r) continue;
            for (int64_t i = lo; i < hi; ++i)
                memcpy((char*)win[s] + (size_t)(i * ld) * b,
                       (const char*)win[r] + (size_t)(i * ld) * b, (size_t)cols * b);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* all_to_all_v                                                              */
/* ------------------------------------------------------------------------ */

/*
 * all_to_all_v ([DO] pld.tensor.all_to_all_v): every rank s holds a packed
 * input [N*MAX_RECV, size] and a target window of the same shape, with
 * MAX_RECV = target_rows // N. For every (s, d), self included:
 *   c = clamp(send_counts_s[d], 0, MAX_RECV)           (two-sided clamp)
 *   recv_counts_d[s] = c                                 (published count)
 *   target_d rows [s*MAX_RECV, s*MAX_RECV + c) = input_s rows [d*MAX_RECV, ...)
 * Target rows beyond the count are never written.
 * Reading: input block d starts at row d*MAX_RECV and the receiver's capacity
 * slot for sender s starts at row s*MAX_RECV (the page fixes the flat
 * [NR*MAX_RECV, SIZE] shapes but not the displacements).
 */
int oracle_all_to_all_v(const void* const* inputs, void* const* targets,
                        const int32_t* const* send_counts, int32_t* const* recv_counts,
                        int nranks, int64_t target_rows, int64_t size, int elem_size)
{
    if (nranks <= 0 || target_rows < 0 || size < 0 || elem_size <= 0) return ORC_BAD_ARG;
    int64_t max_recv = target_rows / nranks;
    size_t row_bytes = (size_t)size * (size_t)elem_size;
    for (int s = 0; s < nranks; ++s) {
        for (int d = 0; d < nranks; ++d) {
            int64_t c = send_counts[s][d];
            if (c < 0) c = 0;
            if (c > max_recv) c = max_recv;
            recv_counts[d][s] = (int32_t)c;
            for (int64_t i = 0; i < c; ++i)
                memcpy((char*)targets[d] + (size_t)(s * max_recv + i) * row_bytes,
                       (const char*)inputs[s] + (size_t)(d * max_recv + i) * row_bytes,
                       row_bytes);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* allreduce, broadcast, symmetric all_to_all                                */
/* ------------------------------------------------------------------------ */

/*
 * allreduce ([DO] "pld.tensor.allreduce": every participating rank's window
 * slice is reduced in place; Sum, Max, Min and Prod). Reading: every window's
 * [rows, cols] box becomes the same value, the reduction over all windows in
 * rank order 0..N-1 (what reduce_scatter followed by allgather produces), so
 * the ranks agree bit for bit. Computed from a snapshot taken before any write.
 */
int oracle_allreduce(void* const* win, int nranks, int64_t rows, int64_t cols,
                     int64_t ld, int op, int dtype)
{
    if (nranks <= 0 || rows < 0 || cols < 0 || (cols > ld && rows > 0)) return ORC_BAD_ARG;
    size_t b = elem_bytes(dtype);
    if (b == 0 || (op != ORC_SUM && op != ORC_MAX && op != ORC_MIN && op != ORC_PROD)) return ORC_BAD_ARG;
    if (rows == 0 || cols == 0) return ORC_OK;
    size_t footprint = (size_t)((rows - 1) * ld + cols) * b;
    void** snap = (void**)malloc(sizeof(void*) * (size_t)nranks);
    for (int r = 0; r < nranks; ++r) {
        snap[r] = malloc(footprint);
        memcpy(snap[r], win[r], footprint);
    }
    for (int r = 0; r < nranks; ++r)
        oracle_treduce((const void* const*)snap, nranks, 0, win[r], rows, cols, ld, op, dtype);
    for (int r = 0; r < nranks; ++r) free(snap[r]);
    free(snap);
    return ORC_OK;
}

/*
 * broadcast ([DO] op table: "replicate root rank's data to all ranks", the
 * result is the window): every other window's [rows, cols] box becomes the
 * root's, bit for bit.
 */
int oracle_broadcast(void* const* win, int nranks, int root, int64_t rows, int64_t cols,
                     int64_t ld, int dtype)
{
    if (nranks <= 0 || root < 0 || root >= nranks || rows < 0 || cols < 0 || (cols > ld && rows > 0))
        return ORC_BAD_ARG;
    size_t b = elem_bytes(dtype);
    if (b == 0) return ORC_BAD_ARG;
    for (int s = 0; s < nranks; ++s) {
        if (s == root) continue;
        for (int64_t i = 0; i < rows; ++i)
            memcpy((char*)win[s] + (size_t)(i * ld) * b, (const char*)win[root] + (size_t)(i * ld) * b,
                   (size_t)cols * b);
    }
    return ORC_OK;
}

/*
 * symmetric all_to_all ([DO] op table: every rank pushes its per-destination
 * chunks to every peer's window). With C = target_rows / N rows per chunk:
 *   target_d rows [s*C, (s+1)*C) = input_s rows [d*C, (d+1)*C)
 * for every (s, d), s == d included; rows at and past N*C are not written.
 */
int oracle_all_to_all(const void* const* inputs, void* const* targets, int nranks,
                      int64_t target_rows, int64_t size, int elem_size)
{
    if (nranks <= 0 || target_rows < 0 || size < 0 || elem_size <= 0) return ORC_BAD_ARG;
    int64_t chunk = target_rows / nranks;
    size_t row_bytes = (size_t)size * (size_t)elem_size;
    for (int s = 0; s < nranks; ++s)
        for (int d = 0; d < nranks; ++d)
            for (int64_t i = 0; i < chunk; ++i)
                memcpy((char*)targets[d] + (size_t)(s * chunk + i) * row_bytes,
                       (const char*)inputs[s] + (size_t)(d * chunk + i) * row_bytes, row_bytes);
    return ORC_OK;
}

/*
 * all_to_all_v combine: the return leg of all_to_all_v, a put from every
 * rank d to every peer s ([DO] "pld.tensor.put" and "pld.tile.remote_store":
 * atomic = kAdd makes the push a combine, peer_region += src, "what an
 * all-to-all combine needs"). With MAX_RECV = target_rows / N and
 * c = clamp(recv_counts_d[s], 0, MAX_RECV), the c rows rank d received from s
 * (its window rows [s*MAX_RECV, s*MAX_RECV + c)) go back to rank s's output
 * rows [d*MAX_RECV, d*MAX_RECV + c):
 *   kNone: output_s row = window_d row, bit for bit;
 *   kAdd:  output_s element = N(W(output_s element) + W(window_d element))
 *          (binary32 add, one RNE narrowing; int32 wraps).
 * Every output row has at most one contributor, so the result does not depend
 * on the order of the pushes. Rows outside the counts are not written.
 */
int oracle_all_to_all_v_combine(const void* const* windows, void* const* outputs,
                                const int32_t* const* recv_counts, int nranks,
                                int64_t target_rows, int64_t size, int atomic, int dtype)
{
    if (nranks <= 0 || target_rows < 0 || size < 0) return ORC_BAD_ARG;
    size_t b = elem_bytes(dtype);
    if (b == 0 || (atomic != ORC_ATOMIC_NONE && atomic != ORC_ATOMIC_ADD)) return ORC_BAD_ARG;
    int64_t max_recv = target_rows / nranks;
    for (int d = 0; d < nranks; ++d) {
        for (int s = 0; s < nranks; ++s) {
            int64_t c = recv_counts[d][s];
            if (c < 0) c = 0;
            if (c > max_recv) c = max_recv;
            for (int64_t i = 0; i < c; ++i) {
                const char* src = (const char*)windows[d] + (size_t)((s * max_recv + i) * size) * b;
                char* dst = (char*)outputs[s] + (size_t)((d * max_recv + i) * size) * b;
                if (atomic == ORC_ATOMIC_NONE) {
                    memcpy(dst, src, (size_t)size * b);
                    continue;
                }
                for (int64_t j = 0; j < size; ++j) {
                    if (dtype == ORC_I32) {
                        ((int32_t*)dst)[j] = (int32_t)((uint32_t)((int32_t*)dst)[j] +
                                                       (uint32_t)((const int32_t*)src)[j]);
                    } else {
                        float acc = widen(dtype, dst, j) + widen(dtype, src, j);
                        narrow_store(dtype, dst, j, acc);
                    }
                }
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Credit barrier                                                            */
/* ------------------------------------------------------------------------ */

/*
 * The self-clearing credit barrier ([DO] "Barrier-signal protocol"), run by a
 * deterministic scheduler. Rank r's signal window holds one cell per source
 * rank: signal[r * N + s]. A call of G generations is, for each rank r:
 *   for g = 1..G:   notify every peer p != r: signal[p*N + r] += 1   (AtomicAdd)
 *                   wait until signal[r*N + s] >= g for every s != r (Ge)
 *   epilogue:       signal[r*N + s] -= G for every s != r            (AtomicAdd)
 * present[r] = 0 models a rank that never arrives. The scheduler visits the
 * present ranks in ascending order, letting each run until it blocks, and
 * repeats until a full pass makes no progress; ranks still blocked then time
 * out. status[r]: 0 = completed, g = timed out waiting in generation g,
 * -1 = not present. `wait_eq` = 1 replaces the Ge comparison by Eq (the page
 * explains why that can hang); it exists to demonstrate that point.
 * The final signal is written back in place.
 */
int oracle_credit_barrier(int nranks, int generations, const int32_t* present, int32_t* signal,
                          int32_t* status, int wait_eq)
{
    if (nranks <= 0 || generations < 0) return ORC_BAD_ARG;
    int N = nranks;
    int* gen = (int*)calloc((size_t)N, sizeof(int));       /* current generation, 1-based */
    int* notified = (int*)calloc((size_t)N, sizeof(int));  /* notified in `gen` already */
    int* done = (int*)calloc((size_t)N, sizeof(int));
    for (int r = 0; r < N; ++r) {
        gen[r] = 1;
        status[r] = present[r] ? 0 : -1;
        done[r] = present[r] ? 0 : 1;
    }
    int progress = 1;
    while (progress) {
        progress = 0;
        for (int r = 0; r < N; ++r) {
            while (!done[r]) {
                if (gen[r] > generations) {                 /* epilogue */
                    for (int s = 0; s < N; ++s)
                        if (s != r) signal[r * N + s] -= generations;
                    done[r] = 1;
                    progress = 1;
                    break;
                }
                if (!notified[r]) {
                    for (int p = 0; p < N; ++p)
                        if (p != r) signal[p * N + r] += 1;
                    notified[r] = 1;
                    progress = 1;
                }
                int ready = 1;
                for (int s = 0; s < N; ++s) {
                    if (s == r) continue;
                    int v = signal[r * N + s];
                    if (wait_eq ? (v != gen[r]) : (v < gen[r])) ready = 0;
                }
                if (!ready) break;                          /* blocked: next rank */
                gen[r] += 1;
                notified[r] = 0;
                progress = 1;
            }
        }
    }
    for (int r = 0; r < N; ++r)
        if (!done[r]) status[r] = gen[r];                   /* timed out in this generation */
    free(gen);
    free(notified);
    free(done);
    return ORC_OK;
}
