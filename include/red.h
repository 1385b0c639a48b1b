/*
 * red.h -- C ABI of libred.so, a GB300 (sm_103a) library of fp32 / int32 axis
 * reductions:
 *
 *   red_full         full-vector sum / max / min of fp32 data to one scalar;
 *   red_rows         per-row sum / max / min of a dense row-major fp32 matrix,
 *                    optionally folding the old destination value in (accum);
 *   red_rows_ragged  the same for packed rows of varying length (CSR offsets);
 *   red_colprod      TCOLPROD column products dst[0,j] = prod_i src[i,j] for
 *                    fp32 and (wrapping) int32 matrices.
 *
 * Sources of the semantics (cited by page title and section):
 *   [TVM] Apache TVM docs, "reduction -> sm100_packed": "Algorithm" (sum of a
 *         1-D float32 vector through an 8-wide packed add.f32x2 fold; max / min
 *         through a 4-wide max3 / min3 fold), "How inputs change the
 *         algorithm" (accum folds the old dst value into the first
 *         accumulator slot), "Demonstration program" (Tx.sum(dst, src,
 *         accum), destination-passing, B == sum(A) for 32 elements).
 *   [BLK] Triton vector-accumulation blog post (imxueqiu.com), the C version
 *         of the block reduce: warp butterfly, shared-memory stage, one
 *         atomic per block.
 *   [PTO] pto-isa docs, "TCOLPROD": "Math Interpretation" (dst[0,j] =
 *         prod_{i<R} src[i,j]), "Constraints" (row-major, same element type
 *         for src and dst, early return when R == 0 or C == 0), "A2A3
 *         implementation checks" (float and int32 among the element types).
 *
 * Conventions shared by every entry point
 *   - Sizes are int64_t.  Every element count (n, rows * len, nnz, R * ld) is
 *     at most 2^44; a larger one returns RED_EINVAL.
 *   - Pointers to data (x, offsets, out) are DEVICE pointers on the current
 *     CUDA device, owned by the caller, which keeps them alive until the work
 *     queued on `stream` has finished.  fp32 / int32 pointers must be 4-byte
 *     aligned and int64 pointers 8-byte aligned; no larger alignment is needed
 *     (the kernels peel an unaligned head and tail off each span).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host.  Kernels are
 *     launched with programmatic dependent launch: a library kernel may be
 *     scheduled onto SMs while the previous kernel on the stream drains, but
 *     it touches memory only after that kernel has completed and its writes
 *     are visible, so effects are ordered exactly as in plain stream order.
 *   - Status codes: RED_OK on success.  RED_EINVAL for bad arguments, detected
 *     on the host before anything is launched (nothing is written then).
 *     RED_ECUDA if a CUDA call or launch fails; RED_ENOMEM if the one-time
 *     workspace allocation fails.  red_last_error() returns a message for the
 *     last failing call of the calling thread.
 *   - Workspace: partial results of the multi-CTA stages live in a workspace
 *     that the library allocates once per device (16 MiB of partials plus
 *     65536 counters, zeroed at allocation), on the first call that needs it.
 *     That first call should therefore come before any CUDA stream capture;
 *     after it, the calls of this header other than red_full_noalloc can be
 *     captured into a CUDA graph and replayed (they then allocate nothing and
 *     synchronise nothing).
 *     The counters reset themselves at the end of every call, so calls on one
 *     device must be ordered (one stream, or streams ordered by events):
 *     two such calls running at the same time on one device race.  The
 *     workspace lives in the device's primary context: after a
 *     cudaDeviceReset the library must not be called on that device again in
 *     the same process (its workspace pointers are stale).
 *   - fp32 sums use round-to-nearest with flush-to-zero packed adds and a
 *     library-chosen summation order: the result equals the exact sum up to
 *     rounding (tests bound it by 1e-5 * sum|x|).  Max / min are exact.
 *     Integer products are exact modulo 2^32.
 *   - NaN inputs are not supported (max / min then return an unspecified
 *     operand); infinities propagate as in IEEE arithmetic.
 */
#ifndef RED_H
#define RED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. */
typedef struct CUstream_st *red_stream_t;

/* Reduction operator.  RED_PROD is accepted by the column reductions only. */
enum red_op { RED_SUM = 0, RED_MAX = 1, RED_MIN = 2, RED_PROD = 3 };

/* Element type of the column reductions (red_cols, red_colprod): float,
 * int32, IEEE binary16, bfloat16, int16, uint16, uint32 -- the element types
 * of [PTO] "A2A3 implementation checks" and "A5 implementation checks". */
enum red_dtype {
    RED_F32 = 0,
    RED_I32 = 1,
    RED_F16 = 2,
    RED_BF16 = 3,
    RED_I16 = 4,
    RED_U16 = 5,
    RED_U32 = 6
};

/* Status codes.  There is no timeout status: no kernel of this library
 * waits on another CTA, stream or device (the last-block stages count
 * arrivals and the last arrival does the fold), so no wait can run out. */
enum red_status { RED_OK = 0, RED_EINVAL = -1, RED_ECUDA = -2, RED_ENOMEM = -3 };

/* Grid stage of red_full (how the per-CTA partials become one scalar). */
enum red_full_mode {
    RED_MODE_AUTO = 0,       /* the measured default: two-pass for sums (deterministic),
                                atomic for max / min (exact in any order) */
    RED_MODE_TWO_PASS = 1,   /* partials to the workspace, then a second kernel */
    RED_MODE_LAST_BLOCK = 2, /* one kernel; the last CTA to finish folds the partials */
    RED_MODE_ATOMIC = 3      /* identity into *out, then one atomic per CTA */
};

/* Tuning knobs for measurement (0 restores the automatic choice). */
enum red_knob {
    RED_KNOB_ROWS_GROUP = 1,   /* lanes per dense row: 1, 2, 4, 8, 16 or 32 */
    RED_KNOB_RAGGED_GROUP = 2, /* lanes per ragged row: 1, 2, 4, 8, 16 or 32 */
    RED_KNOB_COLPROD_SPLITS = 3, /* CTAs along the row axis of red_cols / red_colprod (>= 1) */
    RED_KNOB_FULL_CTAS_PER_SM = 4, /* resident CTAs per SM for red_full (>= 1) */
    RED_KNOB_RAGGED_STAGED = 5, /* red_rows_ragged mapping: 1 CTA-staged tiles, 2 direct (lanes per row) */
    RED_KNOB_ROWS_ALIGNED = 6, /* red_rows on rows of whole 32-byte blocks: 2 = the general row kernel
                                  instead of the aligned one (1 and 0: automatic) */
    RED_KNOB_COLS_LANES = 7    /* red_cols / red_colprod: at most this many lanes per row of a column tile
                                  (1, 2, 4, 8, 16 or 32) */
};

/*
 * red_full -- reduce a 1-D fp32 vector to one scalar.  [TVM] "Algorithm"
 * (the thread-scope fold) applied per thread, then [BLK]'s warp butterfly and
 * shared-memory stage per CTA, then the grid stage set by red_set_full_mode.
 *   op     RED_SUM, RED_MAX or RED_MIN.
 *   x      device pointer to n contiguous floats (may be NULL when n == 0).
 *   n      number of elements, 0 <= n <= 2^44 (a larger n returns RED_EINVAL).
 *   out    device pointer to one float, written with the result.
 *   stream CUDA stream the work is queued on.
 * n == 0: RED_SUM writes 0; RED_MAX / RED_MIN return RED_EINVAL (an empty
 * vector has no extreme).
 */
int red_full(int op, const float *x, int64_t n, float *out, red_stream_t stream);

/*
 * red_full_stats -- sum, max, min and sum of |x| of a 1-D fp32 vector from a
 * single read of x (three red_full calls read it three times).  Each statistic
 * is the one red_full computes ([TVM] "Algorithm": the packed-add sum fold
 * and the max3 / min3 fold side by side in every thread); sum |x| is the sum
 * of the absolute values (the scale of the sum's rounding error).
 *   x      device pointer to n contiguous floats, n >= 1.
 *   out    device pointer to 4 floats: out[0] = sum, out[1] = max,
 *          out[2] = min, out[3] = sum of |x|.
 * n == 0 returns RED_EINVAL (an empty vector has no max or min).  Uses the
 * workspace (last-block grid stage) like red_full.
 */
int red_full_stats(const float *x, int64_t n, float *out, red_stream_t stream);

/*
 * red_rows_stats -- red_full_stats for every row of a row-major fp32 matrix
 * (row r = x[r*len .. r*len+len)), from one read of x:
 * out[4r] = sum, out[4r+1] = max, out[4r+2] = min, out[4r+3] = sum of |x|.
 *   out    device pointer to 4*rows floats, 16-byte aligned.
 * rows == 0 does nothing; len == 0 returns RED_EINVAL (no max or min).
 */
int red_rows_stats(const float *x, int64_t rows, int64_t len, float *out, red_stream_t stream);

/*
 * red_rows -- per-row reduction of a row-major fp32 matrix: row r is
 * x[r*len .. r*len+len), out[r] = op over row r.  With accum != 0 the old
 * value out[r] is folded in as one more operand ([TVM] "How inputs change the
 * algorithm": accum folds the old dst value into the first accumulator slot).
 *   op     RED_SUM, RED_MAX or RED_MIN.
 *   x      device pointer to rows*len floats (leading dimension len).
 *   rows   number of rows, >= 0; len row length, >= 0.
 *   accum  0: overwrite out; non-zero: fold the old out[r] in.
 *   out    device pointer to rows floats (read first when accum != 0).
 * len == 0: RED_SUM writes zeros (accum: leaves out unchanged); RED_MAX /
 * RED_MIN return RED_EINVAL.  rows == 0 does nothing.  Rows of at most
 * RED_THREAD_MAX_LEN floats are reduced as red_rows_thread does (one thread
 * per row, the thread-scope fold), which is the faster layout for them.
 */
int red_rows(int op, const float *x, int64_t rows, int64_t len, int accum, float *out,
             red_stream_t stream);

/*
 * red_rows_thread -- per-row reduction in which one GPU thread reduces each
 * row with the thread-scope fold of [TVM] "Algorithm", exactly as the public
 * device header red_device.cuh defines it (red_dev::thread_sum / thread_max /
 * thread_min<len>): the row is the thread's register vector, and with accum
 * the old out[r] is added into the fold's first accumulator slot ([TVM] "How
 * inputs change the algorithm").  The rounding order of every row's sum is
 * therefore fixed by len alone (the same bits on every GPU, grid and
 * launch); red_rows is faster for long rows.  Row r is x[r*len ..
 * r*len+len).
 *   len    1 .. RED_THREAD_MAX_LEN (the register vector's static length; the
 *          page's gate starts its packed fold at len 8, shorter rows fold
 *          left to right).
 *   other arguments as red_rows.  Invalid len returns RED_EINVAL.
 */
#define RED_THREAD_MAX_LEN 64
int red_rows_thread(int op, const float *x, int64_t rows, int len, int accum, float *out,
                    red_stream_t stream);

/*
 * red_rows_ragged -- per-row reduction of packed rows of varying length:
 * row r is x[offsets[r] .. offsets[r+1]).  Same ops and accum as red_rows.
 *   x        device pointer to nnz floats.
 *   offsets  device pointer to rows+1 int64 values with offsets[0] = 0,
 *            offsets non-decreasing and offsets[rows] = nnz.  The library
 *            cannot check device-resident offsets without synchronising; it
 *            clamps every offset to [0, nnz] (a decreasing pair reads as an
 *            empty row), so it never reads outside x[0 .. nnz), but the
 *            results of invalid offsets are unspecified.
 *   rows     number of rows, >= 0.
 *   nnz      number of values in x, >= 0 (passed by the caller: reading
 *            offsets[rows] from device memory would need a synchronise).
 *   out      device pointer to rows floats (read first when accum != 0).
 * An empty row gives 0 for RED_SUM, -inf for RED_MAX and +inf for RED_MIN
 * (the identity of the fold); with accum the old out[r] is kept.
 * Mapping ("Row mapping (ragged rows)": thread per row with direct loads, or
 * a CTA-staged copy of a row range into shared memory, chosen by
 * measurement): rows of fewer than 11 floats on average go through
 * shared-memory tiles, longer ones to lanes per row with direct loads;
 * RED_KNOB_RAGGED_STAGED forces either, and a RED_KNOB_RAGGED_GROUP setting
 * (lanes per row) implies the direct mapping unless staging is forced.
 */
int red_rows_ragged(int op, const float *x, const int64_t *offsets, int64_t rows, int64_t nnz,
                    int accum, float *out, red_stream_t stream);

/*
 * red_cols -- column reductions of a row-major R x C matrix:
 * out[j] = op_{i=0}^{R-1} x[i*C + j] for 0 <= j < C.  op RED_PROD is [PTO]
 * TCOLPROD ("Math Interpretation"); RED_SUM, RED_MAX and RED_MIN are its
 * column siblings over the same layout.  x and out have the element type
 * `dtype` ([PTO] "Constraints": the same element type on both sides).
 *   Arithmetic: floating types accumulate in fp32 (RED_F16 / RED_BF16 are
 *   widened exactly and the result is rounded to nearest-even once; products
 *   and sums use round-to-nearest fp32 steps, so an fp32 product of R values
 *   is within about R * 2^-24 relative of the exact product); integer sums
 *   and products wrap modulo 2^bits of the type; max / min compare values
 *   (signed for RED_I32 / RED_I16, unsigned for RED_U32 / RED_U16; NaN
 *   inputs are not supported).
 *   x, out  device pointers aligned to the element size; out holds C elements.
 *   R, C    >= 0.  R == 0 or C == 0 returns RED_OK at once and writes nothing
 *           ([PTO] "Constraints": the implementation returns early; the same
 *           rule is kept for the siblings).
 * Bad op or dtype, negative sizes, NULL or misaligned pointers: RED_EINVAL.
 */
int red_cols(int op, int dtype, const void *x, int64_t R, int64_t C, void *out, red_stream_t stream);

/*
 * red_cols_ld -- red_cols on the valid region of a larger row-major matrix:
 * out[j] = op_{i=0}^{R-1} x[i*ld + j] for 0 <= j < C, row stride ld >= C
 * (in elements).  This is [PTO] "Math Interpretation" with R = ValidRow and
 * C = ValidCol of a row-major tile whose allocated width is ld; red_cols is
 * the case ld == C.  Elements of x past column C of each row are never read.
 * Arguments and errors as for red_cols; ld < C, or R * ld beyond the size
 * limit: RED_EINVAL.
 */
int red_cols_ld(int op, int dtype, const void *x, int64_t R, int64_t C, int64_t ld, void *out,
                red_stream_t stream);

/*
 * red_full_typed / red_rows_typed -- red_full and red_rows for every element
 * type of red_cols (enum red_dtype) and every operator including RED_PROD:
 * out[0] = op over x[0..n); out[r] = op over row r = x[r*len .. r*len+len),
 * with accum != 0 folding the old out[r] in as one more operand ([TVM] "How
 * inputs change the algorithm").  Arithmetic as red_cols: floating types
 * accumulate in fp32 and round once to the element type, integer sums and
 * products wrap modulo 2^bits, max / min compare values.  x and out hold the
 * element type and are aligned to its size.
 *   Empty input: RED_SUM writes 0 and RED_PROD writes 1 (with accum, rows are
 *   left unchanged); RED_MAX / RED_MIN return RED_EINVAL.
 * The fp32 fast paths (packed folds, 256-bit loads) are red_full / red_rows;
 * these are the general-type versions.
 */
int red_full_typed(int op, int dtype, const void *x, int64_t n, void *out, red_stream_t stream);
int red_rows_typed(int op, int dtype, const void *x, int64_t rows, int64_t len, int accum, void *out,
                   red_stream_t stream);

/*
 * red_colprod -- [PTO] TCOLPROD: red_cols(RED_PROD, dtype, ...).
 *   dtype  any enum red_dtype; RED_F32 products round to nearest in fp32,
 *          RED_I32 (and the other integer types) wrap modulo 2^bits.
 *   R == 0 or C == 0 returns RED_OK at once and writes nothing ([PTO]
 *   "Constraints": the implementation returns early).
 */
int red_colprod(int dtype, const void *x, int64_t R, int64_t C, void *out, red_stream_t stream);

/*
 * red_full_noalloc -- red_full for callers that cannot allocate device memory.
 * The pages have no counterpart of this call; it exists for the library's
 * users.  red_full allocates a 16 MiB workspace with cudaMalloc on its first
 * call on a device.  Some callers cannot let a library do that: cudaMalloc
 * (and cudaFree) may synchronise the whole device, which a latency-bound
 * serving or real-time loop cannot absorb, and a framework whose own caching
 * allocator has reserved the device memory, or that enforces a memory budget,
 * may see the allocation fail or break its accounting.
 *
 * This call never allocates: it calls no cudaMalloc, cudaFree or allocating
 * library routine.  Its scratch is a fixed array in the library's device
 * memory, RED_NOALLOC_MAX_PARTIALS fp32 partial slots plus one arrival
 * counter (16 KiB + 256 B), which every GPU that loads the library holds
 * until the process exits.  The result is the same reduction as red_full
 * with the last-block grid stage (one kernel; the red_set_full_mode setting
 * does not apply).
 *   op, x, n, out, stream   as for red_full (device pointers, async on stream).
 * Errors: as red_full; in addition RED_EINVAL when the launch would need more
 * CTAs (partial slots) than the scratch holds -- only possible when
 * RED_KNOB_FULL_CTAS_PER_SM asks for more than RED_NOALLOC_MAX_PARTIALS CTAs
 * in all; the message says so.  n itself has no limit beyond red_full's.
 * Set-up: the first call on a device looks up the scratch array's device
 * address (cudaGetSymbolAddress, with that device current) and caches it, so
 * that first call should come before any CUDA stream capture.  The scratch
 * array belongs to the library's device code, which the CUDA driver may load
 * onto a device only when the library first uses that device (lazy module
 * loading); the driver then places the module's code and static data, this
 * array included, in device memory.  So "allocates nothing" holds from the
 * moment the module is resident on the device: a caller that must not see
 * even that load makes one call (or any other call of this library) on the
 * device during its set-up.  A cudaDeviceReset, or any other teardown of the
 * device's primary context, unloads the module and makes the cached address
 * stale: this call must not be used on that device afterwards in the same
 * process (red_full's workspace pointers are invalidated the same way).
 * Sharing: every call on a device uses the same scratch.  Each call first
 * clears the counter on its stream (cudaMemsetAsync, which allocates
 * nothing), and the partials are rewritten before they are read; calls that
 * overlap on the GPU (different streams, not ordered by events) race and
 * give wrong results.
 */
#define RED_NOALLOC_MAX_PARTIALS 4096
int red_full_noalloc(int op, const float *x, int64_t n, float *out, red_stream_t stream);

/* Select the grid stage of red_full (enum red_full_mode).  Process-wide.
 * Returns RED_OK, or RED_EINVAL for an unknown mode. */
int red_set_full_mode(int mode);

/* The current setting of red_set_full_mode (RED_MODE_AUTO by default). */
int red_get_full_mode(void);

/* Set a tuning knob (enum red_knob); value 0 restores the automatic choice.
 * Returns RED_EINVAL for an unknown knob or an out-of-range value. */
int red_set_knob(int knob, int value);

/* Current value of a knob (0 = automatic), or RED_EINVAL for an unknown knob. */
int red_get_knob(int knob);

/* Message for the last non-OK status returned to the calling thread
 * ("" if none).  The string is owned by the library and stays valid until
 * the thread's next failing call. */
const char *red_last_error(void);

/* Free the calling thread's current device's workspace.  The caller must make
 * sure no queued work still uses it (e.g. synchronise the device first); the
 * next call that needs it allocates it again.  Returns RED_OK or RED_ECUDA. */
int red_release_workspace(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads), for counting launches around a timed region. */
uint64_t red_launch_count(void);

/* ABI version of this header: 2 (2: red_get_full_mode returns the setting,
 * RED_MODE_AUTO included, because the automatic grid stage depends on the
 * operator). */
int red_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RED_H */
