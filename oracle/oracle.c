/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the fp32/int32 axis
 * reductions (full-vector sum/max/min, per-row sum/max/min with accum, dense
 * and ragged rows, and TCOLPROD column products).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) includes, links or calls this file.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no header, helper, table or constant with the CUDA sources.
 *
 * Every function below is the plain definition of its result, written out in
 * index order with no blocking, no reordering and no parallelism:
 *   - sums accumulate in double (and also report sum |x| for tolerances);
 *   - max / min compare the fp32 values directly (exact in any order);
 *   - fp32 column products accumulate in double and round to fp32 once;
 *   - int32 column products multiply in uint32, i.e. wrap modulo 2^32.
 * One function is an algorithm rather than a definition: orc_thread_sum
 * takes the steps of the sm100_packed thread-scope fold in the page's order,
 * one fp32 operation each, so that a GPU fold in that order can be checked
 * bit for bit (its result is the sum up to that fixed rounding order).
 *
 * Sources (cited by page title and section):
 *   [TVM]  Apache TVM docs, "reduction -> sm100_packed": sections "Algorithm"
 *          (sum of a 1-D float32 vector; max / min), "How inputs change the
 *          algorithm" (accum folds the old dst value into the first
 *          accumulator slot), "Demonstration program" (B == sum(A)).
 *   [PTO]  pto-isa docs, "TCOLPROD": "Math Interpretation"
 *          (dst[0,j] = prod_{i<R} src[i,j]) and "Constraints" (returns early
 *          when R == 0 or C == 0).
 *
 * Readings where the pages are silent:
 *   - An empty dense input has no max / min: status -1 (error).  An empty
 *     ragged row folds nothing, so its max is -inf and its min +inf (with
 *     accum the old dst value survives); an empty sum is 0.
 *   - The early return of TCOLPROD leaves dst untouched (no identity written).
 *
 * Parity status: every function here is pinned by the CPU tests (page-given
 * 32-element check, closed forms, exact-arithmetic brute force, invariants).
 *
 * Return value of every function but orc_thread_sum: 0 on success, -1 on
 * invalid arguments (orc_thread_sum returns the fp32 result).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)

/* ---------------------------------------------------------------- full --- */

/* [TVM] "Algorithm", sum: the scalar sum of a 1-D float32 vector.
 * *sum = sum_i x[i] and *abs_sum = sum_i |x[i]|, both in double. */
int orc_full_sum(const float *x, int64_t n, double *sum, double *abs_sum)
{
    if (n < 0 || (n > 0 && !x) || !sum || !abs_sum)
        return ORC_EINVAL;
    double s = 0.0, a = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        s += (double)x[i];
        a += fabs((double)x[i]);
    }
    *sum = s;
    *abs_sum = a;
    return ORC_OK;
}

/* [TVM] "Algorithm", max / min: the largest (smallest) element, in fp32.
 * An empty vector has no extreme: -1. */
int orc_full_max(const float *x, int64_t n, float *out)
{
    if (n <= 0 || !x || !out)
        return ORC_EINVAL;
    float m = x[0];
    for (int64_t i = 1; i < n; ++i)
        if (x[i] > m)
            m = x[i];
    *out = m;
    return ORC_OK;
}

int orc_full_min(const float *x, int64_t n, float *out)
{
    if (n <= 0 || !x || !out)
        return ORC_EINVAL;
    float m = x[0];
    for (int64_t i = 1; i < n; ++i)
        if (x[i] < m)
            m = x[i];
    *out = m;
    return ORC_OK;
}

/* ------------------------------------------------------------ row core --- */

/* Sum of seg[0..len), started from `init` (accum: the old dst value goes into
 * the first accumulator slot, [TVM] "How inputs change the algorithm"). */
static double seg_sum(const float *seg, int64_t len, double init, double *abs_out,
                      double abs_init)
{
    double s = init, a = abs_init;
    for (int64_t i = 0; i < len; ++i) {
        s += (double)seg[i];
        a += fabs((double)seg[i]);
    }
    *abs_out = a;
    return s;
}

static float seg_max(const float *seg, int64_t len, float init)
{
    float m = init;
    for (int64_t i = 0; i < len; ++i)
        if (seg[i] > m)
            m = seg[i];
    return m;
}

static float seg_min(const float *seg, int64_t len, float init)
{
    float m = init;
    for (int64_t i = 0; i < len; ++i)
        if (seg[i] < m)
            m = seg[i];
    return m;
}

/* ---------------------------------------------------------- dense rows --- */

/* Row r is x[r*len .. r*len+len) (row-major, leading dimension len).
 * out[r] = (accum ? dst_old[r] : 0) + sum of row r, in double;
 * abs_out[r] = (accum ? |dst_old[r]| : 0) + sum of |row r|. */
int orc_rows_sum(const float *x, int64_t rows, int64_t len, int accum,
                 const float *dst_old, double *out, double *abs_out)
{
    if (rows < 0 || len < 0 || (rows > 0 && (!out || !abs_out)) ||
        (rows > 0 && len > 0 && !x) || (accum && rows > 0 && !dst_old))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        double init = accum ? (double)dst_old[r] : 0.0;
        double ainit = accum ? fabs((double)dst_old[r]) : 0.0;
        out[r] = seg_sum(x + r * len, len, init, &abs_out[r], ainit);
    }
    return ORC_OK;
}

/* out[r] = max over row r (folded with dst_old[r] when accum).  A dense row
 * of length 0 has no max: -1. */
int orc_rows_max(const float *x, int64_t rows, int64_t len, int accum,
                 const float *dst_old, float *out)
{
    if (rows < 0 || len < 0 || (rows > 0 && (!out || !x)) ||
        (accum && rows > 0 && !dst_old) || (rows > 0 && len == 0))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        const float *seg = x + r * len;
        float m = seg_max(seg + 1, len - 1, seg[0]);
        if (accum && dst_old[r] > m)
            m = dst_old[r];
        out[r] = m;
    }
    return ORC_OK;
}

int orc_rows_min(const float *x, int64_t rows, int64_t len, int accum,
                 const float *dst_old, float *out)
{
    if (rows < 0 || len < 0 || (rows > 0 && (!out || !x)) ||
        (accum && rows > 0 && !dst_old) || (rows > 0 && len == 0))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        const float *seg = x + r * len;
        float m = seg_min(seg + 1, len - 1, seg[0]);
        if (accum && dst_old[r] < m)
            m = dst_old[r];
        out[r] = m;
    }
    return ORC_OK;
}

/* --------------------------------------------------------- ragged rows --- */

/* Row r is x[off[r] .. off[r+1]) with off[0] = 0, off non-decreasing and
 * off[rows] the number of values.  Offsets that break this are rejected. */
static int check_offsets(const int64_t *off, int64_t rows)
{
    if (off[0] != 0)
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r)
        if (off[r + 1] < off[r])
            return ORC_EINVAL;
    return ORC_OK;
}

int orc_ragged_sum(const float *x, const int64_t *off, int64_t rows, int accum,
                   const float *dst_old, double *out, double *abs_out)
{
    if (rows < 0 || !off || (rows > 0 && (!out || !abs_out)) ||
        (accum && rows > 0 && !dst_old))
        return ORC_EINVAL;
    if (check_offsets(off, rows) != ORC_OK || (off[rows] > 0 && !x))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        double init = accum ? (double)dst_old[r] : 0.0;
        double ainit = accum ? fabs((double)dst_old[r]) : 0.0;
        out[r] = seg_sum(x + off[r], off[r + 1] - off[r], init, &abs_out[r], ainit);
    }
    return ORC_OK;
}

/* An empty ragged row folds nothing: -inf for max (the old dst value with
 * accum). */
int orc_ragged_max(const float *x, const int64_t *off, int64_t rows, int accum,
                   const float *dst_old, float *out)
{
    if (rows < 0 || !off || (rows > 0 && !out) || (accum && rows > 0 && !dst_old))
        return ORC_EINVAL;
    if (check_offsets(off, rows) != ORC_OK || (off[rows] > 0 && !x))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        float init = accum ? dst_old[r] : -INFINITY;
        out[r] = seg_max(x + off[r], off[r + 1] - off[r], init);
    }
    return ORC_OK;
}

int orc_ragged_min(const float *x, const int64_t *off, int64_t rows, int accum,
                   const float *dst_old, float *out)
{
    if (rows < 0 || !off || (rows > 0 && !out) || (accum && rows > 0 && !dst_old))
        return ORC_EINVAL;
    if (check_offsets(off, rows) != ORC_OK || (off[rows] > 0 && !x))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        float init = accum ? dst_old[r] : INFINITY;
        out[r] = seg_min(x + off[r], off[r + 1] - off[r], init);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------- TCOLPROD --- */

/* [PTO] "Math Interpretation": dst[0,j] = prod_{i=0}^{R-1} src[i,j] for
 * 0 <= j < C, src row-major R x C.  The product of each column is taken in
 * double, in row order, and written both as double (out_d, may be NULL) and
 * rounded once to fp32 (out_f, may be NULL).  [PTO] "Constraints": R == 0 or
 * C == 0 returns early and writes nothing. */
int orc_colprod_f32(const float *x, int64_t R, int64_t C, float *out_f, double *out_d)
{
    if (R < 0 || C < 0)
        return ORC_EINVAL;
    if (R == 0 || C == 0)
        return ORC_OK;
    if (!x || (!out_f && !out_d))
        return ORC_EINVAL;
    for (int64_t j = 0; j < C; ++j) {
        double p = 1.0;
        for (int64_t i = 0; i < R; ++i)
            p *= (double)x[i * C + j];
        if (out_d)
            out_d[j] = p;
        if (out_f)
            out_f[j] = (float)p;
    }
    return ORC_OK;
}

/* Same definition for int32: products wrap modulo 2^32 (done in uint32 so
 * that overflow is defined), then reinterpret as int32. */
int orc_colprod_i32(const int32_t *x, int64_t R, int64_t C, int32_t *out)
{
    if (R < 0 || C < 0)
        return ORC_EINVAL;
    if (R == 0 || C == 0)
        return ORC_OK;
    if (!x || !out)
        return ORC_EINVAL;
    for (int64_t j = 0; j < C; ++j) {
        uint32_t p = 1u;
        for (int64_t i = 0; i < R; ++i)
            p *= (uint32_t)x[i * C + j];
        out[j] = (int32_t)p;
    }
    return ORC_OK;
}

/* ------------------------------------------------- thread-scope fold --- */

/* [TVM] "Algorithm", sum (the sm100_packed thread-scope primitive), with
 * the fp32 rounding order the page fixes, one fp32 operation per step:
 *   n >= 8: s[0..7] = a[0..7]; with accum s[0] = s[0] + dst ("folds the old
 *           dst value into the first accumulator slot"); every further full
 *           chunk of 8 is added lane-wise, s[k] = s[k] + a[c+k]; a remainder
 *           of r < 8 elements is added one at a time into slots 0..r-1
 *           ("handle the remainder scalar"); then the 8 -> 4 -> 2 -> 1
 *           collapse: (s0,s1) += (s2,s3), (s4,s5) += (s6,s7),
 *           (s0,s1) += (s4,s5), result s0 + s1.
 *   n < 8 (below the page's dispatch gate): a left-to-right fold starting
 *           from a[0] (plus dst with accum).
 * Only the order is the page's; each step is a plain fp32 round-to-nearest
 * addition (no denormal can arise from the inputs used). */
float orc_thread_sum(const float *a, int64_t n, int accum, float dst)
{
    if (n <= 0)
        return accum ? dst : 0.0f;
    if (n < 8) {
        float r = a[0];
        if (accum)
            r = r + dst;
        for (int64_t i = 1; i < n; ++i)
            r = r + a[i];
        return r;
    }
    float s[8];
    for (int k = 0; k < 8; ++k)
        s[k] = a[k];
    if (accum)
        s[0] = s[0] + dst;
    int64_t c = 8;
    for (; c + 8 <= n; c += 8)
        for (int k = 0; k < 8; ++k)
            s[k] = s[k] + a[c + k];
    for (int64_t i = c; i < n; ++i)
        s[i - c] = s[i - c] + a[i];
    s[0] = s[0] + s[2];
    s[1] = s[1] + s[3];
    s[4] = s[4] + s[6];
    s[5] = s[5] + s[7];
    s[0] = s[0] + s[4];
    s[1] = s[1] + s[5];
    return s[0] + s[1];
}

/* ------------------------------------------------ column reductions --- */

/* Element types (the A2A3 / A5 lists of pto-isa docs, "TCOLPROD",
 * "Constraints"): 0 float, 1 int32, 2 half, 3 bfloat16, 4 int16,
 * 5 uint16, 6 uint32.  Operators: 0 sum, 1 max, 2 min, 3 product. */
enum { ORC_F32 = 0, ORC_I32 = 1, ORC_F16 = 2, ORC_BF16 = 3, ORC_I16 = 4, ORC_U16 = 5, ORC_U32 = 6 };
enum { ORC_SUM = 0, ORC_MAX = 1, ORC_MIN = 2, ORC_PROD = 3 };

/* IEEE binary16 bits -> double, exactly (sign, 5-bit exponent, 10-bit
 * fraction; subnormals, infinities and NaN included). */
double orc_half_to_double(uint16_t h)
{
    const int sign = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* (1024 + f) * 2^(e-25) */
    return sign ? -v : v;
}

/* bfloat16 bits -> double, exactly: the high half of a binary32. */
double orc_bf16_to_double(uint16_t b)
{
    const uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static int elem_size(int dtype)
{
    switch (dtype) {
    case ORC_F32: case ORC_I32: case ORC_U32: return 4;
    case ORC_F16: case ORC_BF16: case ORC_I16: case ORC_U16: return 2;
    default: return 0;
    }
}

static double elem_f(const void *x, int dtype, int64_t k)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)x)[k];
    case ORC_F16: return orc_half_to_double(((const uint16_t *)x)[k]);
    default: return orc_bf16_to_double(((const uint16_t *)x)[k]);
    }
}

static int64_t elem_i(const void *x, int dtype, int64_t k)
{
    switch (dtype) {
    case ORC_I32: return (int64_t)((const int32_t *)x)[k];
    case ORC_U32: return (int64_t)((const uint32_t *)x)[k];
    case ORC_I16: return (int64_t)((const int16_t *)x)[k];
    default: return (int64_t)((const uint16_t *)x)[k];
    }
}

/* Column reductions of a row-major R x C matrix of a floating type:
 * out[j] = op over rows i of x[i][j] in double (sum and product accumulate
 * in index order; max / min compare directly), abs_out[j] (may be NULL) =
 * sum of |x[i][j]|.  R == 0 or C == 0 returns early, writing nothing (the
 * TCOLPROD rule, applied to the column siblings as well). */
int orc_cols_f(int op, int dtype, const void *x, int64_t R, int64_t C, double *out, double *abs_out)
{
    if (op < ORC_SUM || op > ORC_PROD || !(dtype == ORC_F32 || dtype == ORC_F16 || dtype == ORC_BF16) ||
        R < 0 || C < 0)
        return ORC_EINVAL;
    if (R == 0 || C == 0)
        return ORC_OK;
    if (!x || !out)
        return ORC_EINVAL;
    for (int64_t j = 0; j < C; ++j) {
        double acc = elem_f(x, dtype, j), a = fabs(acc);
        for (int64_t i = 1; i < R; ++i) {
            const double v = elem_f(x, dtype, i * C + j);
            a += fabs(v);
            if (op == ORC_SUM)
                acc += v;
            else if (op == ORC_PROD)
                acc *= v;
            else if (op == ORC_MAX)
                acc = v > acc ? v : acc;
            else
                acc = v < acc ? v : acc;
        }
        out[j] = acc;
        if (abs_out)
            abs_out[j] = a;
    }
    return ORC_OK;
}

/* The same for an integer type: sum and product wrap modulo 2^bits of the
 * type (done in uint64, then reduced to the type's width and read back as
 * the type, so signed results are two's complement); max / min compare the
 * values.  out[j] holds the result as a (sign-extended) int64. */
int orc_cols_i(int op, int dtype, const void *x, int64_t R, int64_t C, int64_t *out)
{
    if (op < ORC_SUM || op > ORC_PROD || !(dtype == ORC_I32 || dtype == ORC_U32 || dtype == ORC_I16 ||
                                           dtype == ORC_U16) ||
        R < 0 || C < 0)
        return ORC_EINVAL;
    if (R == 0 || C == 0)
        return ORC_OK;
    if (!x || !out)
        return ORC_EINVAL;
    const int bits = 8 * elem_size(dtype);
    const uint64_t mask = bits == 64 ? ~0ull : ((1ull << bits) - 1);
    const int is_signed = dtype == ORC_I32 || dtype == ORC_I16;
    for (int64_t j = 0; j < C; ++j) {
        int64_t m = elem_i(x, dtype, j);
        uint64_t w = (uint64_t)m;
        for (int64_t i = 1; i < R; ++i) {
            const int64_t v = elem_i(x, dtype, i * C + j);
            if (op == ORC_SUM)
                w += (uint64_t)v;
            else if (op == ORC_PROD)
                w *= (uint64_t)v;
            else if (op == ORC_MAX)
                m = v > m ? v : m;
            else
                m = v < m ? v : m;
        }
        if (op == ORC_SUM || op == ORC_PROD) {
            w &= mask;
            if (is_signed && (w >> (bits - 1)) & 1u)
                m = (int64_t)w - (int64_t)(mask + 1);
            else
                m = (int64_t)w;
        }
        out[j] = m;
    }
    return ORC_OK;
}

/* ----------------------------------------- typed full and row reductions --- */

/* Row r = x[r*len .. r*len+len) of a floating element type; out[r] = op over
 * the row in double, started from the old dst value when accum ([TVM] "How
 * inputs change the algorithm": the old value is one more operand);
 * abs_out[r] = sum of |row| (+ |old|).  An empty row gives 0 for sum, 1 for
 * product (the old value with accum); empty max / min rows are rejected.  A
 * full vector is the case rows = 1. */
int orc_rows_typed_f(int op, int dtype, const void *x, int64_t rows, int64_t len, int accum,
                     const void *dst_old, double *out, double *abs_out)
{
    if (op < ORC_SUM || op > ORC_PROD || !(dtype == ORC_F32 || dtype == ORC_F16 || dtype == ORC_BF16) ||
        rows < 0 || len < 0 || (rows > 0 && (!out || !abs_out)) || (rows > 0 && len > 0 && !x) ||
        (accum && rows > 0 && !dst_old) || (rows > 0 && len == 0 && (op == ORC_MAX || op == ORC_MIN) && !accum))
        return ORC_EINVAL;
    for (int64_t r = 0; r < rows; ++r) {
        double acc, a = 0.0;
        int64_t k = 0;
        if (accum) {
            acc = elem_f(dst_old, dtype, r);
            a = fabs(acc);
        } else if (len > 0) {
            acc = elem_f(x, dtype, r * len);
            a = fabs(acc);
            k = 1;
        } else {
            acc = op == ORC_PROD ? 1.0 : 0.0;
        }
        for (; k < len; ++k) {
            const double v = elem_f(x, dtype, r * len + k);
            a += fabs(v);
            if (op == ORC_SUM)
                acc += v;
            else if (op == ORC_PROD)
                acc *= v;
            else if (op == ORC_MAX)
                acc = v > acc ? v : acc;
            else
                acc = v < acc ? v : acc;
        }
        out[r] = acc;
        abs_out[r] = a;
    }
    return ORC_OK;
}

/* The same for an integer element type: sums and products wrap modulo
 * 2^bits of the type; out[r] is the result as a sign-extended int64. */
int orc_rows_typed_i(int op, int dtype, const void *x, int64_t rows, int64_t len, int accum,
                     const void *dst_old, int64_t *out)
{
    if (op < ORC_SUM || op > ORC_PROD ||
        !(dtype == ORC_I32 || dtype == ORC_U32 || dtype == ORC_I16 || dtype == ORC_U16) || rows < 0 ||
        len < 0 || (rows > 0 && !out) || (rows > 0 && len > 0 && !x) || (accum && rows > 0 && !dst_old) ||
        (rows > 0 && len == 0 && (op == ORC_MAX || op == ORC_MIN) && !accum))
        return ORC_EINVAL;
    const int bits = 8 * elem_size(dtype);
    const uint64_t mask = (1ull << bits) - 1;
    const int is_signed = dtype == ORC_I32 || dtype == ORC_I16;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t m;
        int64_t k = 0;
        if (accum) {
            m = elem_i(dst_old, dtype, r);
        } else if (len > 0) {
            m = elem_i(x, dtype, r * len);
            k = 1;
        } else {
            m = op == ORC_PROD ? 1 : 0;
        }
        uint64_t w = (uint64_t)m;
        for (; k < len; ++k) {
            const int64_t v = elem_i(x, dtype, r * len + k);
            if (op == ORC_SUM)
                w += (uint64_t)v;
            else if (op == ORC_PROD)
                w *= (uint64_t)v;
            else if (op == ORC_MAX)
                m = v > m ? v : m;
            else
                m = v < m ? v : m;
        }
        if (op == ORC_SUM || op == ORC_PROD) {
            w &= mask;
            m = (is_signed && (w >> (bits - 1)) & 1u) ? (int64_t)w - (int64_t)(mask + 1) : (int64_t)w;
        }
        out[r] = m;
    }
    return ORC_OK;
}
