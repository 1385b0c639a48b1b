// red_ragged_staged.cu -- per-row sum / max / min of ragged rows (row r =
// x[off[r] .. off[r+1])) for short rows: the CTA-staged mapping of the
// ragged row step (a coalesced copy of a row range into shared memory, then
// a per-thread fold; "Row mapping (ragged rows)" of the method: thread per
// row with direct loads versus a CTA-staged copy, chosen by measurement).
// The operation, accum and arithmetic are those of the row kernel: Apache
// TVM docs, "reduction -> sm100_packed" (accum folds the old dst value in
// first; sums with add.rn.ftz).
//
// A CTA takes a contiguous range of tiles of RS_ROWS consecutive rows; for
// each it reads the RS_ROWS + 1 offsets (clamped to [0, nnz], so no load
// ever leaves x) and has the next tile's offsets and (estimated) values
// prefetched into L2.  It then walks the tile in runs of consecutive rows
// whose values fit the shared buffer (the whole rest of the tile when it
// fits, else the longest run found by a binary search over the offsets):
// it copies the run's values with 128-bit loads of their 16-byte aligned
// interior (at most three single floats at each end: every load inside the
// span) and each thread folds its rows of the run from shared memory, the
// old value first (accum), then the row's values in order.  A row that
// alone exceeds the buffer is folded by the whole CTA (128-bit loads, a CTA
// reduction, the old value combined with the result); a row whose offsets
// leave the run's span (offsets that decrease) is folded from global memory.
// With rows of a few floats, one lane per row spends ~10 L1 wavefronts per
// 128 coalesced bytes on scattered 4-byte loads; the staged copy needs one.
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int RS_NT = 256;            // threads per CTA
constexpr int RS_ROWS = 1024;         // rows per tile (4 per thread)
constexpr int RS_CAP = 8192;          // staged floats per tile (32 KB)
constexpr int RS_BATCH = 4;           // 128-bit loads in flight per thread while staging

__device__ __forceinline__ int64_t clamp64(int64_t v, int64_t lo, int64_t hi)
{
    return v < lo ? lo : (v > hi ? hi : v);
}

// Copy x[lo, hi) to s_v[g - base] (base = lo rounded down to a 16-byte
// boundary of x): 128-bit loads of the aligned interior, RS_BATCH in flight
// per thread, single floats for the at most three at each end.
__device__ __forceinline__ void stage_span(const float *__restrict__ x, int64_t x_mis, int64_t lo, int64_t hi,
                                           int64_t base, float *s_v)
{
    const int tid = threadIdx.x;
    const int64_t a = ((lo + x_mis + 3) & ~int64_t(3)) - x_mis;
    const int64_t z = ((hi + x_mis) & ~int64_t(3)) - x_mis;
    const int64_t a4 = a < hi ? a : hi;   // head [lo, a4)
    const int64_t z4 = z > a4 ? z : a4;   // interior [a4, z4), tail [z4, hi)
    const int64_t n4 = (z4 - a4) >> 2;
    for (int64_t c0 = tid; c0 < n4; c0 += (int64_t)RS_BATCH * RS_NT) {
        float4 v[RS_BATCH];
#pragma unroll
        for (int u = 0; u < RS_BATCH; ++u)
            if (c0 + u * RS_NT < n4)
                v[u] = ld4f(x + a4 + 4 * (c0 + u * RS_NT));
#pragma unroll
        for (int u = 0; u < RS_BATCH; ++u)
            if (c0 + u * RS_NT < n4)
                *reinterpret_cast<float4 *>(&s_v[a4 - base + 4 * (c0 + u * RS_NT)]) = v[u];
    }
    if (tid < 4) {
        const int64_t g = lo + tid;
        if (g < a4)
            s_v[g - base] = ld1(x + g);
    } else if (tid < 8) {
        const int64_t g = z4 + (tid - 4);
        if (g < hi)
            s_v[g - base] = ld1(x + g);
    }
}

// One row [ob, oe) folded by the whole CTA; the result (with accum) is
// written by thread 0.
template <int OP>
__device__ __forceinline__ void cta_row(const float *__restrict__ x, int64_t x_mis, int64_t ob, int64_t oe,
                                        int accum, float *o, float *s_red)
{
    const int tid = threadIdx.x;
    Fold<OP> f;
    f.init();
    const int64_t a = ((ob + x_mis + 3) & ~int64_t(3)) - x_mis;
    const int64_t z = ((oe + x_mis) & ~int64_t(3)) - x_mis;
    const int64_t a4 = a < oe ? a : oe;
    const int64_t z4 = z > a4 ? z : a4;
    const int64_t n4 = (z4 - a4) >> 2;
    for (int64_t c0 = tid; c0 < n4; c0 += (int64_t)RS_BATCH * RS_NT) {
        float4 v[RS_BATCH];
#pragma unroll
        for (int u = 0; u < RS_BATCH; ++u)
            v[u] = c0 + u * RS_NT < n4 ? ld4f(x + a4 + 4 * (c0 + u * RS_NT))
                                       : make_float4(Op<OP>::identity(), Op<OP>::identity(), Op<OP>::identity(),
                                                     Op<OP>::identity());
#pragma unroll
        for (int u = 0; u < RS_BATCH; ++u)
            f.quad(v[u]);
    }
    if (tid < 4) {
        if (ob + tid < a4)
            f.scalar(ld1(x + ob + tid));
    } else if (tid < 8) {
        if (z4 + (tid - 4) < oe)
            f.scalar(ld1(x + z4 + (tid - 4)));
    }
    float v = cta_reduce<OP, RS_NT / 32>(f.finish(), s_red);
    if (tid == 0)
        *o = accum ? Op<OP>::combine(*o, v) : v;
    __syncthreads();  // s_red is reused
}

// Bulk prefetch of the bytes [b, e) into L2, rounded inward to 16-byte
// boundaries (no byte outside [b, e) is touched) and capped at 64 KB.
__device__ __forceinline__ void l2_prefetch(const void *b, const void *e)
{
    const uintptr_t lo = ((uintptr_t)b + 15u) & ~(uintptr_t)15u;
    uintptr_t hi = (uintptr_t)e & ~(uintptr_t)15u;
    if (hi > lo + 65536u)
        hi = lo + 65536u;
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
}

template <int OP>
__global__ void __launch_bounds__(RS_NT)
ragged_staged_kernel(const float *__restrict__ x, const int64_t *__restrict__ off, int64_t rows, int64_t nnz,
                     int accum, float *__restrict__ out)
{
    pdl_enter();
    __shared__ int64_t s_off[RS_ROWS + 1];
    __shared__ __align__(16) float s_v[RS_CAP + 4];
    __shared__ float s_red[RS_NT / 32];
    __shared__ int s_i1;
    const int tid = threadIdx.x;
    const int64_t x_mis = (int64_t)(((uintptr_t)x & 15u) >> 2);  // x's offset from a 16-byte boundary
    // each CTA takes a contiguous range of tiles, so that the next tile's
    // values start where this tile's end and can be prefetched into L2
    const int64_t ntiles = (rows + RS_ROWS - 1) / RS_ROWS;
    const int64_t per = (ntiles + gridDim.x - 1) / gridDim.x;
    const int64_t t_end = (int64_t)(blockIdx.x + 1) * per < ntiles ? (int64_t)(blockIdx.x + 1) * per : ntiles;
    for (int64_t t = (int64_t)blockIdx.x * per; t < t_end; ++t) {
        const int64_t r0 = t * RS_ROWS;
        const int nr = (int)(rows - r0 < RS_ROWS ? rows - r0 : RS_ROWS);
        for (int i = tid; i <= nr; i += RS_NT)
            s_off[i] = clamp64(off[r0 + i], 0, nnz);
        __syncthreads();
        if (tid == 0 && t + 1 < t_end) {
            // the next tile's offsets, and its values if as long as this
            // tile's (they start where this tile's end)
            const int64_t q0 = r0 + RS_ROWS;
            const int64_t q1 = q0 + RS_ROWS + 1 < rows + 1 ? q0 + RS_ROWS + 1 : rows + 1;
            l2_prefetch(off + q0, off + q1);
            const int64_t e0 = s_off[nr], span = s_off[nr] - s_off[0];
            if (span > 0)
                l2_prefetch(x + e0, x + (e0 + span < nnz ? e0 + span : nnz));
        }
        int i0 = 0;
        while (i0 < nr) {  // CTA-uniform: every thread sees the same i0, i1
            // the run [i0, i1): a row end i1 whose span from row i0's start
            // fits the buffer, the last one for non-decreasing offsets
            // (binary search by thread 0; it keeps fits(i) true for the
            // lower bound, so it ends on a fitting i1 whatever the offsets).
            // smem index of element g is g - base, base on a 16-byte
            // boundary of x, so 16-byte chunks of x land on 16-byte slots.
            const int64_t lo = s_off[i0];
            const int64_t base = lo - ((lo + x_mis) & 3);
            const int64_t last = s_off[nr];
            int i1 = nr;  // the rest of the tile fits (every thread decides alike)
            if (!(last >= lo && last - base <= RS_CAP + 3)) {
                if (tid == 0) {
                    int a = i0, b = nr;  // fits(a); b does not fit
                    while (b - a > 1) {
                        const int m = (a + b) >> 1;
                        const int64_t hi = s_off[m];
                        if (hi >= lo && hi - base <= RS_CAP + 3)
                            a = m;
                        else
                            b = m;
                    }
                    s_i1 = a;
                }
                __syncthreads();
                i1 = s_i1;
            }
            if (i1 == i0) {
                // row i0 alone is longer than the buffer
                const int64_t oe = s_off[i0 + 1];
                cta_row<OP>(x, x_mis, lo, oe > lo ? oe : lo, accum, out + r0 + i0, s_red);
                i0 += 1;
                continue;
            }
            const int64_t hi = s_off[i1];
            stage_span(x, x_mis, lo, hi, base, s_v);
            __syncthreads();
            for (int i = i0 + tid; i < i1; i += RS_NT) {
                const int64_t ob = s_off[i], oe = s_off[i + 1];
                Fold<OP> f;
                f.init();
                if (accum)
                    f.scalar(out[r0 + i]);
                if (oe > ob) {
                    if (ob >= lo && oe <= hi) {
                        const float *p = s_v + (ob - base);
                        const int L = (int)(oe - ob);
                        for (int k = 0; k < L; ++k)
                            f.scalar(p[k]);
                    } else {
                        for (int64_t g = ob; g < oe; ++g)  // offsets that decrease
                            f.scalar(ld1(x + g));
                    }
                }
                out[r0 + i] = f.finish();
            }
            __syncthreads();  // s_v and s_i1 are rewritten by the next run
            i0 = i1;
        }
    }
}

template <int OP>
int launch_op(const float *x, const int64_t *off, int64_t rows, int64_t nnz, int accum, float *out, cudaStream_t s,
              int sms)
{
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)ragged_staged_kernel<OP>, RS_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows_ragged: staged kernel cannot be resident on this device");
    const int64_t tiles = (rows + RS_ROWS - 1) / RS_ROWS;
    int64_t ctas = (int64_t)sms * occ;
    if (tiles < ctas)
        ctas = tiles;
    if (ctas < 1)
        ctas = 1;
    const cudaError_t e = launch_pdl(ragged_staged_kernel<OP>, dim3((unsigned)ctas), dim3(RS_NT), s, x, off, rows,
                                     nnz, accum, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_ragged staged launch");
}

}  // namespace

int launch_ragged_staged(int op, const float *x, const int64_t *off, int64_t rows, int64_t nnz, int accum,
                         float *out, cudaStream_t s, int sms)
{
    switch (op) {
    case RED_SUM: return launch_op<OP_SUM>(x, off, rows, nnz, accum, out, s, sms);
    case RED_MAX: return launch_op<OP_MAX>(x, off, rows, nnz, accum, out, s, sms);
    default: return launch_op<OP_MIN>(x, off, rows, nnz, accum, out, s, sms);
    }
}

}  // namespace red
