// red_rows.cu -- per-row sum / max / min of dense row-major and of packed
// ragged (CSR-offset) fp32 rows, with the optional accum fold.
//
// A group of G lanes (G = 1, 2, ..., 32) owns one row at a time; a warp holds
// 32/G groups working on 32/G consecutive rows, whose bytes are adjacent in
// memory for both layouts, so a warp's loads stay within one contiguous span.
// Each lane folds its share of the row with the per-thread fold of Apache TVM
// docs, "reduction -> sm100_packed", "Algorithm" (chunks of 8 into the
// packed-add or max3/min3 accumulator), with accum folding the old out[r]
// into the first accumulator slot ("How inputs change the algorithm").  The
// chunks are the row's 32-byte aligned interior blocks, one 256-bit load
// each; the page's "remainder" is the row's unaligned head and tail, read as
// at most three naturally aligned 1-, 2- and 4-float pieces each, so no row
// needs a scalar loop, a short row's loads all go out at once, and every load
// lies inside the row.  The G lanes then combine through a butterfly of
// log2(G) levels.  The loop over rows is warp-uniform so that every shuffle
// has all 32 lanes present; ragged offsets are clamped into [0, nnz] and the
// next row's offsets are fetched one iteration ahead.  For ragged rows lane 0
// also issues bulk L2 prefetches of the warp's next span of values and of
// the offsets two iterations ahead (the scattered short-row loads then hit
// L2).
//
// Few long dense rows go to the split-row path instead (several CTAs per row,
// see red_full.cu).
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int ROWS_NT = 256;
constexpr int ROWS_U = 4;

// Bulk prefetch of the bytes [b, e) into L2 (no registers, no shared memory,
// no L1 miss tracking).  The range is rounded inward to 16-byte boundaries,
// so the prefetch never touches a byte outside [b, e), and capped at 64 KB.
__device__ __forceinline__ void prefetch_l2_bytes(const void *b, const void *e)
{
    const uintptr_t lo = ((uintptr_t)b + 15u) & ~(uintptr_t)15u;
    uintptr_t hi = (uintptr_t)e & ~(uintptr_t)15u;
    if (hi > lo + 65536u)
        hi = lo + 65536u;
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
}

// The floats [b, e) of x.
__device__ __forceinline__ void prefetch_l2(const float *x, int64_t b, int64_t e)
{
    prefetch_l2_bytes(x + b, x + e);
}

// Head and tail pieces of a row: L1-allocating loads (the interior blocks
// bypass L1), so that a row's tail and the next row's head, which usually
// share a 32-byte sector and are read by neighbouring lanes, meet in L1
// (ragged rows of 8..40 floats: 76.3 -> 73.8 us).
__device__ __forceinline__ float4 ld4p(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float2 ld2p(const float *p)
{
    float2 v;
    asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// Resident CTAs per SM: 3 for the general kernel (<= 85 registers); 4 for
// dense rows that start on 32-byte boundaries (ALIGNED: no head or tail
// pieces, so the lean body fits 64 registers and a lane keeps the same four
// blocks in flight with a third more lanes per SM).
template <bool ALIGNED>
constexpr int rows_min_ctas() { return ALIGNED ? 4 : 3; }

template <int OP, int G, bool RAGGED, bool ALIGNED = false>
__global__ void __launch_bounds__(ROWS_NT, rows_min_ctas<ALIGNED>())
rows_kernel(const float *__restrict__ x, const int64_t *__restrict__ off, int64_t rows, int64_t len,
            int64_t nnz, int accum, float *__restrict__ out)
{
    static_assert(!(ALIGNED && RAGGED), "ragged rows start anywhere");
    pdl_enter();
    constexpr int GPW = 32 / G;           // rows per warp at a time
    constexpr int U = ROWS_U;              // blocks in flight per lane
    const int64_t x_mis = (int64_t)(((uintptr_t)x & 31u) >> 2);  // x's offset from a 32-byte boundary
    const float ident = Op<OP>::identity();
    const int lane = threadIdx.x & 31;
    const int gl = lane & (G - 1);  // lane within the group
    const int gw = lane / G;        // group within the warp
    const int64_t warp = ((int64_t)blockIdx.x * ROWS_NT + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * ROWS_NT) >> 5;

    // Grid-stride over rows, GPW rows per warp at a time.  (A contiguous
    // block of rows per warp, which would make each warp's offsets one range,
    // measured 11% slower on ragged rows.)
    const int64_t r_begin = warp * GPW, r_end = rows, step = nwarps * GPW;

    // Row r's extent; for ragged rows the offsets of the next row this lane
    // will fold are loaded one iteration ahead, so that the row loads never
    // wait behind a dependent offsets load.
    auto extent = [&](int64_t r, int64_t &b, int64_t &L) {
        b = 0;
        L = 0;
        if (r >= r_end)
            return;
        if (RAGGED) {
            int64_t ob = off[r], oe = off[r + 1];
            ob = ob < 0 ? 0 : (ob > nnz ? nnz : ob);
            oe = oe < 0 ? 0 : (oe > nnz ? nnz : oe);
            b = ob;
            L = oe > ob ? oe - ob : 0;
        } else {
            b = r * len;
            L = len;
        }
    };
    int64_t b_next, L_next;
    extent(r_begin + gw, b_next, L_next);
    for (int64_t r0 = r_begin; r0 < r_end; r0 += step) {
        const int64_t r = r0 + gw;
        const bool live = r < r_end;
        const int64_t b = b_next, L = L_next;
        extent(r + step, b_next, L_next);
        if (RAGGED && G == 1) {
            // (One lane per row only: with several lanes per row the loads are
            // coalesced already, and the prefetches measured 8-17% slower.)
            // Bulk L2 prefetches by lane 0: the values of the warp's next
            // rows, from its own next row's start (group 0) to the last
            // group's end (both known from the offsets fetched above), and
            // the offsets of the warp's rows two iterations ahead, so that the
            // next iteration's loads and offset fetches hit L2.
            const int64_t ne = __shfl_sync(0xffffffffu, b_next + L_next, 31);
            if (lane == 0) {
                prefetch_l2(x, b_next, ne);
                const int64_t q0 = r0 + 2 * step;
                if (q0 < rows) {
                    const int64_t q1 = q0 + GPW + 1 < rows + 1 ? q0 + GPW + 1 : rows + 1;
                    prefetch_l2_bytes(off + q0, off + q1);
                }
            }
        }
        Fold<OP> f;
        f.init();
        if (live && accum && gl == 0)
            f.scalar(out[r]);
        if (L > 0) {
            // Row [b, e): the aligned interior [a, z) as 256-bit blocks spread
            // over the group's lanes (U in flight per lane), the unaligned
            // head [b, a) and tail [z, e) (0..7 floats each) as at most one
            // 1-, 2- and 4-float piece each, chosen by the bits of their
            // lengths so that every piece is naturally aligned.  Every load
            // lies inside the row.
            const int64_t e = b + L;
            const int64_t a = ALIGNED ? b : ((b + x_mis + 7) & ~int64_t(7)) - x_mis;
            const int64_t z = ALIGNED ? e : ((e + x_mis) & ~int64_t(7)) - x_mis;
            if (ALIGNED) {
                // every row is whole 32-byte blocks from an aligned start
                const int64_t nfull = L >> 3;
                const float *q = x + b;
                for (int64_t c0 = gl; c0 < nfull; c0 += (int64_t)U * G) {
                    float v[U][8];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (c0 + u * G < nfull)
                            ld8(q + 8 * (c0 + u * G), v[u]);
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (c0 + u * G < nfull)
                            f.chunk(v[u]);
                }
            } else if (a <= z) {
                float hs = ident, ts = ident;
                float2 h2 = make_float2(ident, ident), t2 = h2;
                float4 h4 = make_float4(ident, ident, ident, ident), t4 = h4;
                if (gl == 0) {
                    const int h = (int)(a - b);
                    const float *ph = x + b;
                    if (h & 1)
                        hs = ld1(ph);
                    if (h & 2)
                        h2 = ld2p(ph + (h & 1));
                    if (h & 4)
                        h4 = ld4p(ph + (h & 3));
                }
                if (gl == G - 1) {
                    const int t = (int)(e - z);
                    const float *pt = x + z;
                    if (t & 4)
                        t4 = ld4p(pt);
                    if (t & 2)
                        t2 = ld2p(pt + (t & 4));
                    if (t & 1)
                        ts = ld1(pt + (t & 6));
                }
                const int64_t nfull = (z - a) >> 3;
                const float *q = x + a;
                for (int64_t c0 = gl; c0 < nfull; c0 += (int64_t)U * G) {
                    float v[U][8];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (c0 + u * G < nfull)
                            ld8(q + 8 * (c0 + u * G), v[u]);
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (c0 + u * G < nfull)
                            f.chunk(v[u]);
                }
                f.scalar(hs);
                f.scalar(ts);
                f.pair(h2);
                f.pair(t2);
                f.quad(h4);
                f.quad(t4);
            } else {
                // the whole row inside one 32-byte block (fewer than 8
                // floats): every load of the lane out before any fold (a
                // loop with a fold per load would wait out each load in turn)
                constexpr int KMAX = (7 + G - 1) / G;
                float t[KMAX];
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    const int64_t i = b + gl + (int64_t)k * G;
                    t[k] = i < e ? ld1(x + i) : ident;
                }
#pragma unroll
                for (int k = 0; k < KMAX; ++k)
                    f.scalar(t[k]);
            }
        }
        const float v = group_tree<OP, G>(f.finish());
        if (live && gl == 0)
            out[r] = v;
    }
}

template <int OP, int G, bool RAGGED, bool ALIGNED>
int launch_group(const float *x, const int64_t *off, int64_t rows, int64_t len, int64_t nnz, int accum,
                 float *out, cudaStream_t s, int sms)
{
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)rows_kernel<OP, G, RAGGED, ALIGNED>, ROWS_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "row kernel cannot be resident on this device");
    const int64_t rows_per_cta = (int64_t)(ROWS_NT / 32) * (32 / G);
    int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
    const int64_t cap = (int64_t)sms * occ;
    if (ctas > cap)
        ctas = cap;
    if (ctas < 1)
        ctas = 1;
    const cudaError_t e = launch_pdl(rows_kernel<OP, G, RAGGED, ALIGNED>, dim3((unsigned)ctas), dim3(ROWS_NT), s, x,
                                     off, rows, len, nnz, accum, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "row kernel launch");
}

template <int OP, bool RAGGED, bool ALIGNED>
int launch_g(int G, const float *x, const int64_t *off, int64_t rows, int64_t len, int64_t nnz, int accum,
             float *out, cudaStream_t s, int sms)
{
    switch (G) {
    case 1: return launch_group<OP, 1, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    case 2: return launch_group<OP, 2, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    case 4: return launch_group<OP, 4, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    case 8: return launch_group<OP, 8, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    case 16: return launch_group<OP, 16, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    default: return launch_group<OP, 32, RAGGED, ALIGNED>(x, off, rows, len, nnz, accum, out, s, sms);
    }
}

template <bool RAGGED, bool ALIGNED = false>
int launch_op(int op, int G, const float *x, const int64_t *off, int64_t rows, int64_t len, int64_t nnz,
              int accum, float *out, cudaStream_t s, int sms)
{
    switch (op) {
    case OP_SUM: return launch_g<OP_SUM, RAGGED, ALIGNED>(G, x, off, rows, len, nnz, accum, out, s, sms);
    case OP_MAX: return launch_g<OP_MAX, RAGGED, ALIGNED>(G, x, off, rows, len, nnz, accum, out, s, sms);
    default: return launch_g<OP_MIN, RAGGED, ALIGNED>(G, x, off, rows, len, nnz, accum, out, s, sms);
    }
}

// Lanes per row for a (mean) row length: about 32 floats per lane, a power of
// two in 1..32.
int auto_group(int64_t mean_len)
{
    int g = 1;
    while (g < 32 && (int64_t)g * 64 <= mean_len)
        g *= 2;
    return g;
}

}  // namespace

int launch_rows(int op, const float *x, int64_t rows, int64_t len, int accum, float *out, cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    // Rows of at most RED_THREAD_MAX_LEN floats: the thread-scope kernel
    // (tiles of 128 rows staged through shared memory with coalesced loads,
    // one thread per row) beats a lane per row with scattered loads at every
    // such length (rows of 32: 7.0 vs 5.6 TB/s; of 8: 5.0 vs 4.2).
    if (knob(RED_KNOB_ROWS_GROUP) == 0 && len <= RED_THREAD_MAX_LEN)
        return launch_rows_thread(op, x, rows, (int)len, accum, out, s);
    // Long rows go to the segmented kernel (CTAs per row) when there are too
    // few rows to fill the GPU with one lane group per row, and for rows of
    // 32768 floats or more when they outnumber the row kernel's warps (24 per
    // SM): a warp per row would then finish with a partial second pass,
    // while CTAs per 128+ KB row balance over many waves (4096 x 65536: 7.35
    // vs 6.43 TB/s).  With fewer such rows every row has its own warp and
    // the row kernel stays (2500 x 40000: 6.64 vs 6.02); rows of 8K-16K
    // floats stay too (the CTA stage costs more than it gains).  The
    // segmented grid holds one row per gridDim.y index, at most 65535.
    if (knob(RED_KNOB_ROWS_GROUP) == 0 && len >= 8192 &&
        (rows < (int64_t)di.sms * 16 || (len >= 32768 && rows > (int64_t)di.sms * 24 && rows <= 65535)))
        return launch_rows_split(op, x, rows, len, accum, out, s, di);
    const int g = knob(RED_KNOB_ROWS_GROUP) ? knob(RED_KNOB_ROWS_GROUP) : auto_group(len);
    // Rows of whole 32-byte blocks from a 32-byte aligned x: the lean body at
    // 4 CTAs per SM (unless the knob asks for the general kernel).
    if (knob(RED_KNOB_ROWS_ALIGNED) != 2 && (((uintptr_t)x) & 31u) == 0 && len % 8 == 0)
        return launch_op<false, true>(op, g, x, nullptr, rows, len, 0, accum, out, s, di.sms);
    return launch_op<false>(op, g, x, nullptr, rows, len, 0, accum, out, s, di.sms);
}

// Mean ragged row length (floats) below which the staged tiles are used
// (measured, staged vs lanes per row: rows of 2..6 floats 3.84 vs 2.17 TB/s,
// of 4..12 3.88 vs 3.09, of 6..14 3.93 vs 3.83, of 8..16 3.57 vs 4.57).
constexpr int64_t RAGGED_STAGED_MEAN = 11;

int launch_ragged(int op, const float *x, const int64_t *off, int64_t rows, int64_t nnz, int accum,
                  float *out, cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    // Short rows (mean below RAGGED_STAGED_MEAN floats) through shared-memory
    // tiles, longer ones with lanes per row and direct loads; a lanes-per-row
    // setting asks for the direct mapping.
    const int mode = knob(RED_KNOB_RAGGED_STAGED);
    const bool staged = mode == 1 || (mode == 0 && knob(RED_KNOB_RAGGED_GROUP) == 0 && rows > 0 &&
                                      nnz < RAGGED_STAGED_MEAN * rows);
    if (staged)
        return launch_ragged_staged(op, x, off, rows, nnz, accum, out, s, di.sms);
    const int g = knob(RED_KNOB_RAGGED_GROUP) ? knob(RED_KNOB_RAGGED_GROUP)
                                               : auto_group(rows > 0 ? nnz / rows : 0);
    return launch_op<true>(op, g, x, off, rows, 0, nnz, accum, out, s, di.sms);
}

}  // namespace red
