// red_cols.cu -- column reductions dst[0,j] = op_{i<R} src[i,j] of the R x C
// valid region of a row-major matrix with row stride ld >= C: TCOLPROD
// (pto-isa docs, "TCOLPROD", "Math Interpretation") and its column siblings
// sum, max and min, for the element types of that
// page's A2A3 / A5 lists ("Constraints"): float, int32, half, bfloat16,
// int16, uint16, uint32.  dst has src's element type.
//
// Arithmetic: floating types accumulate in fp32 (products __fmul_rn, sums
// __fadd_rn; half and bfloat16 are widened exactly and the result is rounded
// to nearest once); integer sums and products wrap modulo 2^bits of the type
// (done in 32-bit unsigned arithmetic, then truncated for the 16-bit types);
// max / min compare values (signed or unsigned as the type is).
//
// Layout of the work: a CTA of 16 warps owns a tile of lpr*V adjacent
// columns, lpr lanes per row (8 for matrices of many rows, 32 for short ones,
// or the power of two that covers a narrower matrix; the warps take 32/lpr
// consecutive rows per step, so no lane idles).  Each lane owns V adjacent
// columns and keeps V running accumulators (per-thread column
// accumulators); the lane groups of warp w
// walk rows i0 + w*32/lpr, ... in steps of 16*32/lpr rows, each lane reading
// 32 bytes of a row per load (16 bytes for 16-bit types, whose lanes then
// keep 8 rows in flight instead of 4; coalesced, row-major order kept).  The
// loaded words stay raw until they are folded.  The row
// groups of a warp meet in a butterfly, the 16 warps in shared memory (fixed
// order).  gridDim.y CTAs split the rows; with more than one, the CTA
// partials go to the workspace and the CTA that arrives last for its column
// tile folds them, with all its lanes in a fixed order, into dst (the
// arrival is an acquire-release atomic, so no CTA fences or waits).
#include "red_internal.h"
#include "red_prims.cuh"
#include "red_types.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int CP_WY = 16;                // warps per CTA (row interleave)
constexpr int CP_NT = 32 * CP_WY;

// Raw 32-bit words of a lane's V elements of one row: V * sizeof(T) is 32
// (256-bit load, 8 words), 16 (128-bit load, 4 words) or sizeof(T) (one
// element in the low bits of one word).  Rows are held raw while in flight
// and widened only when folded, so 16-bit types keep as many bytes in flight
// per register as 32-bit ones.
template <int DT, int V>
struct RawRow {
    static constexpr int BYTES = V * (int)sizeof(typename Elem<DT>::T);
    static constexpr int W = BYTES >= 16 ? BYTES / 4 : 1;
};

// rows in flight per thread: 128 bytes for the vector paths, 8 elements for
// the one-element path
template <int DT, int V>
__host__ __device__ constexpr int cols_u()
{
    return RawRow<DT, V>::BYTES >= 16 ? 128 / RawRow<DT, V>::BYTES : 8;
}

template <int DT, int V>
__device__ __forceinline__ void load_raw(const typename Elem<DT>::T *p, uint32_t (&w)[RawRow<DT, V>::W])
{
    using T = typename Elem<DT>::T;
    constexpr int W = RawRow<DT, V>::W;
    if constexpr (W == 8) {
        ld8u(reinterpret_cast<const uint32_t *>(p), w);
    } else if constexpr (W == 4) {
        ld4u(reinterpret_cast<const uint32_t *>(p), w);
    } else if constexpr (sizeof(T) == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else {
        w[0] = __ldg(reinterpret_cast<const unsigned short *>(p));
    }
}

// acc[k] = op(acc[k], element k of the raw row), elements in column order.
template <int OP, int DT, int V>
__device__ __forceinline__ void fold_raw(typename Elem<DT>::A (&acc)[V], const uint32_t (&w)[RawRow<DT, V>::W])
{
    using E = Elem<DT>;
    using K = Comb<OP, typename E::A>;
    if constexpr (sizeof(typename E::T) == 4 || V == 1) {
#pragma unroll
        for (int k = 0; k < V; ++k)
            acc[k] = K::op(acc[k], E::widen(w[k]));
    } else {
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
            acc[2 * k] = K::op(acc[2 * k], E::widen(w[k] & 0xffffu));
            acc[2 * k + 1] = K::op(acc[2 * k + 1], E::widen(w[k] >> 16));
        }
    }
}

template <int OP, int DT, int V>
__global__ void __launch_bounds__(CP_NT, 2)
cols_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t R, int64_t C, int64_t ld, int64_t rows_per_split,
            int lpr, typename Elem<DT>::A *__restrict__ part, unsigned *__restrict__ tick,
            typename Elem<DT>::T *__restrict__ out)
{
    pdl_enter();
    using E = Elem<DT>;
    using A = typename E::A;
    using K = Comb<OP, A>;
    constexpr int U = cols_u<DT, V>();
    constexpr int W = RawRow<DT, V>::W;
    __shared__ A s_p[CP_WY][32 * V];
    __shared__ int s_last;

    // lpr lanes (a power of two) cover a row of the tile; the warp's 32 / lpr
    // lane groups take consecutive rows, so narrow matrices keep every lane busy
    const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;
    const int rpw = 32 / lpr;           // rows per warp step
    const int cl = lane & (lpr - 1);    // lane within its row group
    const int sub = lane / lpr;         // row group within the warp
    const int64_t col = ((int64_t)blockIdx.x * lpr + cl) * V;
    const bool live = col < C;  // V > 1 only when C % V == 0
    const int64_t i0 = (int64_t)blockIdx.y * rows_per_split;
    const int64_t i1 = (i0 + rows_per_split < R) ? i0 + rows_per_split : R;
    const int64_t step = (int64_t)CP_WY * rpw;

    A p[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        p[k] = K::identity();
    if (live) {
        // rows i0 + wy*rpw + sub, then every step-th row, below i1: walked as
        // a pointer to the lane's columns of the row, rs elements per step
        const int64_t i = i0 + (int64_t)wy * rpw + sub;
        const typename E::T *r = x + i * ld + col;
        const typename E::T *const end = x + i1 * ld + col;
        const int64_t rs = step * ld;
        for (; r + (U - 1) * rs < end; r += U * rs) {
            uint32_t w[U][W];
#pragma unroll
            for (int u = 0; u < U; ++u)
                load_raw<DT, V>(r + u * rs, w[u]);
#pragma unroll
            for (int u = 0; u < U; ++u)
                fold_raw<OP, DT, V>(p, w[u]);
        }
        // the last (fewer than U) rows: a batch of U / 2, then one at a time
        if constexpr (U >= 4) {
            constexpr int H = U / 2;
            if (r + (H - 1) * rs < end) {
                uint32_t w[H][W];
#pragma unroll
                for (int u = 0; u < H; ++u)
                    load_raw<DT, V>(r + u * rs, w[u]);
#pragma unroll
                for (int u = 0; u < H; ++u)
                    fold_raw<OP, DT, V>(p, w[u]);
                r += H * rs;
            }
        }
        for (; r < end; r += rs) {
            uint32_t w[W];
            load_raw<DT, V>(r, w);
            fold_raw<OP, DT, V>(p, w);
        }
    }
    // the row groups of the warp meet (butterfly over the group bits)
    for (int o = lpr; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < V; ++k)
            p[k] = K::op(p[k], __shfl_xor_sync(0xffffffffu, p[k], o));
    if (sub == 0)
#pragma unroll
        for (int k = 0; k < V; ++k)
            s_p[wy][cl * V + k] = p[k];
    __syncthreads();
    if (wy == 0 && sub == 0) {
#pragma unroll
        for (int w = 1; w < CP_WY; ++w)
#pragma unroll
            for (int k = 0; k < V; ++k)
                p[k] = K::op(p[k], s_p[w][cl * V + k]);
    }
    const bool writer = wy == 0 && sub == 0 && live;

    if (gridDim.y == 1) {
        if (writer)
#pragma unroll
            for (int k = 0; k < V; ++k)
                out[col + k] = E::narrow(p[k]);
        return;
    }
    if (writer)
#pragma unroll
        for (int k = 0; k < V; ++k)
            part[(int64_t)blockIdx.y * C + col + k] = p[k];
    __syncthreads();
    if (threadIdx.x == 0) {
        // release this CTA's partials (ordered before by the barrier) with the
        // arrival; the last arrival acquires every other CTA's partials
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(tick + blockIdx.x) : "memory");
        s_last = prev == gridDim.y - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    // The last CTA folds the gridDim.y partials of its tile with all of its
    // lanes: row group g of warp w takes splits w*rpw+g, w*rpw+g + 16*rpw, ...
    // (a fixed assignment), then the groups meet in a butterfly and the warps
    // in shared memory, in warp order.
    A q[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        q[k] = K::identity();
    if (live)
        for (int64_t sp = (int64_t)wy * rpw + sub; sp < (int64_t)gridDim.y; sp += step)
#pragma unroll
            for (int k = 0; k < V; ++k)
                q[k] = K::op(q[k], ldcg_a<A>(part + sp * C + col + k));
    for (int o = lpr; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < V; ++k)
            q[k] = K::op(q[k], __shfl_xor_sync(0xffffffffu, q[k], o));
    __syncthreads();  // every read of s_p above is done
    if (sub == 0)
#pragma unroll
        for (int k = 0; k < V; ++k)
            s_p[wy][cl * V + k] = q[k];
    __syncthreads();
    if (writer) {
#pragma unroll
        for (int w = 1; w < CP_WY; ++w)
#pragma unroll
            for (int k = 0; k < V; ++k)
                q[k] = K::op(q[k], s_p[w][cl * V + k]);
#pragma unroll
        for (int k = 0; k < V; ++k)
            out[col + k] = E::narrow(q[k]);
    }
    if (threadIdx.x == 0)
        tick[blockIdx.x] = 0;
}

template <int OP, int DT, int V>
int launch_cols(const void *xv, int64_t R, int64_t C, int64_t ld, void *outv, cudaStream_t s, const DeviceInfo &di)
{
    using E = Elem<DT>;
    using T = typename E::T;
    using A = typename E::A;
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)cols_kernel<OP, DT, V>, CP_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_cols: kernel cannot be resident on this device");
    constexpr int U = cols_u<DT, V>();
    // lanes per row: enough V-wide chunks for C columns, a power of two <= 32
    const int64_t chunks = (C + V - 1) / V;
    int lpr = 1;
    while (lpr < 32 && lpr < chunks)
        lpr *= 2;
    // At most 8 lanes per row (tiles of 8 * V columns, 128-256 bytes of a row
    // per lane group) when every lane of an unsplit tile still keeps U rows in
    // flight: narrow tiles are many enough to fill the GPU without splitting
    // the rows, and a split costs a combine at the end of the launch (4096 x
    // 16384: fp32 product 42.2 -> 40.0 us, f16 23.2 -> 21.1 us; 65536 x 1024
    // fp32 sum 43.6 -> 41.2 us).  Short matrices keep wide tiles: a lane then
    // still sees several rows (64 x 65536 int32: 3.9 us, 7.3 with 8 lanes).
    if (lpr > 8 && RawRow<DT, V>::BYTES >= 16 && R >= (int64_t)CP_WY * 4 * U)
        lpr = 8;
    if (knob(RED_KNOB_COLS_LANES) > 0 && lpr > knob(RED_KNOB_COLS_LANES))
        lpr = knob(RED_KNOB_COLS_LANES);
    const int rpw = 32 / lpr;
    const int64_t tile_cols = (int64_t)lpr * V;
    const int64_t tiles = (C + tile_cols - 1) / tile_cols;
    if (tiles > 0x7fffffffLL)
        return fail(RED_EINVAL, "red_cols: C too large");
    // Row splits (each warp keeps at least U rows).  When the tiles alone
    // fill at least 80% of the resident slots the rows are not split (no
    // combine: 4096 x 16384 fp32 in 256 CTAs, 40.0 us; with 4 splits of 64
    // wider tiles 42.2).  Otherwise a wave of CTAs carries a fixed cost of a
    // few microseconds (the CTAs' ramp, the split combine), so when one wave
    // of at least 80% of the resident slots gives each CTA at most 2 MiB to
    // stream, that single wave is taken, as full as the tiles allow.
    // Otherwise the smallest count whose CTAs fill their waves to at least 90%
    // (more splits add partial traffic and per-CTA overhead), else the count
    // with the best wave efficiency.
    int64_t splits = knob(RED_KNOB_COLPROD_SPLITS);
    if (splits <= 0 && (double)tiles >= 0.8 * (double)((int64_t)di.sms * occ))
        splits = 1;
    if (splits <= 0) {
        const int64_t slots = (int64_t)di.sms * occ;
        int64_t smax = R / ((int64_t)CP_WY * U * rpw);
        if (smax > 4096)
            smax = 4096;
        if (smax < 1)
            smax = 1;
        const int64_t one = slots / tiles < smax ? slots / tiles : smax;  // single-wave count
        const double cta_bytes = (double)R * (double)C * (double)sizeof(T) / (double)(tiles * (one > 0 ? one : 1));
        if (one >= 1 && (double)(tiles * one) >= 0.8 * (double)slots && cta_bytes <= 2.0 * 1024 * 1024) {
            splits = one;
        } else {
            splits = 1;
            double best = -1.0;
            for (int64_t sp = 1; sp <= smax; ++sp) {
                const int64_t ctas = tiles * sp;
                const double eff = (double)ctas / (double)(((ctas + slots - 1) / slots) * slots);
                if (eff >= 0.9) {
                    splits = sp;
                    break;
                }
                if (eff > best) {
                    best = eff;
                    splits = sp;
                }
            }
        }
    }
    if (splits > R)
        splits = R;
    if (splits > 65535)
        splits = 65535;
    if (splits * C > (int64_t)WS_PART_ELEMS)
        splits = (int64_t)WS_PART_ELEMS / C;
    if (tiles > WS_TICKETS)
        splits = 1;
    if (splits < 1)
        splits = 1;
    const int64_t rps = (R + splits - 1) / splits;
    splits = (R + rps - 1) / rps;  // no empty split
    Workspace ws;
    if (splits > 1) {
        const int st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    const dim3 grid((unsigned)tiles, (unsigned)splits);
    const cudaError_t e = launch_pdl(cols_kernel<OP, DT, V>, grid, dim3(CP_NT), s, static_cast<const T *>(xv), R, C, ld,
                                     rps, lpr, static_cast<A *>(ws.part), ws.tick, static_cast<T *>(outv));
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_cols launch");
}

// Vector width by alignment: 32-byte rows and base -> 256-bit loads,
// 16-byte -> 128-bit, otherwise one element per lane.
template <int OP, int DT>
int launch_cols_dt(const void *x, int64_t R, int64_t C, int64_t ld, void *out, cudaStream_t s, const DeviceInfo &di)
{
    constexpr int SZ = (int)sizeof(typename Elem<DT>::T);
    const uintptr_t a = (uintptr_t)x;
    // Every row start keeps the alignment (ld), and C is a whole number of
    // vectors, so a lane's V columns never pass column C (neither the reads
    // of a row nor the writes to out).
    const int64_t row_bytes = ld * SZ, valid_bytes = C * SZ;
    // 16-bit types take 128-bit loads (8 columns and 8 rows in flight per
    // lane) unless the lanes see too few rows to fill 8 loads each
    const bool wide = SZ == 4 || R < (int64_t)CP_WY * 8;
    if (wide && row_bytes % 32 == 0 && valid_bytes % 32 == 0 && a % 32 == 0)
        return launch_cols<OP, DT, 32 / SZ>(x, R, C, ld, out, s, di);
    if (row_bytes % 16 == 0 && valid_bytes % 16 == 0 && a % 16 == 0)
        return launch_cols<OP, DT, 16 / SZ>(x, R, C, ld, out, s, di);
    return launch_cols<OP, DT, 1>(x, R, C, ld, out, s, di);
}

template <int OP>
int launch_cols_op(int dtype, const void *x, int64_t R, int64_t C, int64_t ld, void *out, cudaStream_t s,
                   const DeviceInfo &di)
{
    switch (dtype) {
    case RED_F32: return launch_cols_dt<OP, RED_F32>(x, R, C, ld, out, s, di);
    case RED_I32: return launch_cols_dt<OP, RED_I32>(x, R, C, ld, out, s, di);
    case RED_F16: return launch_cols_dt<OP, RED_F16>(x, R, C, ld, out, s, di);
    case RED_BF16: return launch_cols_dt<OP, RED_BF16>(x, R, C, ld, out, s, di);
    case RED_I16: return launch_cols_dt<OP, RED_I16>(x, R, C, ld, out, s, di);
    case RED_U16: return launch_cols_dt<OP, RED_U16>(x, R, C, ld, out, s, di);
    default: return launch_cols_dt<OP, RED_U32>(x, R, C, ld, out, s, di);
    }
}

}  // namespace

int launch_cols(int op, int dtype, const void *x, int64_t R, int64_t C, int64_t ld, void *out, cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    switch (op) {
    case RED_SUM: return launch_cols_op<RED_SUM>(dtype, x, R, C, ld, out, s, di);
    case RED_MAX: return launch_cols_op<RED_MAX>(dtype, x, R, C, ld, out, s, di);
    case RED_MIN: return launch_cols_op<RED_MIN>(dtype, x, R, C, ld, out, s, di);
    default: return launch_cols_op<RED_PROD>(dtype, x, R, C, ld, out, s, di);
    }
}

}  // namespace red
